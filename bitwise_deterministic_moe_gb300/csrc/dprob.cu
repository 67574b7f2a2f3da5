// Unfused private-slot dprob epilogue and the fixed-order slot combine.
//
// "Trillion-Parameter Pretraining Goes Bitwise-Deterministic: NVIDIA Cuts the
// Determinism Tax to About 2%", section "Interpretation": each N-tile writes
// a private slot, and the slots are combined in a fixed order after all
// writers finish.  The unfused epilogue reproduces the fused one's arithmetic
// exactly (same fixed tree per 128-column slot), so both give the same bits.
#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int SLOT = DMOE_SLOT_COLS;

// A warp takes eight consecutive permuted rows and walks their slots.  Four
// lanes share a row: lane k4 holds the 16-byte group k4 of each 64-byte
// quarter of the slot (columns 32*ch + 8*k4 .. +7, ch = 0..3), so one load
// instruction reads 64 contiguous bytes of each of eight rows of expert_out
// (and of their tokens' grad_out rows).  Each lane chains its products over
// ch, folds them with slot_tree, and two xor-shuffles give
// (L0 + L1) + (L2 + L3): the fused epilogue's tree, so the bits are the same.
// grad_out rows are read by every choice of their token (L2 evict-last);
// expert_out streams through once (evict-first).
constexpr int EPI_THREADS = 256;
constexpr int EPI_ROWS_PER_WARP = 8;

__global__ void __launch_bounds__(EPI_THREADS)
dprob_epilogue_kernel(const uint16_t* __restrict__ grad_out, const uint16_t* __restrict__ expert_out,
                      const int32_t* __restrict__ offsets, const int32_t* __restrict__ row_src, int R, int E,
                      int topk, int N, int S, float* __restrict__ slots, int* status) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int k4 = lane & 3;
  const long long warp_id = ((long long)blockIdx.x * EPI_THREADS + threadIdx.x) >> 5;
  const int rows = offsets[E];
  if (warp_id == 0 && lane == 0 && rows != R) record_error(status, DMOE_ERR_ROUTING);
  const long long r0 = warp_id * EPI_ROWS_PER_WARP;
  if (r0 >= R) return;                                   // whole warp
  const int r = int(r0) + (lane >> 2);
  bool ok = r < R && r < rows;
  int tok = 0;
  if (ok) {
    const int src = row_src[r];
    if (unsigned(src) >= unsigned(R)) {                  // corrupt row_src: report, never index with it
      record_error(status, DMOE_ERR_ROUTING);
      ok = false;
    } else {
      tok = src / topk;
    }
  }
  const uint16_t* g = grad_out + size_t(tok) * N + k4 * 8;
  const uint16_t* y = expert_out + size_t(ok ? r : 0) * N + k4 * 8;
  const uint64_t pol_keep = policy_evict_last();
  const uint64_t pol_stream = policy_evict_first();
#pragma unroll 2
  for (int s = 0; s < S; ++s) {
    uint4 gv[4], yv[4];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      gv[ch] = ok ? ldg_nc_v4_hint(g + s * SLOT + ch * 32, pol_keep) : make_uint4(0u, 0u, 0u, 0u);
      yv[ch] = ok ? ldg_nc_v4_hint(y + s * SLOT + ch * 32, pol_stream) : make_uint4(0u, 0u, 0u, 0u);
    }
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = 0.0f;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) slot_accumulate8(a, gv[ch], yv[ch]);
    float part = slot_tree(a);
    part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
    part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 2));
    if (k4 == 0 && ok) slots[size_t(s) * R + r] = part;
  }
}

// One thread per permuted row: ascending-slot fp32 sum, scattered to dprob.
// The general form, for any R, S and alignment.
template <int S_STATIC>
__global__ void __launch_bounds__(256)
dprob_combine_kernel(const float* __restrict__ slots, const int32_t* __restrict__ row_src, int R, int S,
                     float* __restrict__ dprob) {
  pdl_begin();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const int nS = S_STATIC > 0 ? S_STATIC : S;
  float v[S_STATIC > 0 ? S_STATIC : 1];
  float acc;
  if (S_STATIC > 0) {
#pragma unroll
    for (int s = 0; s < nS; ++s) v[s] = __ldg(slots + size_t(s) * R + r);
    acc = v[0];
#pragma unroll
    for (int s = 1; s < nS; ++s) acc = __fadd_rn(acc, v[s]);
  } else {
    acc = slots[r];
    for (int s = 1; s < nS; ++s) acc = __fadd_rn(acc, __ldg(slots + size_t(s) * R + r));
  }
  const int dst = row_src[r];
  if (unsigned(dst) < unsigned(R)) dprob[dst] = acc;   // a corrupt index is skipped, never written through
}

// Positional chunk fingerprints of row_src and dprob taken by the combine
// itself (the mode-0 hash of dmoe_fingerprint: per chunk the sum mod 2^64 of
// fmix32(word_i ^ i*0x9E3779B9) over its 32-bit words, finalized as
// sm64(sum ^ (c << 32) ^ chunk_length)).  The combine reads every row_src word
// and writes every dprob word once, so it forms the terms from values it
// already holds.  Sums are integers mod 2^64, so the order in which warps and
// blocks add them does not matter: warp sums go into the block's shared
// accumulators, block sums into the workspace's, and the last block to finish
// finalizes the hashes and zeroes the accumulators for the next call.
struct FpFuse {
  unsigned long long* acc;   // [2 * kFpMaxChunks] in the workspace: row_src chunks, then dprob chunks
  int* done;                 // finished-block counter in the workspace
  unsigned long long* src_hash;
  unsigned long long* dprob_hash;
  int chunk_words;           // chunk_bytes / 4, a multiple of 128
  int nch;                   // chunks of each buffer (R*4 bytes), <= kFpMaxChunks
};

__device__ __forceinline__ uint32_t fp_fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  return h;
}

__device__ __forceinline__ uint64_t fp_sm64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ uint64_t fp_term(uint32_t w, uint32_t i) { return fp_fmix32(w ^ (i * 0x9E3779B9u)); }

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// One thread's terms (row_src words 4i..4i+3, all in one chunk because a
// chunk is a multiple of 128 words; dprob words dst.x..w, each in its own
// chunk) summed per chunk over the warp and the block, then into the
// workspace; then the thread's dprob stores (a corrupt index skipped, never
// written through); the last block finalizes.  Every thread of the block
// calls it (active = 0 for threads past R: no terms, no stores).
template <bool FP>
__device__ __forceinline__ void combine_fp_block(const FpFuse& f, int active, int i, int4 dst, float4 v, int R,
                                                 float* __restrict__ dprob) {
  __shared__ unsigned long long bacc[2 * kFpMaxChunks];
  __shared__ int last;
  const int t = threadIdx.x;
  const int lane = t & 31;
  if (t < 2 * kFpMaxChunks) bacc[t] = 0;
  __syncthreads();
  uint64_t hs[kFpMaxChunks], hd[kFpMaxChunks];
#pragma unroll
  for (int c = 0; c < kFpMaxChunks; ++c) hs[c] = hd[c] = 0;
  if (active) {
    const int d[4] = {dst.x, dst.y, dst.z, dst.w};
    const float x[4] = {v.x, v.y, v.z, v.w};
    const int cs = (4 * i) / f.chunk_words;
    uint64_t s4 = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      s4 += fp_term(uint32_t(d[k]), uint32_t(4 * i + k));
      if (unsigned(d[k]) < unsigned(R)) {
        const int cd = d[k] / f.chunk_words;
        const uint64_t term = fp_term(__float_as_uint(x[k]), uint32_t(d[k]));
#pragma unroll
        for (int c = 0; c < kFpMaxChunks; ++c)
          if (c == cd) hd[c] += term;
      }
    }
#pragma unroll
    for (int c = 0; c < kFpMaxChunks; ++c)
      if (c == cs) hs[c] += s4;
  }
#pragma unroll
  for (int c = 0; c < kFpMaxChunks; ++c) {
    if (c >= f.nch) break;
    if (__any_sync(0xffffffffu, hs[c] != 0)) {
      const uint64_t w = warp_sum_u64(hs[c]);
      if (lane == 0) atomicAdd(&bacc[c], (unsigned long long)w);
    }
    if (__any_sync(0xffffffffu, hd[c] != 0)) {
      const uint64_t w = warp_sum_u64(hd[c]);
      if (lane == 0) atomicAdd(&bacc[kFpMaxChunks + c], (unsigned long long)w);
    }
  }
  __syncthreads();
  if (t < 2 * kFpMaxChunks) {
    const unsigned long long b = bacc[t];
    if (b != 0) atomicAdd(f.acc + t, b);
  }
  __syncthreads();
  if (t == 0) {
    // release: the fence is cumulative over the block's adds above (ordered
    // before it by the barrier), so they are visible before the count; on the
    // last block, acquire every other block's adds before the reads below
    fence_acq_rel_gpu();
    last = atomicAdd(f.done, 1) == int(gridDim.x) - 1;
    if (last) fence_acq_rel_gpu();
  }
  // the dprob stores go out after the block's sums are published, so that the
  // fence above does not wait for them
  if (active) {
    if (unsigned(dst.x) < unsigned(R)) dprob[dst.x] = v.x;
    if (unsigned(dst.y) < unsigned(R)) dprob[dst.y] = v.y;
    if (unsigned(dst.z) < unsigned(R)) dprob[dst.z] = v.z;
    if (unsigned(dst.w) < unsigned(R)) dprob[dst.w] = v.w;
  }
  __syncthreads();
  if (!last) return;
  // the last block: every other block's sums are in the workspace (thread 0's
  // acquire, ordered before these reads by the barrier)
  if (t < 2 * kFpMaxChunks) {
    const int c = t % kFpMaxChunks;
    const unsigned long long sum = atomicExch(f.acc + t, 0ull);   // read, and leave zero for the next call
    if (c < f.nch) {
      const long long words = (long long)R - (long long)c * f.chunk_words;
      const uint64_t len = uint64_t(words < f.chunk_words ? words : f.chunk_words) * 4;
      const uint64_t h = fp_sm64(uint64_t(sum) ^ (uint64_t(c) << 32) ^ len);
      if (t < kFpMaxChunks) f.src_hash[c] = h;
      else f.dprob_hash[c] = h;
    }
  }
  if (t == 0) atomicExch(f.done, 0);
}

// The vectorised form (R % 4 == 0, slots and row_src 16-byte aligned): a
// thread owns four consecutive rows and reads each slot's four values with
// one 16-byte load, all of its S loads in flight at once, so the pass moves
// the slot buffer in few, wide requests.  Each row is still summed on its own
// in ascending s from slot 0, so the bits equal the general form's.  FP: also
// the fingerprints above (every thread then stays to the block's reduction).
template <int S_STATIC, bool FP>
__global__ void __launch_bounds__(256)
dprob_combine_v4_kernel(const float* __restrict__ slots, const int32_t* __restrict__ row_src, int R, int S,
                        float* __restrict__ dprob, FpFuse f) {
  pdl_begin();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;   // group of rows 4i .. 4i+3
  const bool active = 4ll * i < R;
  if (!FP && !active) return;
  if (FP && !active) {
    combine_fp_block<FP>(f, 0, 0, make_int4(-1, -1, -1, -1), make_float4(0.f, 0.f, 0.f, 0.f), R, dprob);
    return;
  }
  const int nS = S_STATIC > 0 ? S_STATIC : S;
  const float4* p = reinterpret_cast<const float4*>(slots) + i;
  const size_t stride = size_t(R) / 4;                   // one slot, in float4
  float4 acc = __ldg(p);
  if (S_STATIC > 0) {
    float4 v[S_STATIC > 1 ? S_STATIC - 1 : 1];
#pragma unroll
    for (int s = 1; s < nS; ++s) v[s - 1] = __ldg(p + size_t(s) * stride);
#pragma unroll
    for (int s = 1; s < nS; ++s) {
      acc.x = __fadd_rn(acc.x, v[s - 1].x);
      acc.y = __fadd_rn(acc.y, v[s - 1].y);
      acc.z = __fadd_rn(acc.z, v[s - 1].z);
      acc.w = __fadd_rn(acc.w, v[s - 1].w);
    }
  } else {
    for (int s = 1; s < nS; ++s) {
      const float4 v = __ldg(p + size_t(s) * stride);
      acc.x = __fadd_rn(acc.x, v.x);
      acc.y = __fadd_rn(acc.y, v.y);
      acc.z = __fadd_rn(acc.z, v.z);
      acc.w = __fadd_rn(acc.w, v.w);
    }
  }
  const int4 dst = __ldg(reinterpret_cast<const int4*>(row_src) + i);
  if (FP) {
    combine_fp_block<FP>(f, 1, i, dst, acc, R, dprob);   // also stores dprob
    return;
  }
  // a corrupt index is skipped, never written through
  if (unsigned(dst.x) < unsigned(R)) dprob[dst.x] = acc.x;
  if (unsigned(dst.y) < unsigned(R)) dprob[dst.y] = acc.y;
  if (unsigned(dst.z) < unsigned(R)) dprob[dst.z] = acc.z;
  if (unsigned(dst.w) < unsigned(R)) dprob[dst.w] = acc.w;
}

}  // namespace

cudaError_t launch_dprob_epilogue(const void* grad_out, const void* expert_out, const int32_t* offsets,
                                  const int32_t* row_src, int R, int E, int topk, int N, float* slots,
                                  int* status, cudaStream_t stream) {
  const int S = N / SLOT;
  if (R == 0 || S == 0) return cudaSuccess;
  const long long warps = (R + EPI_ROWS_PER_WARP - 1) / EPI_ROWS_PER_WARP;
  const unsigned grid = unsigned((warps * 32 + EPI_THREADS - 1) / EPI_THREADS);
  return launch_chained(dprob_epilogue_kernel, dim3(grid), dim3(EPI_THREADS), 0, stream,
                        static_cast<const uint16_t*>(grad_out), static_cast<const uint16_t*>(expert_out), offsets,
                        row_src, R, E, topk, N, S, slots, status);
}

cudaError_t launch_dprob_combine(const float* slots, const int32_t* row_src, int R, int S, float* dprob,
                                 cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const bool v4 = R % 4 == 0 && ((reinterpret_cast<uintptr_t>(slots) | reinterpret_cast<uintptr_t>(row_src)) & 15) == 0;
  if (v4) {
    const unsigned grid = unsigned((R / 4 + 255) / 256);
    const FpFuse f{};
    switch (S) {
      case 1: return launch_chained(dprob_combine_v4_kernel<1, false>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
      case 2: return launch_chained(dprob_combine_v4_kernel<2, false>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
      case 16: return launch_chained(dprob_combine_v4_kernel<16, false>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
      default: return launch_chained(dprob_combine_v4_kernel<0, false>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
    }
  }
  const unsigned grid = unsigned((R + 255) / 256);
  switch (S) {
    case 1: return launch_chained(dprob_combine_kernel<1>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
    case 2: return launch_chained(dprob_combine_kernel<2>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
    case 16: return launch_chained(dprob_combine_kernel<16>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
    default: return launch_chained(dprob_combine_kernel<0>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
  }
}

cudaError_t launch_dprob_combine_fp(const float* slots, const int32_t* row_src, int R, int S, float* dprob,
                                    size_t chunk_bytes, unsigned long long* fp_acc, int* fp_done,
                                    uint64_t* src_hash, uint64_t* dprob_hash, cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const size_t nbytes = size_t(R) * 4;
  const size_t nch = (nbytes + chunk_bytes - 1) / chunk_bytes;
  const bool v4 = R % 4 == 0 && ((reinterpret_cast<uintptr_t>(slots) | reinterpret_cast<uintptr_t>(row_src)) & 15) == 0;
  if (!v4 || nch > size_t(kFpMaxChunks) || chunk_bytes % 512 != 0 || chunk_bytes / 4 > 0x7FFFFFFFull) {
    // the combine, then a separate fingerprint pass over each buffer
    cudaError_t e = launch_dprob_combine(slots, row_src, R, S, dprob, stream);
    if (e == cudaSuccess) e = launch_fingerprint(row_src, nbytes, 4, 0, chunk_bytes, 0, src_hash, stream);
    if (e == cudaSuccess) e = launch_fingerprint(dprob, nbytes, 4, 0, chunk_bytes, 0, dprob_hash, stream);
    return e;
  }
  FpFuse f;
  f.acc = fp_acc;
  f.done = fp_done;
  f.src_hash = reinterpret_cast<unsigned long long*>(src_hash);
  f.dprob_hash = reinterpret_cast<unsigned long long*>(dprob_hash);
  f.chunk_words = int(chunk_bytes / 4);
  f.nch = int(nch);
  const unsigned grid = unsigned((R / 4 + 255) / 256);
  switch (S) {
    case 1: return launch_chained(dprob_combine_v4_kernel<1, true>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
    case 2: return launch_chained(dprob_combine_v4_kernel<2, true>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
    case 16: return launch_chained(dprob_combine_v4_kernel<16, true>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
    default: return launch_chained(dprob_combine_v4_kernel<0, true>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob, f);
  }
}

}  // namespace dmoe
