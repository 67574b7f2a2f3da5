// Deterministic routing indices: a stable counting sort of the R = T*topk
// routed entries by expert id.
//
// Routing maps are order-sensitive data ("NVIDIA fait passer le déterminisme
// bit à bit de Megatron Core à 2432 GPU ...", section "Méthodologie de
// débogage du non-déterminisme"), so every position is derived from counts and
// prefix sums, never from atomic position tickets:
//   1. histogram: one warp per block of 1024 entries (all 32 loads per lane
//      issued up front) counts ids per expert (integer counts are
//      order-independent);
//   2. block scan: one warp per expert turns its per-block counts into
//      exclusive prefixes (within-expert rank base of each block);
//   3. expert scan: one CTA scans the per-expert totals into expert_offsets;
//   4. scatter: one warp per block walks its entries in order, 32 at a time;
//      entries with equal ids are ranked by lane (match.any) and a per-expert
//      running counter advances chunk by chunk, which keeps the sort stable.
//      The same store can write the inverse map row_of[i] = position, which
//      the token combine uses to find each (token, choice)'s row.
// Scratch: counts int32 [E][nblk] and totals int32 [E].
#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int kEntriesPerBlock = 1024;

__global__ void __launch_bounds__(32)
hist_kernel(const int32_t* __restrict__ ids, long long R, int E, int nblk, int32_t* __restrict__ counts,
            int* status) {
  pdl_begin();
  __shared__ int cnt[DMOE_MAX_EXPERTS];
  const int lane = threadIdx.x;
  const int b = blockIdx.x;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  // all 32 loads of this lane in flight at once (the block is latency-bound)
  const long long i0 = (long long)b * kEntriesPerBlock + lane;
  int v[kEntriesPerBlock / 32];
#pragma unroll
  for (int k = 0; k < kEntriesPerBlock / 32; ++k) {
    const long long i = i0 + 32ll * k;
    v[k] = (i < R) ? __ldg(ids + i) : 0;
  }
  __syncwarp();
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kEntriesPerBlock / 32; ++k) {
    if (i0 + 32ll * k >= R) continue;
    const int e = v[k];
    if (e < 0 || e >= E) {
      bad = true;
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  if (bad) record_error(status, DMOE_ERR_ROUTING);
  __syncwarp();
  for (int e = lane; e < E; e += 32) counts[(size_t)e * nblk + b] = cnt[e];
}

// One warp per expert: exclusive prefix over that expert's per-block counts.
__global__ void __launch_bounds__(256)
block_scan_kernel(int32_t* __restrict__ counts, int E, int nblk, int32_t* __restrict__ totals) {
  pdl_begin();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= E) return;
  int32_t* row = counts + (size_t)warp * nblk;
  int carry = 0;
  for (int b0 = 0; b0 < nblk; b0 += 32) {
    int i = b0 + lane;
    int v = (i < nblk) ? row[i] : 0;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += u;
    }
    if (i < nblk) row[i] = carry + x - v;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) totals[warp] = carry;
}

// Single CTA of 1024 threads: offsets[0..E] = exclusive scan of totals.
__global__ void __launch_bounds__(1024)
expert_scan_kernel(const int32_t* __restrict__ totals, int E, int32_t* __restrict__ offsets) {
  pdl_begin();
  __shared__ int wsum[32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  int v = (tid < E) ? totals[tid] : 0;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += u;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
    int y = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, y, d);
      if (lane >= d) y += u;
    }
    wsum[lane] = y - w;  // exclusive prefix of warp sums
  }
  __syncthreads();
  const int incl = x + wsum[warp];
  if (tid < E) offsets[tid] = incl - v;
  if (tid == E - 1) offsets[E] = incl;
}

__global__ void __launch_bounds__(32)
scatter_kernel(const int32_t* __restrict__ ids, long long R, int E, int nblk, const int32_t* __restrict__ counts,
               const int32_t* __restrict__ offsets, int32_t* __restrict__ row_src,
               int32_t* __restrict__ row_of) {
  pdl_begin();
  __shared__ int next[DMOE_MAX_EXPERTS];
  const int lane = threadIdx.x;
  const int b = blockIdx.x;
  const long long i0 = (long long)b * kEntriesPerBlock + lane;
  int v[kEntriesPerBlock / 32];
#pragma unroll
  for (int k = 0; k < kEntriesPerBlock / 32; ++k) {
    const long long i = i0 + 32ll * k;
    v[k] = (i < R) ? __ldg(ids + i) : -1;
  }
  for (int e = lane; e < E; e += 32) next[e] = offsets[e] + counts[(size_t)e * nblk + b];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int k = 0; k < kEntriesPerBlock / 32; ++k) {
    const long long i = i0 + 32ll * k;
    int e = v[k];
    const bool ok = e >= 0 && e < E;
    if (!ok) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    const int base = ok ? next[e] : 0;
    __syncwarp();
    if (ok) {
      row_src[base + rank] = (int32_t)i;
      if (row_of) row_of[i] = base + rank;
      if (rank == 0) next[e] = base + __popc(peers);
    }
    __syncwarp();
  }
}

}  // namespace

size_t routing_scratch_bytes(long long R, int E) {
  long long nblk = (R + kEntriesPerBlock - 1) / kEntriesPerBlock;
  size_t b = size_t(E) * size_t(nblk) * 4 + size_t(E) * 4;
  return (b + 255) & ~size_t(255);
}

cudaError_t launch_permute(const int32_t* topk_ids, long long R, int E, int32_t* offsets, int32_t* row_src,
                           int32_t* row_of, void* scratch, int* status, cudaStream_t stream) {
  const int nblk = int((R + kEntriesPerBlock - 1) / kEntriesPerBlock);
  int32_t* counts = static_cast<int32_t*>(scratch);
  int32_t* totals = counts + size_t(E) * nblk;
  cudaError_t e = cudaSuccess;
  if (nblk > 0) e = launch_chained(hist_kernel, dim3(nblk), dim3(32), 0, stream, topk_ids, R, E, nblk, counts, status);
  if (e == cudaSuccess)
    e = launch_chained(block_scan_kernel, dim3((E * 32 + 255) / 256), dim3(256), 0, stream, counts, E, nblk, totals);
  if (e == cudaSuccess) e = launch_chained(expert_scan_kernel, dim3(1), dim3(1024), 0, stream, totals, E, offsets);
  if (e == cudaSuccess && nblk > 0)
    e = launch_chained(scatter_kernel, dim3(nblk), dim3(32), 0, stream, topk_ids, R, E, nblk, counts, offsets,
                       row_src, row_of);
  return e;
}

}  // namespace dmoe
