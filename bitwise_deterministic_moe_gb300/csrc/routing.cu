// Deterministic routing indices: a stable counting sort of the R = T*topk
// routed entries by expert id.
//
// Routing maps are order-sensitive data ("NVIDIA fait passer le déterminisme
// bit à bit de Megatron Core à 2432 GPU ...", section "Méthodologie de
// débogage du non-déterminisme"), so every position is derived from counts and
// prefix sums, never from atomic position tickets:
//   1. histogram: one 1024-thread CTA per block of 1024 entries counts ids per
//      expert in shared memory (integer counts do not depend on the order of
//      the increments);
//   2. block scan: one warp per expert turns its per-block counts into
//      exclusive prefixes (within-expert rank base of each block), 256 blocks
//      per round with all loads in flight; the last
//      CTA to finish (a counter in the workspace, reset by that CTA) scans the
//      per-expert totals into expert_offsets;
//   3. scatter: the 32 warps of a CTA rank a block's 1024 entries at once --
//      match.any gives the rank among equal ids inside a warp, and an
//      exclusive scan over the warps of a [32 x E] shared table of per-warp
//      counts gives the entries of earlier warps -- so the sort is stable.
//      The same store can write the inverse map row_of[i] = position, which
//      the token combine uses to find each (token, choice)'s row.
// Scratch: counts int32 [E][nblk] and totals int32 [E].
#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int kEntriesPerBlock = 1024;   // = threads of the histogram and scatter CTAs
constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kEntriesPerBlock)
hist_kernel(const int32_t* __restrict__ ids, long long R, int E, int nblk, int32_t* __restrict__ counts,
            int* status) {
  __shared__ int cnt[DMOE_MAX_EXPERTS];
  pdl_begin();
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  for (int e = tid; e < E; e += kEntriesPerBlock) cnt[e] = 0;
  __syncthreads();
  const long long i = (long long)b * kEntriesPerBlock + tid;
  if (i < R) {
    const int e = __ldg(ids + i);
    if (e < 0 || e >= E) record_error(status, DMOE_ERR_ROUTING);
    else atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kEntriesPerBlock) counts[(size_t)e * nblk + b] = cnt[e];
}

// One warp per expert: exclusive prefix over that expert's per-block counts.
// The last CTA to finish then scans the totals into offsets[0..E].
__global__ void __launch_bounds__(kScanThreads)
block_scan_kernel(int32_t* __restrict__ counts, int E, int nblk, int32_t* __restrict__ totals,
                  int32_t* __restrict__ offsets, int* done_counter) {
  __shared__ int last_s;
  __shared__ int wsum[kScanThreads / 32];
  pdl_begin();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp < E) {
    // batches of 256 blocks: lane l owns blocks 8l..8l+7 of a batch, all
    // eight loads in flight before the warp scan of the lane sums
    int32_t* row = counts + (size_t)warp * nblk;
    int carry = 0;
    for (int b0 = 0; b0 < nblk; b0 += 256) {
      int v[8];
      int sum = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = b0 + lane * 8 + k;
        v[k] = (i < nblk) ? row[i] : 0;
        sum += v[k];
      }
      int x = sum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += u;
      }
      int run = carry + x - sum;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = b0 + lane * 8 + k;
        if (i < nblk) row[i] = run;
        run += v[k];
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) totals[warp] = carry;
  }
  // last CTA: offsets = exclusive scan of totals (E <= 1024 = 4 x 256)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last_s = atomicAdd(done_counter, 1) == int(gridDim.x) - 1;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  const int tid = threadIdx.x, w = tid >> 5;
  int v[4];
  int s = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = tid * 4 + k;
    v[k] = e < E ? __ldcg(totals + e) : 0;
    s += v[k];
  }
  int x = s;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += u;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  int run = x - s;
  for (int j = 0; j < w; ++j) run += wsum[j];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = tid * 4 + k;
    if (e < E) offsets[e] = run;
    run += v[k];
  }
  if (tid == kScanThreads - 1) offsets[E] = run;   // the last thread's running sum is the grand total
  if (tid == 0) *done_counter = 0;                 // every CTA has arrived: ready for the next call
}

// One 1024-thread CTA per block of 1024 entries; dynamic shared memory holds
// the per-warp counts table [32][E] and next[E].
__global__ void __launch_bounds__(kEntriesPerBlock)
scatter_kernel(const int32_t* __restrict__ ids, long long R, int E, int nblk, const int32_t* __restrict__ counts,
               const int32_t* __restrict__ offsets, int32_t* __restrict__ row_src, int32_t* __restrict__ row_of) {
  extern __shared__ int sm[];
  int* wcnt = sm;                       // [32][E]: entries of expert e in warp w, then the exclusive scan over w
  int* base = sm + 32 * E;              // [E]: first position of expert e's entries of this block
  pdl_begin();
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  for (int k = tid; k < 32 * E; k += kEntriesPerBlock) wcnt[k] = 0;
  for (int e = tid; e < E; e += kEntriesPerBlock) base[e] = __ldg(offsets + e) + counts[(size_t)e * nblk + b];
  __syncthreads();
  const long long i = (long long)b * kEntriesPerBlock + tid;
  int e = (i < R) ? __ldg(ids + i) : -1;
  if (e < 0 || e >= E) e = -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = tid; x < E; x += kEntriesPerBlock) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = wcnt[w * E + x];
      wcnt[w * E + x] = run;
      run += c;
    }
  }
  __syncthreads();
  if (e >= 0) {
    const int pos = base[e] + wcnt[warp * E + e] + rank;
    row_src[pos] = (int32_t)i;
    if (row_of) row_of[i] = pos;
  }
}

}  // namespace

size_t routing_scratch_bytes(long long R, int E) {
  long long nblk = (R + kEntriesPerBlock - 1) / kEntriesPerBlock;
  size_t b = size_t(E) * size_t(nblk) * 4 + size_t(E) * 4;
  return (b + 255) & ~size_t(255);
}

cudaError_t launch_permute(const int32_t* topk_ids, long long R, int E, int32_t* offsets, int32_t* row_src,
                           int32_t* row_of, void* scratch, int* status, int* done_counter, cudaStream_t stream) {
  const int nblk = int((R + kEntriesPerBlock - 1) / kEntriesPerBlock);
  int32_t* counts = static_cast<int32_t*>(scratch);
  int32_t* totals = counts + size_t(E) * nblk;
  cudaError_t e = cudaSuccess;
  if (nblk > 0)
    e = launch_chained(hist_kernel, dim3(nblk), dim3(kEntriesPerBlock), 0, stream, topk_ids, R, E, nblk, counts,
                       status);
  if (e == cudaSuccess)
    e = launch_chained(block_scan_kernel, dim3((E * 32 + kScanThreads - 1) / kScanThreads), dim3(kScanThreads), 0,
                       stream, counts, E, nblk, totals, offsets, done_counter);
  if (e == cudaSuccess && nblk > 0) {
    const size_t smem = size_t(33) * E * sizeof(int);
    if (smem > 48 * 1024) {
      e = ensure_kernel_smem(reinterpret_cast<const void*>(scatter_kernel), int(33 * DMOE_MAX_EXPERTS * sizeof(int)));
      if (e != cudaSuccess) return e;
    }
    e = launch_chained(scatter_kernel, dim3(nblk), dim3(kEntriesPerBlock), smem, stream, topk_ids, R, E, nblk,
                       counts, offsets, row_src, row_of);
  }
  return e;
}

}  // namespace dmoe
