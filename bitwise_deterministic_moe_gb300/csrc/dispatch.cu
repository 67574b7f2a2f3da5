// Dispatch gather and routing-probability-weighted token combine: the steps
// either side of the grouped GEMM.
//
//   gather:   x_perm[r, :] = hidden[row_src[r] / topk, :]          (bit copy)
//   combine:  y[t, n] = bf16_rn( sum_{j = 0..topk-1} prob[t, j] * expert_out[row_of[t*topk + j], n] )
//             fp32 fused multiply-add chain from +0, j ascending.
//
// dprob is the derivative of this combine with respect to prob ("Trillion-
// Parameter Pretraining Goes Bitwise-Deterministic: NVIDIA Cuts the
// Determinism Tax to About 2%", section "Interpretation").  Both kernels give
// every output element to exactly one thread, which sums in a fixed order, so
// the bits do not depend on the grid or on scheduling; routing maps and
// dispatch outputs are the order-sensitive data the pages fingerprint ("NVIDIA
// fait passer le déterminisme bit à bit de Megatron Core à 2432 GPU ...",
// section "Méthodologie de débogage du non-déterminisme").
//
// Both are HBM passes with 16-byte accesses:
//   gather  one warp per permuted row; hidden rows (read topk times) are kept
//           in L2 with an evict-last hint, x_perm is streamed out evict-first.
//   combine a group of warps per token; the token's topk row ids and weights
//           are staged in shared memory, then each thread keeps up to eight
//           16-byte row loads in flight and folds them in ascending j.
#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxTopkCombine = DMOE_COMBINE_MAX_TOPK;
constexpr int kVecPerLane = 8;   // 16-byte vectors in flight per lane

__global__ void __launch_bounds__(kThreads)
dispatch_gather_kernel(const uint4* __restrict__ hidden, const int32_t* __restrict__ row_src, int R, int topk,
                       int V, uint4* __restrict__ x_perm, int* status) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarps;
  const uint64_t keep = policy_evict_last();
  const uint64_t stream = policy_evict_first();
  const long long nsrc = (long long)R;   // flat routing indices live in [0, R)
  for (int r = warp; r < R; r += nwarps) {
    const int src = __ldg(row_src + r);
    if (src < 0 || src >= nsrc) {
      if (lane == 0) record_error(status, DMOE_ERR_ROUTING);
      continue;
    }
    const uint4* in = hidden + (size_t)(src / topk) * V;
    uint4* out = x_perm + (size_t)r * V;
    for (int c0 = 0; c0 < V; c0 += 32 * kVecPerLane) {
      uint4 v[kVecPerLane];
#pragma unroll
      for (int u = 0; u < kVecPerLane; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < V) v[u] = ldg_nc_v4_hint(in + c, keep);
      }
#pragma unroll
      for (int u = 0; u < kVecPerLane; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < V) stg_v4_hint(out + c, v[u], stream);
      }
    }
  }
}

// fp32 fused multiply-add of one weighted 8-column bf16 vector into acc.
__device__ __forceinline__ void weighted_accumulate8(float (&acc)[8], float p, const uint4& x) {
  acc[0] = __fmaf_rn(p, bf16lo(x.x), acc[0]);
  acc[1] = __fmaf_rn(p, bf16hi(x.x), acc[1]);
  acc[2] = __fmaf_rn(p, bf16lo(x.y), acc[2]);
  acc[3] = __fmaf_rn(p, bf16hi(x.y), acc[3]);
  acc[4] = __fmaf_rn(p, bf16lo(x.z), acc[4]);
  acc[5] = __fmaf_rn(p, bf16hi(x.z), acc[5]);
  acc[6] = __fmaf_rn(p, bf16lo(x.w), acc[6]);
  acc[7] = __fmaf_rn(p, bf16hi(x.w), acc[7]);
}

// WPT warps per token, kWarps / WPT tokens per block and loop iteration.
template <int WPT>
__global__ void __launch_bounds__(kThreads, 4)
token_combine_kernel(const uint4* __restrict__ expert_out, const float* __restrict__ probs,
                     const int32_t* __restrict__ row_of, int T, int topk, int V, int R, uint4* __restrict__ y,
                     int* status) {
  constexpr int GPB = kWarps / WPT;        // token groups per block
  constexpr int GT = 32 * WPT;             // threads per token group
  __shared__ int s_row[GPB][kMaxTopkCombine];
  __shared__ float s_p[GPB][kMaxTopkCombine];
  pdl_begin();
  const uint64_t stream = policy_evict_first();
  const int g = threadIdx.x / GT;
  const int gt = threadIdx.x % GT;
  const int per_iter = gridDim.x * GPB;
  const int iters = (T + per_iter - 1) / per_iter;
  for (int it = 0; it < iters; ++it) {
    const int t0 = (it * gridDim.x + blockIdx.x) * GPB;
    for (int i = threadIdx.x; i < GPB * topk; i += kThreads) {
      const int gg = i / topk, j = i % topk;
      const int t = t0 + gg;
      int r = -1;
      float p = 0.f;
      if (t < T) {
        const size_t f = (size_t)t * topk + j;
        r = __ldg(row_of + f);
        p = __ldg(probs + f);
        if (r < 0 || r >= R) {
          record_error(status, DMOE_ERR_ROUTING);
          r = -1;
        }
      }
      s_row[gg][j] = r;
      s_p[gg][j] = p;
    }
    __syncthreads();
    const int t = t0 + g;
    if (t < T) {
      for (int c = gt; c < V; c += GT) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
        for (int j0 = 0; j0 < topk; j0 += kVecPerLane) {
          uint4 x[kVecPerLane];
#pragma unroll
          for (int u = 0; u < kVecPerLane; ++u) {
            const int j = j0 + u;
            const int r = (j < topk) ? s_row[g][j] : -1;
            if (r >= 0) x[u] = ldg_nc_v4_hint(expert_out + (size_t)r * V + c, stream);
          }
#pragma unroll
          for (int u = 0; u < kVecPerLane; ++u) {
            const int j = j0 + u;
            if (j < topk && s_row[g][j] >= 0) weighted_accumulate8(acc, s_p[g][j], x[u]);
          }
        }
        uint4 o;
        o.x = pack_bf16x2_rn(acc[0], acc[1]);
        o.y = pack_bf16x2_rn(acc[2], acc[3]);
        o.z = pack_bf16x2_rn(acc[4], acc[5]);
        o.w = pack_bf16x2_rn(acc[6], acc[7]);
        y[(size_t)t * V + c] = o;
      }
    }
    __syncthreads();
  }
}

int blocks_for(long long work_blocks) {
  const long long cap = (long long)device_sm_count() * 8;
  long long b = work_blocks < cap ? work_blocks : cap;
  return int(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_dispatch_gather(const void* hidden, const int32_t* row_src, int R, int topk, int H,
                                   void* x_perm, int* status, cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const int V = H / 8;
  const int grid = blocks_for((R + kWarps - 1) / kWarps);
  return launch_chained(dispatch_gather_kernel, dim3(grid), dim3(kThreads), 0, stream,
                        static_cast<const uint4*>(hidden), row_src, R, topk, V, static_cast<uint4*>(x_perm),
                        status);
}

cudaError_t launch_token_combine(const void* expert_out, const float* probs, const int32_t* row_of, int T,
                                 int topk, int N, int R, void* y, int* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (topk > kMaxTopkCombine) return cudaErrorInvalidValue;
  const int V = N / 8;
  const int warps_needed = (V + 31) / 32;
  const uint4* eo = static_cast<const uint4*>(expert_out);
  uint4* out = static_cast<uint4*>(y);
  if (warps_needed <= 1)
    return launch_chained(token_combine_kernel<1>, dim3(blocks_for((T + 7) / 8)), dim3(kThreads), 0, stream, eo,
                          probs, row_of, T, topk, V, R, out, status);
  if (warps_needed <= 2)
    return launch_chained(token_combine_kernel<2>, dim3(blocks_for((T + 3) / 4)), dim3(kThreads), 0, stream, eo,
                          probs, row_of, T, topk, V, R, out, status);
  if (warps_needed <= 4)
    return launch_chained(token_combine_kernel<4>, dim3(blocks_for((T + 1) / 2)), dim3(kThreads), 0, stream, eo,
                          probs, row_of, T, topk, V, R, out, status);
  return launch_chained(token_combine_kernel<8>, dim3(blocks_for(T)), dim3(kThreads), 0, stream, eo, probs, row_of,
                        T, topk, V, R, out, status);
}

}  // namespace dmoe
