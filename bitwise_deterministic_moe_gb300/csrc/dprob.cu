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

// One thread per (row r, slot s), r fastest so the slot stores coalesce.
__global__ void __launch_bounds__(256)
dprob_epilogue_kernel(const uint16_t* __restrict__ grad_out, const uint16_t* __restrict__ expert_out,
                      const int32_t* __restrict__ offsets, const int32_t* __restrict__ row_src, int R, int E,
                      int topk, int N, int S, float* __restrict__ slots, int* status) {
  pdl_begin();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)R * S) return;
  const int s = int(idx / R);
  const int r = int(idx - (long long)s * R);
  const int rows = offsets[E];
  if (idx == 0 && rows != R) record_error(status, DMOE_ERR_ROUTING);
  if (r >= rows) return;
  const int src = row_src[r];
  if (unsigned(src) >= unsigned(R)) {
    record_error(status, DMOE_ERR_ROUTING);
    return;
  }
  const int tok = src / topk;
  const uint16_t* g = grad_out + size_t(tok) * N + size_t(s) * SLOT;
  const uint16_t* y = expert_out + size_t(r) * N + size_t(s) * SLOT;
  float part[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = 0.0f;
#pragma unroll
    for (int gi = k; gi < SLOT / 8; gi += 4) {
      const uint4 gv = ldg_nc_v4(g + gi * 8);
      const uint4 yv = ldg_nc_v4(y + gi * 8);
      slot_accumulate8(a, gv, yv);
    }
    part[k] = slot_tree(a);
  }
  slots[size_t(s) * R + r] = slot_parts(part[0], part[1], part[2], part[3]);
}

// One thread per permuted row: ascending-slot fp32 sum, scattered to dprob.
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

}  // namespace

cudaError_t launch_dprob_epilogue(const void* grad_out, const void* expert_out, const int32_t* offsets,
                                  const int32_t* row_src, int R, int E, int topk, int N, float* slots,
                                  int* status, cudaStream_t stream) {
  const int S = N / SLOT;
  const long long total = (long long)R * S;
  if (total == 0) return cudaSuccess;
  const unsigned grid = unsigned((total + 255) / 256);
  return launch_chained(dprob_epilogue_kernel, dim3(grid), dim3(256), 0, stream,
                        static_cast<const uint16_t*>(grad_out), static_cast<const uint16_t*>(expert_out), offsets,
                        row_src, R, E, topk, N, S, slots, status);
}

cudaError_t launch_dprob_combine(const float* slots, const int32_t* row_src, int R, int S, float* dprob,
                                 cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const unsigned grid = unsigned((R + 255) / 256);
  switch (S) {
    case 1: return launch_chained(dprob_combine_kernel<1>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
    case 2: return launch_chained(dprob_combine_kernel<2>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
    case 16: return launch_chained(dprob_combine_kernel<16>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
    default: return launch_chained(dprob_combine_kernel<0>, dim3(grid), dim3(256), 0, stream, slots, row_src, R, S, dprob);
  }
}

}  // namespace dmoe
