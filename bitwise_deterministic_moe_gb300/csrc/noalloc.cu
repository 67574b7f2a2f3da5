// moe_grouped_gemm_dprob_noalloc: the deterministic grouped GEMM + private-slot
// dprob path for callers that cannot allocate device memory.
//
// Who needs it: code hosted inside another runtime that hands it only its
// input and output buffers -- a plugin or custom-op interface with a fixed
// signature and no allocation hook, or an engine whose device memory is
// carved up in advance -- and latency-critical loops that must not call
// cudaMalloc (which can synchronise the device and take milliseconds).  Such a
// caller has nowhere to get the [S, R] fp32 slot buffer that
// moe_grouped_gemm_dprob takes as scratch.
//
// Here the slots live in one file-scope device array of fixed size that the
// library owns.  Every GPU that loads this library keeps that array for the
// life of the process.  All calls share it, so calls whose work overlaps on
// the GPU (different streams, or different host threads) race on it; calls
// ordered on one stream are fine.  Nothing in it has to start at zero: each
// call writes every slot it later reads, and the array simply keeps the last
// call's contents.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

// 4 Mi fp32 slot values = 16 MiB: S * R <= 4,194,304 (e.g. R <= 262,144 rows at N = 2048).
constexpr size_t kNoallocSlotFloats = size_t(DMOE_NOALLOC_MAX_SLOT_VALUES);

static __device__ __align__(256) float g_noalloc_slots[kNoallocSlotFloats];
// the grouped GEMM's dynamic tile counters; zero at load, left at zero by every launch
static __device__ __align__(256) int g_noalloc_sched[2];

// Device addresses of g_noalloc_slots and g_noalloc_sched for the current device.  In host code the
// symbol's name is only a host-side stand-in, so the real address is fetched
// once per device with that device current.
cudaError_t noalloc_ptrs(float** slots_out, int** sched_out) {
  static std::mutex mu;
  static float* ptrs[64] = {nullptr};
  static int* sched[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_slots);
    if (e != cudaSuccess) return e;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&q, g_noalloc_sched);
    if (e != cudaSuccess) return e;
    ptrs[dev] = static_cast<float*>(p);
    sched[dev] = static_cast<int*>(q);
  }
  *slots_out = ptrs[dev];
  *sched_out = sched[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dmoe

using namespace dmoe;

extern "C" dmoe_status moe_grouped_gemm_dprob_noalloc(const void* X_perm, const void* W,
                                                      const int32_t* expert_offsets, int R, int E, int K, int N,
                                                      void* expert_out, const void* grad_out,
                                                      const int32_t* row_src, int T, int topk, float* dprob,
                                                      const dmoe_launch* launch, dmoe_stream_t stream) {
  if (!W || !expert_offsets || !grad_out || !row_src || !dprob) return DMOE_ERR_INVALID_ARG;
  if (R < 0 || E < 1 || K < 1 || N < 1 || T < 0 || topk < 1) return DMOE_ERR_INVALID_ARG;
  if (R > 0 && (!X_perm || !expert_out)) return DMOE_ERR_INVALID_ARG;
  if ((long long)T * topk != R) return DMOE_ERR_INVALID_ARG;
  const uintptr_t align = reinterpret_cast<uintptr_t>(X_perm) | reinterpret_cast<uintptr_t>(W) |
                          reinterpret_cast<uintptr_t>(expert_out) | reinterpret_cast<uintptr_t>(grad_out);
  if (align & 15) return DMOE_ERR_INVALID_ARG;
  if (E > DMOE_MAX_EXPERTS || K % 8 != 0 || K > 65536 || N % DMOE_SLOT_COLS != 0 || N > 65536)
    return DMOE_ERR_UNSUPPORTED;
  if ((long long)E * N >= (1ll << 31)) return DMOE_ERR_UNSUPPORTED;
  const int S = N / DMOE_SLOT_COLS;
  if ((unsigned long long)S * (unsigned long long)R > kNoallocSlotFloats) return DMOE_ERR_UNSUPPORTED;
  if (launch && launch->num_ctas < 0) return DMOE_ERR_INVALID_ARG;

  float* slots = nullptr;
  int* sched = nullptr;
  if (noalloc_ptrs(&slots, &sched) != cudaSuccess) return DMOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmArgs a{};
  a.X = X_perm; a.W = W; a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.out = expert_out;
  a.grad_out = grad_out; a.row_src = row_src; a.topk = topk;
  a.slots = slots;
  a.status = nullptr;   // no caller workspace: device-side errors are not recorded
  a.sched = sched;
  a.num_ctas = launch ? launch->num_ctas : 0;
  a.flags = launch ? launch->flags : 0;
  if (launch_grouped_gemm(GemmMode::kSlots, a, s) != cudaSuccess) return DMOE_ERR_CUDA;
  if (launch_dprob_combine(slots, row_src, R, S, dprob, s) != cudaSuccess) return DMOE_ERR_CUDA;
  return DMOE_OK;
}
