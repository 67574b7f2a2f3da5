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
// ordered on one stream are fine.  Nothing in the slot array has to start at
// zero: each call writes every slot it later reads, and the array simply
// keeps the last call's contents.  The GEMM's two tile counters, which must
// start at zero, are cleared on the caller's stream before every launch, so
// an overlap that disturbed them cannot leak into later ordered calls.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

// 4 Mi fp32 slot values = 16 MiB: S * R <= 4,194,304 (e.g. R <= 262,144 rows at N = 2048).
constexpr size_t kNoallocSlotFloats = size_t(DMOE_NOALLOC_MAX_SLOT_VALUES);

static __device__ __align__(256) float g_noalloc_slots[kNoallocSlotFloats];
// the grouped GEMM's dynamic tile counters: zero at load, cleared on the
// caller's stream before every launch (and left at zero by every launch)
static __device__ __align__(256) int g_noalloc_sched[2];

// The CUDA context current on the calling thread, as a 64-bit id that is
// never reused within the process (cuCtxGetId), so an address cached for a
// context that was destroyed (cudaDeviceReset, a context created by other
// code) is never handed to a later one.  The driver entry points are looked
// up at run time, as the tensor-map encoder is.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

cudaError_t current_context_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_cur = []() -> CtxGetCurrentFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(ptr);
    return nullptr;
  }();
  static const CtxGetIdFn get_id = []() -> CtxGetIdFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetIdFn>(ptr);
    return nullptr;
  }();
  if (!get_cur || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device addresses of g_noalloc_slots and g_noalloc_sched in the current
// context.  In host code a __device__ array's name is only a host-side
// stand-in, so the real address is looked up (cudaGetSymbolAddress) the first
// time a context calls, with that context's device current, and cached under
// the context's id.  That first call may load the library's device code into
// the context, which is why it has to come before any stream capture.
cudaError_t noalloc_ptrs(float** slots_out, int** sched_out) {
  struct Entry {
    unsigned long long ctx;
    float* slots;
    int* sched;
  };
  constexpr int kEntries = 64;
  static std::mutex mu;
  static Entry cache[kEntries] = {};
  static int used = 0;
  unsigned long long ctx = 0;
  std::lock_guard<std::mutex> lock(mu);
  if (current_context_id(&ctx) == cudaSuccess) {
    for (int i = 0; i < used; ++i) {
      if (cache[i].ctx == ctx) {
        *slots_out = cache[i].slots;
        *sched_out = cache[i].sched;
        return cudaSuccess;
      }
    }
  }
  // set-up for this context: the runtime makes the current device's primary
  // context current here if no context is yet
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_slots);
  if (e != cudaSuccess) return e;
  void* q = nullptr;
  e = cudaGetSymbolAddress(&q, g_noalloc_sched);
  if (e != cudaSuccess) return e;
  e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  Entry ent{ctx, static_cast<float*>(p), static_cast<int*>(q)};
  if (used < kEntries) {
    cache[used++] = ent;
  } else {
    // more contexts than entries over the process's life: reuse the oldest
    for (int i = 1; i < kEntries; ++i) cache[i - 1] = cache[i];
    cache[kEntries - 1] = ent;
  }
  *slots_out = ent.slots;
  *sched_out = ent.sched;
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
  // The counters must be zero when the GEMM starts.  A finished launch leaves
  // them at zero, but two launches that overlapped on the GPU (a documented
  // misuse) can leave them off; clearing them here on the caller's stream
  // keeps such a race from skipping tiles in every later, ordered call.
  // cudaMemsetAsync allocates nothing.
  if (cudaMemsetAsync(sched, 0, 2 * sizeof(int), s) != cudaSuccess) return DMOE_ERR_CUDA;
  if (launch_grouped_gemm(GemmMode::kSlots, a, s) != cudaSuccess) return DMOE_ERR_CUDA;
  if (launch_dprob_combine(slots, row_src, R, S, dprob, s) != cudaSuccess) return DMOE_ERR_CUDA;
  return DMOE_OK;
}
