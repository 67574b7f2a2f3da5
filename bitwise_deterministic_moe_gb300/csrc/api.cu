// C ABI of libdmoe.so (declared in include/dmoe.h): argument validation on
// the host, then launches on the caller's stream.  The library allocates
// nothing; all memory, including the workspace, belongs to the caller.
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace dmoe {

int device_sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (int(cache.size()) <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

cudaError_t ensure_kernel_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& d : done)
    if (d.first == kernel && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(kernel, dev);
  return e;
}

int cached_per_device(const void* key, int (*compute)()) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<const void*, int>, int>> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& c : cache)
    if (c.first.first == key && c.first.second == dev) return c.second;
  const int v = compute();
  if (v > 0) cache.push_back({{key, dev}, v});
  return v;
}

namespace {

uint64_t sm64_host(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

int dtype_size(int dt) {
  switch (dt) {
    case DMOE_U8: case DMOE_I8: case DMOE_BOOL: return 1;
    case DMOE_I16: case DMOE_F16: case DMOE_BF16: case DMOE_U16: return 2;
    case DMOE_I32: case DMOE_F32: case DMOE_U32: return 4;
    case DMOE_I64: case DMOE_F64: case DMOE_U64: return 8;
    default: return 0;
  }
}

// widening rule of the xor mode: 0 zero-extend, 1 sign-extend, 2 f16, 3 bf16, 4 f32, 5 f64 (bits as is)
int xor_kind(int dt) {
  switch (dt) {
    case DMOE_I8: case DMOE_I16: case DMOE_I32: case DMOE_I64: return 1;
    case DMOE_F16: return 2;
    case DMOE_BF16: return 3;
    case DMOE_F32: return 4;
    case DMOE_F64: return 5;
    default: return 0;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

dmoe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DMOE_OK;
  return DMOE_ERR_CUDA;
}

// Workspace status region: status word at byte 0, the GEMM's dynamic tile
// counters (two ints, left at zero by every launch) at byte 64.
int* status_ptr(void* ws) { return static_cast<int*>(ws); }
int* sched_ptr(void* ws) { return reinterpret_cast<int*>(static_cast<char*>(ws) + 64); }
// the routing block scan's finished-block counter at byte 128
int* route_counter_ptr(void* ws) { return reinterpret_cast<int*>(static_cast<char*>(ws) + 128); }
// the fingerprinting combine's finished-block counter at byte 132 and its
// 2 * kFpMaxChunks uint64 accumulators at byte 160 (both left at zero)
int* fp_done_ptr(void* ws) { return reinterpret_cast<int*>(static_cast<char*>(ws) + 132); }
unsigned long long* fp_acc_ptr(void* ws) {
  return reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + 160);
}
static_assert(160 + 2 * kFpMaxChunks * 8 <= DMOE_WS_STATUS_BYTES, "status region layout");

dmoe_status check_gemm_shape(const void* X, const void* W, const int32_t* off, int R, int E, int K, int N,
                             const void* out, void* ws, size_t ws_bytes) {
  if (!W || !off) return DMOE_ERR_INVALID_ARG;
  if (R < 0 || E < 1 || K < 1 || N < 1) return DMOE_ERR_INVALID_ARG;
  if (R > 0 && (!X || !out)) return DMOE_ERR_INVALID_ARG;   // X_perm / expert_out may be null when R == 0
  if (!aligned16(X) || !aligned16(W) || !aligned16(out)) return DMOE_ERR_INVALID_ARG;
  if (E > DMOE_MAX_EXPERTS || K % 8 != 0 || K > 65536 || N % DMOE_SLOT_COLS != 0 || N > 65536)
    return DMOE_ERR_UNSUPPORTED;
  if ((long long)E * N >= (1ll << 31)) return DMOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < DMOE_WS_STATUS_BYTES) return DMOE_ERR_WORKSPACE;
  return DMOE_OK;
}

}  // namespace
}  // namespace dmoe

using namespace dmoe;

extern "C" {

const char* dmoe_status_string(int status) {
  switch (status) {
    case DMOE_OK: return "ok";
    case DMOE_ERR_INVALID_ARG: return "invalid argument";
    case DMOE_ERR_UNSUPPORTED: return "unsupported shape";
    case DMOE_ERR_ROUTING: return "invalid routing data (expert id or offsets)";
    case DMOE_ERR_TIMEOUT: return "device wait timed out";
    case DMOE_ERR_CUDA: return "CUDA error";
    case DMOE_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int dmoe_version(void) { return 10000; }

size_t dmoe_workspace_bytes(int T, int topk, int E) {
  if (T < 0 || topk < 0 || E < 1) return 0;
  // the region after the status word is the routing scratch, reused as the
  // serialized control's counters (calls sharing a workspace are ordered)
  const long long R = (long long)T * topk;
  size_t scratch = routing_scratch_bytes(R, E);
  const size_t flags = (serial_flag_bytes(R, E) + 255) & ~size_t(255);
  if (flags > scratch) scratch = flags;
  return DMOE_WS_STATUS_BYTES + scratch;
}

dmoe_status dmoe_read_status(void* ws, dmoe_stream_t stream) {
  if (!ws) return DMOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return DMOE_ERR_CUDA;
  if (v != 0) {
    e = cudaMemsetAsync(ws, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return DMOE_ERR_CUDA;
  }
  return static_cast<dmoe_status>(v);
}

dmoe_status dmoe_reserve_l2_persisting(size_t bytes, size_t* granted) {
  int dev = 0, max_persist = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_persist, cudaDevAttrMaxPersistingL2CacheSize, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
    cudaGetLastError();
    return DMOE_ERR_CUDA;
  }
  // at most half of L2: a larger set-aside starves the streamed operands
  size_t cap = size_t(l2) / 2;
  if (size_t(max_persist) < cap) cap = size_t(max_persist);
  const size_t want = bytes < cap ? bytes : cap;
  size_t now = 0;
  if (cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, want) != cudaSuccess ||
      cudaDeviceGetLimit(&now, cudaLimitPersistingL2CacheSize) != cudaSuccess) {
    cudaGetLastError();
    return DMOE_ERR_CUDA;
  }
  if (granted) *granted = now;
  return DMOE_OK;
}

dmoe_status dmoe_permute_indices(const int32_t* topk_ids, int T, int topk, int E, int32_t* expert_offsets,
                                 int32_t* row_src, int32_t* row_of, void* ws, size_t ws_bytes,
                                 dmoe_stream_t stream) {
  if (T < 0 || topk < 0 || E < 1 || !expert_offsets) return DMOE_ERR_INVALID_ARG;
  if (E > DMOE_MAX_EXPERTS) return DMOE_ERR_UNSUPPORTED;
  const long long R = (long long)T * topk;
  if (R >= (1ll << 31)) return DMOE_ERR_UNSUPPORTED;
  if (R > 0 && (!topk_ids || !row_src)) return DMOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < dmoe_workspace_bytes(T, topk, E)) return DMOE_ERR_WORKSPACE;
  void* scratch = static_cast<char*>(ws) + DMOE_WS_STATUS_BYTES;
  return cuda_status(launch_permute(topk_ids, R, E, expert_offsets, row_src, row_of, scratch, status_ptr(ws), route_counter_ptr(ws),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

dmoe_status moe_grouped_gemm_fwd(const void* X_perm, const void* W, const int32_t* expert_offsets, int R, int E,
                                 int K, int N, void* expert_out, const dmoe_launch* launch, void* ws,
                                 size_t ws_bytes, dmoe_stream_t stream) {
  dmoe_status st = check_gemm_shape(X_perm, W, expert_offsets, R, E, K, N, expert_out, ws, ws_bytes);
  if (st != DMOE_OK) return st;
  GemmArgs a{};
  a.X = X_perm; a.W = W; a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.out = expert_out;
  a.status = status_ptr(ws);
  a.sched = sched_ptr(ws);
  a.num_ctas = launch ? launch->num_ctas : 0;
  a.flags = launch ? launch->flags : 0;
  if (a.num_ctas < 0) return DMOE_ERR_INVALID_ARG;
  return cuda_status(launch_grouped_gemm(GemmMode::kFwd, a, reinterpret_cast<cudaStream_t>(stream)));
}

static dmoe_status check_dprob_args(const void* grad_out, const int32_t* row_src, int R, int T, int topk) {
  if (!grad_out || !row_src || T < 0 || topk < 1) return DMOE_ERR_INVALID_ARG;
  if ((long long)T * topk != R) return DMOE_ERR_INVALID_ARG;
  if (!aligned16(grad_out)) return DMOE_ERR_INVALID_ARG;
  return DMOE_OK;
}

dmoe_status moe_grouped_gemm_dprob(const void* X_perm, const void* W, const int32_t* expert_offsets, int R, int E,
                                   int K, int N, void* expert_out, const void* grad_out, const int32_t* row_src,
                                   int T, int topk, float* slots, float* dprob, const dmoe_launch* launch, void* ws,
                                   size_t ws_bytes, dmoe_stream_t stream) {
  dmoe_status st = check_gemm_shape(X_perm, W, expert_offsets, R, E, K, N, expert_out, ws, ws_bytes);
  if (st != DMOE_OK) return st;
  st = check_dprob_args(grad_out, row_src, R, T, topk);
  if (st != DMOE_OK) return st;
  if (!slots || !dprob) return DMOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmArgs a{};
  a.X = X_perm; a.W = W; a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.out = expert_out;
  a.grad_out = grad_out; a.row_src = row_src; a.topk = topk;
  a.slots = slots;
  a.status = status_ptr(ws);
  a.sched = sched_ptr(ws);
  a.num_ctas = launch ? launch->num_ctas : 0;
  a.flags = launch ? launch->flags : 0;
  if (a.num_ctas < 0) return DMOE_ERR_INVALID_ARG;
  cudaError_t e = launch_grouped_gemm(GemmMode::kSlots, a, s);
  if (e != cudaSuccess) return DMOE_ERR_CUDA;
  return cuda_status(launch_dprob_combine(slots, row_src, R, N / DMOE_SLOT_COLS, dprob, s));
}

dmoe_status moe_grouped_gemm_dprob_fp(const void* X_perm, const void* W, const int32_t* expert_offsets, int R,
                                      int E, int K, int N, void* expert_out, const void* grad_out,
                                      const int32_t* row_src, int T, int topk, float* slots, float* dprob,
                                      size_t chunk_bytes, uint64_t* row_src_hash, uint64_t* dprob_hash,
                                      const dmoe_launch* launch, void* ws, size_t ws_bytes, dmoe_stream_t stream) {
  dmoe_status st = check_gemm_shape(X_perm, W, expert_offsets, R, E, K, N, expert_out, ws, ws_bytes);
  if (st != DMOE_OK) return st;
  st = check_dprob_args(grad_out, row_src, R, T, topk);
  if (st != DMOE_OK) return st;
  if (!slots || !dprob) return DMOE_ERR_INVALID_ARG;
  if (chunk_bytes == 0 || chunk_bytes % 512 != 0) return DMOE_ERR_INVALID_ARG;
  if (R > 0 && (!row_src_hash || !dprob_hash)) return DMOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmArgs a{};
  a.X = X_perm; a.W = W; a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.out = expert_out;
  a.grad_out = grad_out; a.row_src = row_src; a.topk = topk;
  a.slots = slots;
  a.status = status_ptr(ws);
  a.sched = sched_ptr(ws);
  a.num_ctas = launch ? launch->num_ctas : 0;
  a.flags = launch ? launch->flags : 0;
  if (a.num_ctas < 0) return DMOE_ERR_INVALID_ARG;
  cudaError_t e = launch_grouped_gemm(GemmMode::kSlots, a, s);
  if (e != cudaSuccess) return DMOE_ERR_CUDA;
  return cuda_status(launch_dprob_combine_fp(slots, row_src, R, N / DMOE_SLOT_COLS, dprob, chunk_bytes,
                                             fp_acc_ptr(ws), fp_done_ptr(ws), row_src_hash, dprob_hash, s));
}

dmoe_status moe_grouped_gemm_dprob_atomic(const void* X_perm, const void* W, const int32_t* expert_offsets, int R,
                                          int E, int K, int N, void* expert_out, const void* grad_out,
                                          const int32_t* row_src, int T, int topk, float* dprob,
                                          const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                          dmoe_stream_t stream) {
  dmoe_status st = check_gemm_shape(X_perm, W, expert_offsets, R, E, K, N, expert_out, ws, ws_bytes);
  if (st != DMOE_OK) return st;
  st = check_dprob_args(grad_out, row_src, R, T, topk);
  if (st != DMOE_OK) return st;
  if (!dprob) return DMOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (R > 0) {
    cudaError_t e = cudaMemsetAsync(dprob, 0, size_t(R) * sizeof(float), s);
    if (e != cudaSuccess) return DMOE_ERR_CUDA;
  }
  GemmArgs a{};
  a.X = X_perm; a.W = W; a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.out = expert_out;
  a.grad_out = grad_out; a.row_src = row_src; a.topk = topk;
  a.dprob = dprob;
  a.status = status_ptr(ws);
  a.sched = sched_ptr(ws);
  a.num_ctas = launch ? launch->num_ctas : 0;
  a.flags = launch ? launch->flags : 0;
  if (a.num_ctas < 0) return DMOE_ERR_INVALID_ARG;
  return cuda_status(launch_grouped_gemm(GemmMode::kAtomic, a, s));
}

dmoe_status moe_grouped_gemm_dprob_serial(const void* X_perm, const void* W, const int32_t* expert_offsets, int R,
                                          int E, int K, int N, void* expert_out, const void* grad_out,
                                          const int32_t* row_src, int T, int topk, float* dprob,
                                          const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                          dmoe_stream_t stream) {
  dmoe_status st = check_gemm_shape(X_perm, W, expert_offsets, R, E, K, N, expert_out, ws, ws_bytes);
  if (st != DMOE_OK) return st;
  st = check_dprob_args(grad_out, row_src, R, T, topk);
  if (st != DMOE_OK) return st;
  if (!dprob) return DMOE_ERR_INVALID_ARG;
  const size_t fbytes = serial_flag_bytes(R, E);
  if (ws_bytes < DMOE_WS_STATUS_BYTES + fbytes) return DMOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* wflags = reinterpret_cast<int*>(static_cast<char*>(ws) + DMOE_WS_STATUS_BYTES);
  if (R > 0) {
    cudaError_t e = cudaMemsetAsync(wflags, 0, fbytes, s);
    if (e != cudaSuccess) return DMOE_ERR_CUDA;
  }
  GemmArgs a{};
  a.X = X_perm; a.W = W; a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.out = expert_out;
  a.grad_out = grad_out; a.row_src = row_src; a.topk = topk;
  a.dprob = dprob;
  a.wflags = wflags;
  a.status = status_ptr(ws);
  a.sched = sched_ptr(ws);
  a.num_ctas = launch ? launch->num_ctas : 0;
  a.flags = launch ? launch->flags : 0;
  if (a.num_ctas < 0) return DMOE_ERR_INVALID_ARG;
  return cuda_status(launch_grouped_gemm(GemmMode::kSerial, a, s));
}

dmoe_status moe_grouped_gemm_wgrad(const void* X_perm, const void* dY, const int32_t* expert_offsets, int R, int E,
                                   int K, int N, float* dW, int accumulate, const dmoe_launch* launch, void* ws,
                                   size_t ws_bytes, dmoe_stream_t stream) {
  if (!expert_offsets || !dW || R < 0 || E < 1 || K < 1 || N < 1) return DMOE_ERR_INVALID_ARG;
  if (R > 0 && (!X_perm || !dY)) return DMOE_ERR_INVALID_ARG;
  if (!aligned16(X_perm) || !aligned16(dY) || !aligned16(dW)) return DMOE_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return DMOE_ERR_INVALID_ARG;
  if (E > DMOE_MAX_EXPERTS || K % 8 != 0 || K > 65536 || N % DMOE_SLOT_COLS != 0 || N > 65536)
    return DMOE_ERR_UNSUPPORTED;
  if ((long long)E * N >= (1ll << 31)) return DMOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < DMOE_WS_STATUS_BYTES) return DMOE_ERR_WORKSPACE;
  WgradArgs a{};
  a.X = X_perm; a.dY = dY; a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.dW = dW;
  a.accumulate = accumulate;
  a.status = status_ptr(ws);
  a.sched = sched_ptr(ws);
  a.num_ctas = launch ? launch->num_ctas : 0;
  if (a.num_ctas < 0) return DMOE_ERR_INVALID_ARG;
  return cuda_status(launch_grouped_wgrad(a, reinterpret_cast<cudaStream_t>(stream)));
}

dmoe_status moe_dprob_epilogue(const void* grad_out, const void* expert_out, const int32_t* expert_offsets,
                               const int32_t* row_src, int R, int E, int T, int topk, int N, float* slots,
                               dmoe_stream_t stream) {
  if (!expert_out || !expert_offsets || !slots || R < 0 || E < 1 || N < 1) return DMOE_ERR_INVALID_ARG;
  dmoe_status st = check_dprob_args(grad_out, row_src, R, T, topk);
  if (st != DMOE_OK) return st;
  if (!aligned16(expert_out)) return DMOE_ERR_INVALID_ARG;
  if (E > DMOE_MAX_EXPERTS || N % DMOE_SLOT_COLS != 0) return DMOE_ERR_UNSUPPORTED;
  // no workspace argument: device-side routing errors are not reported here
  return cuda_status(launch_dprob_epilogue(grad_out, expert_out, expert_offsets, row_src, R, E, topk, N, slots,
                                           nullptr, reinterpret_cast<cudaStream_t>(stream)));
}

dmoe_status moe_dprob_combine(const float* slots, const int32_t* row_src, int R, int S, int T, int topk,
                              float* dprob, dmoe_stream_t stream) {
  if (!slots || !row_src || !dprob || R < 0 || S < 1 || T < 0 || topk < 1) return DMOE_ERR_INVALID_ARG;
  if ((long long)T * topk != R) return DMOE_ERR_INVALID_ARG;
  return cuda_status(launch_dprob_combine(slots, row_src, R, S, dprob, reinterpret_cast<cudaStream_t>(stream)));
}

dmoe_status moe_dispatch_gather(const void* hidden, const int32_t* row_src, int T, int topk, int H, void* x_perm,
                                void* ws, size_t ws_bytes, dmoe_stream_t stream) {
  if (T < 0 || topk < 1 || H < 1) return DMOE_ERR_INVALID_ARG;
  const long long R = (long long)T * topk;
  if (R >= (1ll << 31)) return DMOE_ERR_UNSUPPORTED;
  if (H % 8 != 0 || H > 65536) return DMOE_ERR_UNSUPPORTED;
  if (R > 0 && (!hidden || !row_src || !x_perm)) return DMOE_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(x_perm)) return DMOE_ERR_INVALID_ARG;
  if (ws && ws_bytes < DMOE_WS_STATUS_BYTES) return DMOE_ERR_WORKSPACE;
  return cuda_status(launch_dispatch_gather(hidden, row_src, int(R), topk, H, x_perm, ws ? status_ptr(ws) : nullptr,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

dmoe_status moe_token_combine(const void* expert_out, const float* probs, const int32_t* row_of, int T, int topk,
                              int N, void* y, void* ws, size_t ws_bytes, dmoe_stream_t stream) {
  if (T < 0 || topk < 1 || N < 1) return DMOE_ERR_INVALID_ARG;
  const long long R = (long long)T * topk;
  if (R >= (1ll << 31)) return DMOE_ERR_UNSUPPORTED;
  if (N % 8 != 0 || N > 65536 || topk > DMOE_COMBINE_MAX_TOPK) return DMOE_ERR_UNSUPPORTED;
  if (T > 0 && (!expert_out || !probs || !row_of || !y)) return DMOE_ERR_INVALID_ARG;
  if (!aligned16(expert_out) || !aligned16(y)) return DMOE_ERR_INVALID_ARG;
  if (ws && ws_bytes < DMOE_WS_STATUS_BYTES) return DMOE_ERR_WORKSPACE;
  return cuda_status(launch_token_combine(expert_out, probs, row_of, T, topk, N, int(R), y,
                                          ws ? status_ptr(ws) : nullptr, reinterpret_cast<cudaStream_t>(stream)));
}

dmoe_status dmoe_quantize_mxfp8(const void* x, int rows, int cols, uint8_t* values, uint8_t* scales,
                                dmoe_stream_t stream) {
  if (rows < 0 || cols < 0) return DMOE_ERR_INVALID_ARG;
  if (cols % 32 != 0) return DMOE_ERR_UNSUPPORTED;
  const long long n = (long long)rows * cols;
  if (n > 0 && (!x || !values || !scales)) return DMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(values)) return DMOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_mxfp8(x, n, values, scales, reinterpret_cast<cudaStream_t>(stream)));
}

dmoe_status dmoe_quantize_nvfp4(const void* x, int rows, int cols, uint8_t* packed, uint8_t* scales, float* s_enc,
                                void* ws, size_t ws_bytes, dmoe_stream_t stream) {
  if (rows < 0 || cols < 0 || !s_enc) return DMOE_ERR_INVALID_ARG;
  if (cols % 16 != 0) return DMOE_ERR_UNSUPPORTED;
  const long long n = (long long)rows * cols;
  if (n > 0 && (!x || !packed || !scales)) return DMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(packed) & 7) != 0) return DMOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < DMOE_WS_STATUS_BYTES + 4) return DMOE_ERR_WORKSPACE;
  unsigned int* scratch = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + DMOE_WS_STATUS_BYTES);
  return cuda_status(
      launch_quantize_nvfp4(x, n, packed, scales, s_enc, scratch, reinterpret_cast<cudaStream_t>(stream)));
}

// Block-scaled grouped GEMM (+ private-slot dprob when grad_out is given).
static dmoe_status block_scaled_call(int kind, const uint8_t* Xq, const uint8_t* Xs, const float* Xg,
                                     const uint8_t* Wq, const uint8_t* Ws, const float* Wg,
                                     const int32_t* expert_offsets, int R, int E, int K, int N, void* expert_out,
                                     const void* grad_out, const int32_t* row_src, int T, int topk, float* slots,
                                     float* dprob, const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                     dmoe_stream_t stream) {
  if (!Wq || !Ws || !expert_offsets) return DMOE_ERR_INVALID_ARG;
  if (R < 0 || E < 1 || K < 1 || N < 1) return DMOE_ERR_INVALID_ARG;
  if (R > 0 && (!Xq || !Xs || !expert_out)) return DMOE_ERR_INVALID_ARG;
  if (kind == 1 && (!Xg || !Wg)) return DMOE_ERR_INVALID_ARG;
  if (!aligned16(Xq) || !aligned16(Xs) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(expert_out))
    return DMOE_ERR_INVALID_ARG;
  const int kmul = kind == 0 ? 512 : 256;   // whole 16-byte scale rows for the tensor maps
  if (E > DMOE_MAX_EXPERTS || K % kmul != 0 || K > 65536 || N % DMOE_SLOT_COLS != 0 || N > 65536)
    return DMOE_ERR_UNSUPPORTED;
  if ((long long)E * N >= (1ll << 31)) return DMOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < DMOE_WS_STATUS_BYTES) return DMOE_ERR_WORKSPACE;
  if (launch && launch->num_ctas < 0) return DMOE_ERR_INVALID_ARG;
  if (grad_out) {
    dmoe_status st = check_dprob_args(grad_out, row_src, R, T, topk);
    if (st != DMOE_OK) return st;
    if (!slots || !dprob) return DMOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  BlockScaledArgs a{};
  a.kind = kind;
  a.Xq = Xq; a.Xs = Xs; a.Wq = Wq; a.Ws = Ws;
  a.s_enc_x = Xg; a.s_enc_w = Wg;
  a.offsets = expert_offsets;
  a.R = R; a.E = E; a.K = K; a.N = N;
  a.out = expert_out;
  a.grad_out = grad_out; a.row_src = row_src; a.topk = topk;
  a.slots = slots;
  a.status = status_ptr(ws);
  a.sched = sched_ptr(ws);
  a.num_ctas = launch ? launch->num_ctas : 0;
  a.narrow = (launch && (launch->flags & DMOE_LAUNCH_NARROW_TILES)) ? 1 : 0;
  if (launch_grouped_gemm_block_scaled(a, s) != cudaSuccess) return DMOE_ERR_CUDA;
  if (!grad_out) return DMOE_OK;
  return cuda_status(launch_dprob_combine(slots, row_src, R, N / DMOE_SLOT_COLS, dprob, s));
}

dmoe_status moe_grouped_gemm_dprob_mxfp8(const uint8_t* X_q, const uint8_t* X_scales, const uint8_t* W_q,
                                         const uint8_t* W_scales, const int32_t* expert_offsets, int R, int E, int K,
                                         int N, void* expert_out, const void* grad_out, const int32_t* row_src, int T,
                                         int topk, float* slots, float* dprob, const dmoe_launch* launch, void* ws,
                                         size_t ws_bytes, dmoe_stream_t stream) {
  return block_scaled_call(0, X_q, X_scales, nullptr, W_q, W_scales, nullptr, expert_offsets, R, E, K, N, expert_out,
                           grad_out, row_src, T, topk, slots, dprob, launch, ws, ws_bytes, stream);
}

dmoe_status moe_grouped_gemm_dprob_nvfp4(const uint8_t* X_packed, const uint8_t* X_scales, const float* X_s_enc,
                                         const uint8_t* W_packed, const uint8_t* W_scales, const float* W_s_enc,
                                         const int32_t* expert_offsets, int R, int E, int K, int N, void* expert_out,
                                         const void* grad_out, const int32_t* row_src, int T, int topk, float* slots,
                                         float* dprob, const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                         dmoe_stream_t stream) {
  return block_scaled_call(1, X_packed, X_scales, X_s_enc, W_packed, W_scales, W_s_enc, expert_offsets, R, E, K, N,
                           expert_out, grad_out, row_src, T, topk, slots, dprob, launch, ws, ws_bytes, stream);
}

size_t dmoe_fingerprint_num_chunks(size_t nbytes, size_t chunk_bytes) {
  if (chunk_bytes == 0) return 0;
  return (nbytes + chunk_bytes - 1) / chunk_bytes;
}

dmoe_status dmoe_fingerprint(const void* data, size_t nbytes, int dtype, int ndim, const int64_t* shape,
                             size_t chunk_bytes, int mode, uint64_t* chunk_hash, uint64_t* header_hash,
                             dmoe_stream_t stream) {
  const int es = dtype_size(dtype);
  if (es == 0 || ndim < 0 || (ndim > 0 && !shape) || !header_hash) return DMOE_ERR_INVALID_ARG;
  if (chunk_bytes == 0 || chunk_bytes % 16 != 0 || (mode != 0 && mode != 1)) return DMOE_ERR_INVALID_ARG;
  long long numel = 1;
  for (int d = 0; d < ndim; ++d) {
    if (shape[d] < 0) return DMOE_ERR_INVALID_ARG;
    numel *= shape[d];
  }
  if ((unsigned long long)numel * es != nbytes) return DMOE_ERR_INVALID_ARG;
  if (nbytes > 0 && (!data || !chunk_hash)) return DMOE_ERR_INVALID_ARG;
  if (mode == 1 && (reinterpret_cast<uintptr_t>(data) % es) != 0) return DMOE_ERR_INVALID_ARG;
  uint64_t h = sm64_host(uint64_t(dtype));
  h = sm64_host(h ^ uint64_t(ndim));
  for (int d = 0; d < ndim; ++d) h = sm64_host(h ^ uint64_t(shape[d]));
  h = sm64_host(h ^ uint64_t(numel));
  h = sm64_host(h ^ uint64_t(nbytes));
  *header_hash = h;
  return cuda_status(launch_fingerprint(data, nbytes, es, xor_kind(dtype), chunk_bytes, mode, chunk_hash,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
