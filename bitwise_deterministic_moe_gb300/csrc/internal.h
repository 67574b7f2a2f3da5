// Host-side launchers shared between the kernel translation units and the
// C-ABI layer (api.cu).  All pointers are device pointers; validation of
// user arguments happens in api.cu before any launcher is called.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dmoe {

enum class GemmMode : int { kFwd = 0, kSlots = 1, kAtomic = 2, kSerial = 3 };

struct GemmArgs {
  const void* X;              // bf16 [R, K]
  const void* W;              // bf16 [E, N, K]
  const int32_t* offsets;     // [E+1]
  int R, E, K, N;
  void* out;                  // bf16 [R, N]
  const void* grad_out;       // bf16 [T, N]   (slots / atomic)
  const int32_t* row_src;     // [R]           (slots / atomic)
  int topk;
  float* slots;               // [S, R]        (slots)
  float* dprob;               // [T*topk]      (atomic, serial)
  int* wflags;                // serial: per (m-tile, row quarter) count of slots already added; zeroed
                              // by the launcher before each launch
  int* status;                // device status word (may be null: errors not recorded)
  int* sched;                 // 2 device ints, zero between launches: dynamic tile counter
  int num_ctas;               // 0 = one per SM
  int flags;                  // dmoe_launch.flags
};

cudaError_t launch_grouped_gemm(GemmMode mode, const GemmArgs& a, cudaStream_t stream);       // CTA pairs
cudaError_t launch_grouped_gemm_1sm(GemmMode mode, const GemmArgs& a, cudaStream_t stream);   // single CTAs

// block-scaled grouped GEMM (MXFP8 / NVFP4 operands) with the slot epilogue
struct BlockScaledArgs {
  int kind;                   // 0 = MXFP8 (E4M3 + E8M0 per 32), 1 = NVFP4 (packed E2M1 + E4M3 per 16 + tensor scale)
  const void* Xq;             // [R, K] codes (MXFP8) or [R, K/2] packed (NVFP4)
  const void* Xs;             // [R, K/32] or [R, K/16] scale bytes
  const void* Wq;             // [E*N, K] or [E*N, K/2]
  const void* Ws;             // [E*N, K/32] or [E*N, K/16]
  const float* s_enc_x;       // NVFP4 tensor scales (device fp32), else null
  const float* s_enc_w;
  const int32_t* offsets;     // [E+1]
  int R, E, K, N;
  void* out;                  // bf16 [R, N]
  const void* grad_out;       // bf16 [T, N]; null = forward only
  const int32_t* row_src;     // [R]
  int topk;
  float* slots;               // [N/128, R]
  int* status;
  int* sched;
  int num_ctas;
  int narrow;                 // MXFP8: one-slot tiles even when N allows two-slot ones
};
cudaError_t launch_grouped_gemm_block_scaled(const BlockScaledArgs& a, cudaStream_t stream);

// grouped-GEMM weight gradient: dW[e] (+)= dY_e^T X_e
struct WgradArgs {
  const void* X;              // bf16 [R, K]
  const void* dY;             // bf16 [R, N]
  const int32_t* offsets;     // [E+1]
  int R, E, K, N;
  float* dW;                  // fp32 [E, N, K]
  int accumulate;             // 0: overwrite, 1: add to the existing values
  int* status;
  int* sched;
  int num_ctas;
};
cudaError_t launch_grouped_wgrad(const WgradArgs& a, cudaStream_t stream);

// block-scaled encodings (n = elements, a multiple of the block)
cudaError_t launch_quantize_mxfp8(const void* x, long long n, void* vals, void* scales, cudaStream_t stream);
cudaError_t launch_quantize_nvfp4(const void* x, long long n, void* packed, void* scales, float* s_enc,
                                  unsigned int* amax_scratch, cudaStream_t stream);

// serialized-writer control: bytes of its per-(m-tile, row quarter) counters
size_t serial_flag_bytes(long long R, int E);

// routing
size_t routing_scratch_bytes(long long R, int E);
// done_counter: one int of the workspace, zero between calls (the last block of
// the block scan resets it)
cudaError_t launch_permute(const int32_t* topk_ids, long long R, int E, int32_t* offsets, int32_t* row_src,
                           int32_t* row_of, void* scratch, int* status, int* done_counter, cudaStream_t stream);

// dispatch gather and token combine (status may be null: errors not recorded)
cudaError_t launch_dispatch_gather(const void* hidden, const int32_t* row_src, int R, int topk, int H,
                                   void* x_perm, int* status, cudaStream_t stream);
cudaError_t launch_token_combine(const void* expert_out, const float* probs, const int32_t* row_of, int T,
                                 int topk, int N, int R, void* y, int* status, cudaStream_t stream);

// dprob (unfused epilogue and fixed-order combine)
cudaError_t launch_dprob_epilogue(const void* grad_out, const void* expert_out, const int32_t* offsets,
                                  const int32_t* row_src, int R, int E, int topk, int N, float* slots,
                                  int* status, cudaStream_t stream);
cudaError_t launch_dprob_combine(const float* slots, const int32_t* row_src, int R, int S, float* dprob,
                                 cudaStream_t stream);
// The combine plus the positional chunk fingerprints of row_src and dprob,
// taken inside the combine when each buffer has at most kFpMaxChunks chunks
// (accumulators and a finished-block counter in the workspace, left zero);
// otherwise the combine and two fingerprint launches.
constexpr int kFpMaxChunks = 6;
cudaError_t launch_dprob_combine_fp(const float* slots, const int32_t* row_src, int R, int S, float* dprob,
                                    size_t chunk_bytes, unsigned long long* fp_acc, int* fp_done,
                                    uint64_t* src_hash, uint64_t* dprob_hash, cudaStream_t stream);

// fingerprint
cudaError_t launch_fingerprint(const void* data, size_t nbytes, int elem_size, int xor_kind, size_t chunk_bytes,
                               int mode, uint64_t* chunk_hash, cudaStream_t stream);

int device_sm_count();

// One-time per-device setup of launchers, safe with several host threads and
// several GPUs in one process: the dynamic shared-memory limit of a kernel
// (set once per kernel and device), and a per-(key, device) cached integer
// (computed by `compute` on first use; a value <= 0 is not cached).
cudaError_t ensure_kernel_smem(const void* kernel, int bytes);
int cached_per_device(const void* key, int (*compute)());

}  // namespace dmoe
