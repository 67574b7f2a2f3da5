/*
 * dmoe.h -- C ABI of libdmoe.so: a bitwise-deterministic MoE grouped GEMM with
 * a fused routing-probability-gradient (dprob) epilogue, for GB300 (sm_103a).
 *
 * The operation (from "Trillion-Parameter Pretraining Goes Bitwise-
 * Deterministic: NVIDIA Cuts the Determinism Tax to About 2%", section
 * "Interpretation", and "NVIDIA fait passer le déterminisme bit à bit de
 * Megatron Core à 2432 GPU avec seulement 2% de surcoût", section
 * "Optimisation pour le Nemotron à mille milliards de paramètres"): in the
 * grouped-GEMM epilogue several N-tiles contribute to the same dprob[token];
 * accumulating them at one address makes the result depend on arrival order.
 * Instead each N-tile writes a private slot and the slots are combined in a
 * fixed order once all writers are done, so tiles still run in parallel and
 * the result is identical run to run.
 *
 * Notation: T tokens, topk experts per token, E experts, R = T*topk permuted
 * rows, K reduction (FFN intermediate) dim, N output (latent) dim, S =
 * ceil(N/128) private slots per row.  Row r of the permuted layout came from
 * the flat routing index row_src[r] = t*topk + j (token t, choice j).
 *
 * Conventions for every entry point:
 *  - Every pointer is a DEVICE pointer unless marked "host".  All memory is
 *    owned by the caller; the library never allocates or frees.  (The one
 *    exception is the fixed scratch array of moe_grouped_gemm_dprob_noalloc.)
 *  - Arrays are dense, row-major, contiguous.  bf16 arrays are passed as
 *    void* holding IEEE bfloat16 values.  X_perm, W, expert_out and grad_out
 *    must be 16-byte aligned (TMA and 16-byte vector access).
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).  The
 *    return value reports host-side validation and launch errors only.
 *    Errors found on the device (bad routing data, a wait that timed out)
 *    are written to the status word at the start of the workspace `ws` and
 *    read back with dmoe_read_status().
 *  - Results are bitwise identical for any num_ctas >= 1, any stream, and
 *    any number of concurrent calls on separate output buffers and separate
 *    workspaces.  A workspace holds the grouped GEMM's dynamic tile counter:
 *    calls that share one must be ordered on one stream.
 */
#ifndef DMOE_H_
#define DMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dmoe_stream_t;   /* a cudaStream_t */

typedef enum dmoe_status {
    DMOE_OK = 0,
    DMOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misalignment, R != T*topk */
    DMOE_ERR_UNSUPPORTED = 2,   /* shape outside the supported range (see each call) */
    DMOE_ERR_ROUTING = 3,       /* device: expert id outside [0,E) or offsets not a partition of [0,R) */
    DMOE_ERR_TIMEOUT = 4,       /* device: a pipeline wait exceeded its limit; outputs are undefined */
    DMOE_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
    DMOE_ERR_WORKSPACE = 6      /* workspace missing or smaller than the *_workspace_bytes query */
} dmoe_status;

/* Element type codes recorded in fingerprint headers. */
typedef enum dmoe_dtype {
    DMOE_U8 = 0, DMOE_I8 = 1, DMOE_I16 = 2, DMOE_I32 = 3, DMOE_I64 = 4,
    DMOE_F16 = 5, DMOE_BF16 = 6, DMOE_F32 = 7, DMOE_F64 = 8, DMOE_BOOL = 9,
    DMOE_U16 = 10, DMOE_U32 = 11, DMOE_U64 = 12
} dmoe_dtype;

/* Launch options of the grouped GEMM.  num_ctas = persistent CTAs (0 = as
 * many as can be resident); any value gives the same bits.  Two kernels
 * implement every call and give bitwise identical results: one SM per
 * 128x256 tile, or CTA pairs (2-SM tensor-core MMA) per 256x256 tile, chosen
 * by default from the mean rows per expert (pairs when R >= 512*E).  On the
 * pair kernel an odd num_ctas is rounded down to even (minimum 2) and capped
 * at the resident count.  flags, OR-ed:
 *   DMOE_LAUNCH_SINGLE_CTA  force the single-CTA kernel
 *   DMOE_LAUNCH_CTA_PAIRS   force the CTA-pair kernel
 *   DMOE_LAUNCH_NARROW_TILES  block-scaled MXFP8 calls: one-slot (128 x 128)
 *     tiles even where N allows two-slot (128 x 256) ones; same bits
 *   DMOE_LAUNCH_TEST_STALL  exercise the failure path: the first CTA arms one
 *     pipeline stage but never loads it, so the wait on it runs out (after a
 *     200 ms limit instead of the usual 2 s), the kernel records
 *     DMOE_ERR_TIMEOUT, unwinds and frees its tensor memory; outputs are
 *     then undefined and the context stays usable. */
typedef struct dmoe_launch {
    int num_ctas;
    int flags;
} dmoe_launch;
#define DMOE_LAUNCH_TEST_STALL 1
#define DMOE_LAUNCH_SINGLE_CTA 2
#define DMOE_LAUNCH_CTA_PAIRS 4
#define DMOE_LAUNCH_NARROW_TILES 8

/* Supported shapes of the grouped GEMM calls:
 *   1 <= E <= DMOE_MAX_EXPERTS, 8 <= K <= 65536 with K % 8 == 0,
 *   128 <= N <= 65536 with N % 128 == 0, 0 <= R < 2^31, E*N < 2^31. */
#define DMOE_MAX_EXPERTS 1024
#define DMOE_SLOT_COLS 128          /* columns per private dprob slot */
#define DMOE_WS_STATUS_BYTES 256    /* status word region at the start of ws */

const char* dmoe_status_string(int status);
int dmoe_version(void);

/* Workspace needed by every call below for a problem with T tokens, topk
 * choices and E experts (status word, the grouped GEMM's tile counters, and
 * routing scratch, which the serialized-writer control reuses for its turn
 * counters).  The caller allocates it once, ZERO-FILLED, and may reuse
 * it for every call on that problem size; every call leaves the counters at
 * zero.  Calls that share a workspace must be ordered on one stream. */
size_t dmoe_workspace_bytes(int T, int topk, int E);

/* Reads (synchronising `stream`) and clears the device status word in ws.
 * Returns DMOE_OK or the first device-side error recorded since the last read. */
dmoe_status dmoe_read_status(void* ws, dmoe_stream_t stream);

/*
 * Routing indices: a deterministic permutation of the R routed (token, choice)
 * entries into expert-contiguous rows.  Routing maps are order-sensitive data
 * ("NVIDIA fait passer ...", section "Méthodologie de débogage du
 * non-déterminisme"), so the order is fixed: expert ascending, and within an
 * expert the flat index t*topk+j ascending (a stable counting sort).
 *   topk_ids        int32 [T, topk], ids in [0, E) (duplicates allowed)
 *   expert_offsets  int32 [E+1] out: exclusive prefix of per-expert counts
 *   row_src         int32 [R]   out: flat index of each permuted row
 *   row_of          int32 [R]   out, optional (may be null): the inverse,
 *                   row_of[t*topk + j] = the row that holds (t, j), as used by
 *                   moe_token_combine
 * Positions come from per-block counts and prefix sums, never from atomic
 * position tickets.  An id outside [0,E) sets DMOE_ERR_ROUTING in ws; the
 * outputs are then undefined.  T*topk may be 0.
 */
dmoe_status dmoe_permute_indices(const int32_t* topk_ids, int T, int topk, int E,
                                 int32_t* expert_offsets, int32_t* row_src, int32_t* row_of,
                                 void* ws, size_t ws_bytes, dmoe_stream_t stream);

/*
 * Dispatch gather: the expert-permuted input rows from the token hidden
 * states, the step before the experts.  Every (token, choice) row is a copy:
 *     x_perm[r, :] = hidden[row_src[r] / topk, :]        (bits unchanged)
 * Dispatch outputs are order-sensitive data ("NVIDIA fait passer ...",
 * section "Méthodologie de débogage du non-déterminisme"); the row order is
 * the fixed one of dmoe_permute_indices, so x_perm is identical run to run.
 *   hidden   bf16 [T, H]      (any 2-byte type: only bits are moved)
 *   row_src  int32 [T*topk]   from dmoe_permute_indices
 *   x_perm   bf16 [T*topk, H] out
 * H % 8 == 0, H <= 65536 (16-byte rows); hidden and x_perm 16-byte aligned.
 * ws: null, or a workspace of at least DMOE_WS_STATUS_BYTES whose status word
 * receives DMOE_ERR_ROUTING for a row_src entry outside [0, T*topk) (that
 * row is then left unwritten).  T may be 0.
 */
dmoe_status moe_dispatch_gather(const void* hidden, const int32_t* row_src, int T, int topk, int H,
                                void* x_perm, void* ws, size_t ws_bytes, dmoe_stream_t stream);

/*
 * Token combine: each token's output is the routing-probability-weighted sum
 * of its expert output rows, the step after the experts and the function
 * whose derivative with respect to prob is dprob ("Trillion-Parameter
 * Pretraining ...", section "Interpretation"):
 *     y[t, n] = bf16_rn( sum_{j = 0..topk-1} prob[t, j] * expert_out[row_of[t*topk + j], n] )
 * accumulated in fp32 as a fused multiply-add chain from +0 in ascending j,
 * then rounded once to bf16 (nearest even).  One thread owns each output
 * vector, so the bits never depend on the grid or on scheduling.
 *   expert_out  bf16 [T*topk, N]   permuted rows (moe_grouped_gemm_* output)
 *   probs       fp32 [T, topk]
 *   row_of      int32 [T*topk]     from dmoe_permute_indices
 *   y           bf16 [T, N]        out
 * N % 8 == 0, N <= 65536, topk <= DMOE_COMBINE_MAX_TOPK; expert_out and y
 * 16-byte aligned.  ws as for moe_dispatch_gather: a row_of entry outside
 * [0, T*topk) records DMOE_ERR_ROUTING and that term is dropped.
 */
#define DMOE_COMBINE_MAX_TOPK 64
dmoe_status moe_token_combine(const void* expert_out, const float* probs, const int32_t* row_of,
                              int T, int topk, int N, void* y, void* ws, size_t ws_bytes,
                              dmoe_stream_t stream);

/*
 * Grouped GEMM (FFN-out projection into the latent dim): for every expert e
 * and permuted row r in [off[e], off[e+1]):
 *     expert_out[r, n] = bf16_rn( sum_c X_perm[r, c] * W[e, n, c] )
 * fp32 accumulation on the tensor cores, one rounding to bf16 (nearest even).
 *   X_perm          bf16 [R, K]       rows in expert-permuted order
 *   W               bf16 [E, N, K]    per-expert weight, K contiguous
 *   expert_offsets  int32 [E+1]       off[0] = 0, non-decreasing, off[E] = R
 *   expert_out      bf16 [R, N]       out
 * Offsets that are not a partition of [0,R) set DMOE_ERR_ROUTING and skip the
 * GEMM.  ws: at least DMOE_WS_STATUS_BYTES bytes.
 */
dmoe_status moe_grouped_gemm_fwd(const void* X_perm, const void* W, const int32_t* expert_offsets,
                                 int R, int E, int K, int N, void* expert_out,
                                 const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                 dmoe_stream_t stream);

/*
 * Grouped GEMM with the fused private-slot dprob epilogue and the fixed-order
 * combine (the deterministic path).  Besides expert_out as above:
 *     slots[s, r] = sum over the 128 columns n of slot s of
 *                   float(grad_out[t(r), n]) * float(expert_out[r, n])
 * using the STORED bf16 expert_out value, summed in this fixed tree: the
 * slot's 16 groups of 8 columns are split into four parts k = g mod 4; part k
 * keeps eight fp32 partials a_j = sum over its groups g = k, k+4, k+8, k+12
 * (ascending) of p[8g+j] (fused multiply-add from +0) and folds them as
 * L_k = ((a0+a1)+(a2+a3))+((a4+a5)+(a6+a7)); the slot value is
 * (L_0+L_1)+(L_2+L_3).  Each N-tile writes only its own slots.  Then, after
 * all writers are done,
 *     dprob[row_src[r]] = (((slots[0,r] + slots[1,r]) + slots[2,r]) + ...)
 * in ascending slot order, fp32.
 *   grad_out  bf16 [T, N]      gradient at the expert-combine output, by token
 *   row_src   int32 [R]        from dmoe_permute_indices
 *   slots     fp32 [S, R]      scratch owned by the caller (S = N/128)
 *   dprob     fp32 [T, topk]   out
 * R must equal T*topk.
 */
dmoe_status moe_grouped_gemm_dprob(const void* X_perm, const void* W, const int32_t* expert_offsets,
                                   int R, int E, int K, int N, void* expert_out,
                                   const void* grad_out, const int32_t* row_src, int T, int topk,
                                   float* slots, float* dprob,
                                   const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                   dmoe_stream_t stream);

/*
 * The deterministic path with the fingerprints of its order-sensitive data
 * ("NVIDIA fait passer ...", section "Méthodologie de débogage du
 * non-déterminisme": the routing map and the outputs are fingerprinted on the
 * GPU, chunk by chunk): moe_grouped_gemm_dprob, and in the same call the
 * mode-0 (positional, raw bits) chunk hashes of row_src and of dprob exactly
 * as dmoe_fingerprint computes them with the same chunk_bytes.  The combine
 * reads every row_src word and writes every dprob word, so it forms the hash
 * terms itself, with no further pass over memory, when each buffer (R*4
 * bytes) has at most 6 chunks and the combine takes its vectorised form
 * (R % 4 == 0, slots and row_src 16-byte aligned); otherwise the call runs a
 * fingerprint pass over each buffer after the combine.  The header hashes
 * (dtype, shape) are the caller's, as for dmoe_fingerprint.  If row_src is
 * not a permutation of [0, R) the dprob hash covers the values the combine
 * wrote, which may differ from the buffer's.
 *   chunk_bytes   > 0, a multiple of 512
 *   row_src_hash  uint64 [dmoe_fingerprint_num_chunks(R*4, chunk_bytes)] out
 *   dprob_hash    uint64 [dmoe_fingerprint_num_chunks(R*4, chunk_bytes)] out
 * The status region of ws holds the sums between the combine's blocks and is
 * left at zero, so calls sharing ws must be ordered on one stream (as for
 * every call).  Other arguments and errors as for moe_grouped_gemm_dprob.
 */
dmoe_status moe_grouped_gemm_dprob_fp(const void* X_perm, const void* W, const int32_t* expert_offsets,
                                      int R, int E, int K, int N, void* expert_out,
                                      const void* grad_out, const int32_t* row_src, int T, int topk,
                                      float* slots, float* dprob,
                                      size_t chunk_bytes, uint64_t* row_src_hash, uint64_t* dprob_hash,
                                      const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                      dmoe_stream_t stream);

/*
 * L2 residency of grad_out for the dprob epilogue.  Every grad_out row is
 * gathered by topk different tiles at different times while the weights and
 * expert_out stream through L2; the epilogue loads it with an L2 evict-last
 * policy, and such lines are kept resident only inside the context's
 * persisting-L2 set-aside, which is empty unless the process sets one.  This
 * host call sets it (cudaLimitPersistingL2CacheSize of the current device's
 * context) to `bytes` clamped to [0, min(the device maximum, L2 size / 2)]
 * and writes the value then in effect to *granted (may be null; the runtime
 * may round the request up to its own granularity).  Size it to
 * grad_out (T*N*2 bytes) once, before the calls; 0 releases it.  It is a
 * context-wide setting: it also takes up to that much L2 away from the
 * normal accesses of every other kernel of the process, and it ends with the
 * context.  No other call of this library changes it.  Results never depend
 * on it, only timing.  May synchronize the device.  DMOE_ERR_CUDA if a
 * runtime query or the setting is refused.
 */
dmoe_status dmoe_reserve_l2_persisting(size_t bytes, size_t* granted);

/*
 * The nondeterministic control (the original form the pages describe): the
 * same GEMM and per-slot partials, but every partial is added with an fp32
 * atomicAdd into dprob[row_src[r]] after the call zero-fills dprob on
 * `stream`.  The order of the additions depends on CTA scheduling, so the
 * low bits of dprob may differ run to run.  Kept only to measure the
 * determinism tax.
 */
dmoe_status moe_grouped_gemm_dprob_atomic(const void* X_perm, const void* W, const int32_t* expert_offsets,
                                          int R, int E, int K, int N, void* expert_out,
                                          const void* grad_out, const int32_t* row_src, int T, int topk,
                                          float* dprob,
                                          const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                          dmoe_stream_t stream);

/*
 * Grouped-GEMM weight gradient (the FFN-out projection's wgrad), deterministic:
 *     dW[e, n, c] = sum over rows r in [off[e], off[e+1]) of dY[r, n] * X_perm[r, c]
 * (accumulate = 1: dW[e, n, c] += that sum, one fp32 addition per element).
 * A weight-gradient path is one of the workloads whose determinism overhead
 * the pages measure ("Trillion-Parameter Pretraining ...", section
 * "Synopsis").  Every 128 x 256 output tile is reduced by one CTA over all of
 * its expert's rows, in ascending blocks of 64 rows, with fp32 accumulation on
 * the tensor cores: there are no split-K partials and no atomics, so the bits
 * do not depend on num_ctas, the stream or the schedule.  An expert without
 * rows gets dW[e] = 0 (unchanged when accumulating).
 *   X_perm          bf16 [R, K]      the forward GEMM's input rows
 *   dY              bf16 [R, N]      gradient at expert_out, same row order
 *   expert_offsets  int32 [E+1]      a partition of [0, R); otherwise
 *                                    DMOE_ERR_ROUTING and dW is left unwritten
 *   dW              fp32 [E, N, K]   out (16-byte aligned)
 * Shapes as for the forward GEMM: N % 128 == 0, K % 8 == 0, both <= 65536,
 * 1 <= E <= DMOE_MAX_EXPERTS.  launch->flags is ignored.
 */
dmoe_status moe_grouped_gemm_wgrad(const void* X_perm, const void* dY, const int32_t* expert_offsets,
                                   int R, int E, int K, int N, float* dW, int accumulate,
                                   const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                   dmoe_stream_t stream);

/*
 * The serialized-writer control: deterministic without private slots.  The
 * same GEMM and per-slot partials, but the writers of one row take turns:
 * slot s of a block of 32 rows is added into dprob only after slots
 * 0..s-1 of those rows have been (a counter per m-tile and row quarter in
 * the workspace, acquire/release ordered), so
 *     dprob[row_src[r]] = ((P[0,r] + P[1,r]) + P[2,r]) + ...
 * bitwise equal to moe_grouped_gemm_dprob, while the N-tiles of one m-tile
 * wait on one another instead of writing in parallel -- the parallelism the
 * pages say serialising gives up ("Trillion-Parameter Pretraining ...",
 * section "Interpretation").  Kept only as a timing point between the
 * atomic control and the private-slot path.
 *  - Always runs the single-CTA kernel (DMOE_LAUNCH_CTA_PAIRS is ignored).
 *  - Every tile is claimed from the workspace counter by a CTA already
 *    running, in n-tile-major order (n-tile 0 of every m-tile, then n-tile
 *    1, ...), so a writer only waits on earlier-claimed tiles held by running
 *    CTAs and the turns always advance, whatever num_ctas is.  (In the
 *    m-tile-major order of the other calls the turns convoy behind the tile
 *    queues; n-tile-major gives up the X-row reuse in L2 instead.)
 *  - Uses the workspace region after the status word (dmoe_workspace_bytes
 *    covers it) and zero-fills it on `stream` before the kernel.
 *  - A turn that does not come within the wait limit records
 *    DMOE_ERR_TIMEOUT; outputs are then undefined.
 */
dmoe_status moe_grouped_gemm_dprob_serial(const void* X_perm, const void* W, const int32_t* expert_offsets,
                                          int R, int E, int K, int N, void* expert_out,
                                          const void* grad_out, const int32_t* row_src, int T, int topk,
                                          float* dprob,
                                          const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                          dmoe_stream_t stream);

/*
 * No-allocation variant of moe_grouped_gemm_dprob.  The pages have no
 * counterpart; it exists for callers that cannot allocate device memory:
 * code hosted by another runtime that only hands it input and output buffers
 * (a plugin or custom-op interface with no allocation hook, an engine whose
 * memory is partitioned in advance) and latency-critical loops that must not
 * call cudaMalloc, which can synchronise the device.
 *
 * Same inputs, outputs and bits as moe_grouped_gemm_dprob, but the [S, R]
 * slot scratch lives in a fixed-size device array owned by the library
 * (DMOE_NOALLOC_MAX_SLOT_VALUES fp32 values = 16 MiB, held on every GPU that
 * loads the library until the process exits), and no workspace is taken.
 *  - S * R > DMOE_NOALLOC_MAX_SLOT_VALUES returns DMOE_ERR_UNSUPPORTED.
 *  - Allocates nothing: no cudaMalloc/cudaFree, no allocating library call.
 *  - The first call in each CUDA context (once per device, and again after
 *    cudaDeviceReset or under a context created by other code) looks up the
 *    array's device address (cudaGetSymbolAddress, with that device current)
 *    and caches it under the context's id; make that first call before any
 *    stream capture.
 *  - All calls share the one array and it keeps the last call's contents
 *    (nothing in it needs to start at zero); calls whose work overlaps on
 *    the GPU (other streams, other threads) race on it and on the GEMM's
 *    tile counters, and their outputs are undefined.  Each call clears those
 *    two counters on its stream (an 8-byte cudaMemsetAsync, no allocation)
 *    before its GEMM starts, so a race never affects later calls that are
 *    ordered on one stream.
 *  - Device-side errors (bad routing data, a timed-out wait) are not
 *    recorded; outputs are then undefined.  Use moe_grouped_gemm_dprob with a
 *    workspace to have them reported.
 */
#define DMOE_NOALLOC_MAX_SLOT_VALUES 4194304
dmoe_status moe_grouped_gemm_dprob_noalloc(const void* X_perm, const void* W, const int32_t* expert_offsets,
                                           int R, int E, int K, int N, void* expert_out,
                                           const void* grad_out, const int32_t* row_src, int T, int topk,
                                           float* dprob, const dmoe_launch* launch, dmoe_stream_t stream);

/*
 * Unfused private-slot epilogue: the slot partials of moe_grouped_gemm_dprob
 * computed from an expert_out already in memory, with the identical
 * arithmetic, so the result is bitwise equal to the fused epilogue's slots.
 *   grad_out bf16 [T,N], expert_out bf16 [R,N], expert_offsets int32 [E+1]
 *   (rows r >= off[E] are skipped), row_src int32 [R], slots fp32 [S,R] out.
 */
dmoe_status moe_dprob_epilogue(const void* grad_out, const void* expert_out, const int32_t* expert_offsets,
                               const int32_t* row_src, int R, int E, int T, int topk, int N,
                               float* slots, dmoe_stream_t stream);

/*
 * Fixed-order slot combine: dprob[row_src[r]] = sum of slots[0..S-1, r],
 * left to right in ascending s, fp32.  Bitwise equal to the combine inside
 * moe_grouped_gemm_dprob.
 *   slots fp32 [S, R], row_src int32 [R], dprob fp32 [T*topk] out (R == T*topk).
 */
dmoe_status moe_dprob_combine(const float* slots, const int32_t* row_src, int R, int S, int T, int topk,
                              float* dprob, dmoe_stream_t stream);

/*
 * Block-scaled low-precision encodings of a bf16 tensor [rows, cols]: the
 * MXFP8 / NVFP4 operand forms whose encoded values and scale buffers the pages
 * fingerprint ("NVIDIA fait passer ...", section "Méthodologie de débogage du
 * non-déterminisme").  Every byte is a function of its own block (and, for
 * NVFP4, of the tensor maximum, an order-independent reduction), computed with
 * round-to-nearest-even conversions, so the bytes are identical on every run;
 * fingerprint them with dmoe_fingerprint (dtype DMOE_U8).  Inputs are finite
 * bf16 values except where stated.
 *
 * MXFP8 (OCP Microscaling Formats v1.0): each run of 32 consecutive values of
 * a row shares one E8M0 scale X = 2^s, s = floor(log2(amax)) - 8, clamped to
 * s >= -127 (an all-zero block gets s = -127); elements are E4M3 codes of
 * v / X, nearest even, saturating at +-448.  A block holding a NaN or an
 * infinity gets scale 0xFF and elements 0x7F.
 *   values  uint8 [rows, cols]       E4M3 codes (16-byte aligned)
 *   scales  uint8 [rows, cols / 32]  biased exponents s + 127
 * cols % 32 == 0; x 16-byte aligned.
 */
dmoe_status dmoe_quantize_mxfp8(const void* x, int rows, int cols, uint8_t* values, uint8_t* scales,
                                dmoe_stream_t stream);

/*
 * NVFP4: 16-value blocks of E2M1 elements with an E4M3 block scale and an fp32
 * tensor scale, every step in binary32 in this order:
 *   S_enc = 2688 / max|x| over the tensor   (2688 = 448 * 6; 1 for an all-zero tensor)
 *   s_b   = E4M3((amax_b / 6) * S_enc)      per block, nearest even, saturating
 *   q_i   = E2M1((x_i * S_enc) / s_b)       nearest even, saturating at +-6; 0 if s_b == 0
 * Decoded value: q_i * s_b / S_enc.
 *   packed  uint8 [rows, cols / 2]   two codes per byte, element 2i in the low nibble (8-byte aligned)
 *   scales  uint8 [rows, cols / 16]  E4M3 codes
 *   s_enc   fp32 [1], device, out
 * cols % 16 == 0; x 16-byte aligned; ws: at least DMOE_WS_STATUS_BYTES + 4
 * bytes (the tensor maximum is reduced there).
 */
dmoe_status dmoe_quantize_nvfp4(const void* x, int rows, int cols, uint8_t* packed, uint8_t* scales, float* s_enc,
                                void* ws, size_t ws_bytes, dmoe_stream_t stream);

/*
 * Block-scaled grouped GEMM with the private-slot dprob epilogue: the expert
 * GEMM of moe_grouped_gemm_dprob with MXFP8 or NVFP4 operands, in the
 * encodings dmoe_quantize_mxfp8 / dmoe_quantize_nvfp4 produce ("NVIDIA fait
 * passer le déterminisme bit à bit de Megatron Core à 2432 GPU ...", section
 * "Méthodologie de débogage du non-déterminisme": MXFP8 and NVFP4 values and
 * scale buffers are part of the fingerprinted path; "Nemotron 3 Ultra 的 tech
 * report ...", NVFP4 pretraining section).
 *   expert_out[r, n] = bf16_rne( sum_c dec(X)[r, c] * dec(W[e])[n, c] )
 * for rows r of expert e, with dec the block-scaled decoding:
 *   MXFP8: dec = E4M3(code) * 2^(scale - 127), one E8M0 scale per 32 values
 *          of a row (scale 0xFF decodes to NaN);
 *   NVFP4: dec = E2M1(code) * E4M3(scale) / S_enc, one E4M3 scale per 16
 *          values, S_enc the operand's fp32 tensor scale.
 * When grad_out is given, the slots and dprob follow exactly as in
 * moe_grouped_gemm_dprob (128-column private slots from the stored bf16
 * output, fixed in-slot tree, fixed-order combine); grad_out == NULL computes
 * expert_out only (row_src, T, topk, slots and dprob are then ignored).
 *   MXFP8: X_q uint8 [R, K], X_scales uint8 [R, K/32], W_q uint8 [E, N, K],
 *          W_scales uint8 [E*N, K/32]; K % 512 == 0.
 *   NVFP4: X_packed uint8 [R, K/2] (element 2i in the low nibble), X_scales
 *          uint8 [R, K/16], X_s_enc fp32 [1] (device); W_packed uint8
 *          [E, N, K/2], W_scales uint8 [E*N, K/16], W_s_enc fp32 [1];
 *          K % 256 == 0.
 *   expert_offsets int32 [E+1], expert_out bf16 [R, N], grad_out bf16 [T, N],
 *   row_src int32 [R], slots fp32 [N/128, R], dprob fp32 [T, topk].
 * All pointers are device memory owned by the caller, operand and scale
 * arrays 16-byte aligned.  1 <= E <= DMOE_MAX_EXPERTS, N % 128 == 0,
 * K, N <= 65536, E * N < 2^31; other shapes return DMOE_ERR_UNSUPPORTED.
 * Accumulation is fp32 on the tensor cores in a fixed k order, so results
 * are bitwise identical for any num_ctas and any stream; device-side errors
 * (offsets, row_src) go to the workspace status word as in
 * moe_grouped_gemm_dprob.  Tiles run on single CTAs: MXFP8 with an even
 * number of 128-column slots (N % 256 == 0) uses 128 x 256 tiles (one
 * N = 256 MMA per step over both slots), otherwise 128 x 128; both give the
 * same bits, and launch->flags = DMOE_LAUNCH_NARROW_TILES forces 128 x 128.
 * Other flags are ignored.
 */
dmoe_status moe_grouped_gemm_dprob_mxfp8(const uint8_t* X_q, const uint8_t* X_scales, const uint8_t* W_q,
                                         const uint8_t* W_scales, const int32_t* expert_offsets, int R, int E, int K,
                                         int N, void* expert_out, const void* grad_out, const int32_t* row_src, int T,
                                         int topk, float* slots, float* dprob, const dmoe_launch* launch, void* ws,
                                         size_t ws_bytes, dmoe_stream_t stream);
dmoe_status moe_grouped_gemm_dprob_nvfp4(const uint8_t* X_packed, const uint8_t* X_scales, const float* X_s_enc,
                                         const uint8_t* W_packed, const uint8_t* W_scales, const float* W_s_enc,
                                         const int32_t* expert_offsets, int R, int E, int K, int N, void* expert_out,
                                         const void* grad_out, const int32_t* row_src, int T, int topk, float* slots,
                                         float* dprob, const dmoe_launch* launch, void* ws, size_t ws_bytes,
                                         dmoe_stream_t stream);

/*
 * Chunk-wise tensor fingerprint ("NVIDIA fait passer ...", section "Méthodologie
 * de débogage du non-déterminisme": fingerprints computed on the GPU, with
 * shape, dtype and element count recorded, chunk-wise for order-sensitive
 * data).  The bytes [0, nbytes) are cut into chunks of chunk_bytes (the last
 * may be shorter) and each chunk c gets one 64-bit hash in chunk_hash[c]:
 *   mode 0 (positional, raw bits): words w_i = little-endian uint32 at byte
 *     4i (tail zero-padded), i the word index in the whole buffer;
 *     acc = sum_i fmix32(w_i ^ (i * 0x9E3779B9 mod 2^32)) mod 2^64 over the chunk;
 *     chunk_hash[c] = sm64(acc ^ (c << 32) ^ chunk_length_in_bytes),
 *     fmix32 = MurmurHash3's finalizer, sm64 = splitmix64's output function.
 *   mode 1 (xor): xor over the chunk's elements widened to 64 bits (floats to
 *     binary64 bit patterns, signed ints sign-extended, unsigned zero-extended),
 *     the reduction torch.hash_tensor applies to a whole tensor.  NaN
 *     payloads are not specified.
 * header_hash (HOST out) = sm64 chain over (dtype, ndim, shape[0..ndim-1],
 *   numel, nbytes): h = sm64(dtype); h = sm64(h ^ v) for each v in order.
 *   data       device, any alignment (16-byte alignment takes the fast path)
 *   shape      HOST int64 [ndim]; nbytes must equal numel * element size
 *   chunk_bytes  > 0, multiple of 16
 *   chunk_hash uint64 [dmoe_fingerprint_num_chunks(nbytes, chunk_bytes)] out
 */
size_t dmoe_fingerprint_num_chunks(size_t nbytes, size_t chunk_bytes);
dmoe_status dmoe_fingerprint(const void* data, size_t nbytes, int dtype, int ndim, const int64_t* shape,
                             size_t chunk_bytes, int mode, uint64_t* chunk_hash, uint64_t* header_hash,
                             dmoe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DMOE_H_ */
