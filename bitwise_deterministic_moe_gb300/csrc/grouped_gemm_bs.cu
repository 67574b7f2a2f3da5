// Block-scaled grouped GEMM with the private-slot dprob epilogue, for MXFP8
// and NVFP4 operands, on GB300 (sm_103a) tensor cores.
//
// The pages fingerprint MXFP8 and NVFP4 tensors -- encoded values and scale
// buffers -- in the MoE path ("NVIDIA fait passer le déterminisme bit à bit
// de Megatron Core à 2432 GPU ...", section "Méthodologie de débogage du
// non-déterminisme"), and the model they train runs its GEMMs in NVFP4
// ("Nemotron 3 Ultra 的 tech report ...", NVFP4 pretraining section).  This
// kernel consumes exactly the encodings dmoe_quantize_mxfp8 / _nvfp4 produce
// and computes the same expert GEMM and private-slot dprob as the bf16 path
// ("Trillion-Parameter Pretraining Goes Bitwise-Deterministic ...", section
// "Interpretation"): Y[r, n] = sum_c dec(X)[r, c] * dec(W[e])[n, c] with dec
// the block-scaled decoding, rounded once to bf16; each 128-column N-tile
// writes its own dprob slot with the bf16 path's fixed tree, and the slots
// are combined by the same fixed-order pass.
//
//   MXFP8: E4M3 codes, one E8M0 scale per 32 values of a row;
//          tcgen05.mma .kind::mxf8f6f4.block_scale.scale_vec::1X, K = 32 per MMA
//   NVFP4: packed E2M1 codes, one E4M3 scale per 16 values, one fp32 tensor
//          scale S_enc per operand (value = q * s / S_enc);
//          tcgen05.mma .kind::mxf4nvf4.block_scale.scale_vec::4X, K = 64 per
//          MMA, and the epilogue multiplies by 1 / (S_enc(X) * S_enc(W))
//
// Design (one CTA per SM, persistent, 384 threads), in the shape of the bf16
// single-CTA kernel with 128 x 128 tiles (one tile = one slot):
//   warp 0  TMA producer: per stage the A and B operand boxes (128 rows x 128
//           bytes, 128-byte swizzle) and two 128-row x 16-byte boxes of their
//           scale bytes.
//   warp 1  MMA issuer (one thread): copies the stage's scale blocks into
//           tensor memory (tcgen05.cp .32x128b.warpx4), then four block-scaled
//           MMAs; three fp32 accumulators in tensor memory.
//   warps 2-9  epilogue, two groups of four (one warp per TMEM lane quarter,
//           32 rows x 128 columns): the groups take alternate tiles, so two
//           tiles' epilogues (bf16 rounding, expert_out stores, the slot's dot
//           products) run while the next tile accumulates -- a tile is only
//           4 (NVFP4) or 8 (MXFP8) short stages at K = 1024.
//   warp 10 scale transposer: rearranges each stage's scale box into the
//           layout the tensor core reads -- the scale of operand row r sits
//           in tensor-memory lane r (A) or r mod 32 (B), column r / 32 -- as
//           32-row x 16-byte blocks whose word (j, c) is the scale of tile
//           row 32c + j.
//   warp 11 tile scheduler (expert tables in registers, decoded tiles queued
//           ahead of use).
// Each output element is produced by one tile with a fixed k order and a
// fixed epilogue tree, so results do not depend on the grid, the stream or
// the order in which tiles run.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tile_sched.cuh"

namespace dmoe {

bool make_tmap_2d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, uint64_t rows, uint64_t cols,
                  uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                  CUtensorMapL2promotion promotion);
bool make_tmap_bf16_store32(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t cols);

namespace {

constexpr int BM = 128;                       // rows per tile (UMMA M)
constexpr int BN = 128;                       // columns per tile (UMMA N) = one slot
constexpr int ROWB = 128;                     // operand bytes per row per stage (one swizzle row)
constexpr int A_BYTES = BM * ROWB;            // 16 KB
constexpr int B_BYTES = BN * ROWB;            // 16 KB
constexpr int SFBOX_BYTES = 128 * 16;         // TMA box of scale bytes: 128 rows x 16 bytes
constexpr int SFBLK_BYTES = 32 * 16;          // one .32x128b tcgen05.cp source: 32 rows x 16 bytes
constexpr int SF256_BYTES = 128 * 32;         // one .128x256b tcgen05.cp source: 128 rows x 32 bytes
constexpr int ACC_BUFS = 3;

constexpr int TMEM_COLS = 512;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_GROUPS = 2;
constexpr int EPI_WARPS = 4 * EPI_GROUPS;
constexpr int SF_WARP = EPI_WARP0 + EPI_WARPS;    // 10
constexpr int SCHED_WARP = SF_WARP + 1;           // 11
constexpr int NUM_THREADS = 32 * (SCHED_WARP + 1);
constexpr int SLOT = DMOE_SLOT_COLS;
constexpr int TQ = 4;
constexpr int HEAVY_MT = 3;
constexpr int STG_BYTES = 32 * 64;
static_assert(BN == SLOT, "one tile is one slot");

// Per-format layout: stage bytes (operands, the two scale boxes, the
// scale sources of the tensor-memory copies), the scale columns a stage
// takes in tensor memory, and the stage count that shared and tensor memory
// allow next to the accumulators.
//   MXFP8: one 32-row x 16-byte block per operand (one .32x128b.warpx4 copy
//          each, 4 columns; the four MMAs take the four bytes of a word).
//   NVFP4: two 128-row x 32-byte sources per operand (four .128x256b copies,
//          8 columns each; every MMA takes a whole word): 32 columns.  An
//          MMA's scale address must sit on a multiple of 4 columns, so the
//          four MMAs of a stage read A at columns 4 kk and B at 16 + 4 kk.
//   TW = 2 (MXFP8 only): a tile is two adjacent slots (128 x 256) -- one
//          256-row B box and one N = 256 MMA per 32-byte step over both
//          slots (fewer, wider MMAs keep the tensor pipe busier than two
//          N = 128 MMAs sharing the A box; each output element's sum is the
//          same), the B scales of the two halves in adjacent 4-column blocks
//          (row r at column r / 32 across them): 4 + 8 scale columns a stage
//          (16 with the 4-column alignment), one 256-column accumulator
//          pair, and four stages: the epilogue stores from registers, so it
//          needs no staging buffers.
// MXFP8 scale boxes live outside the stages, in a ring of two slots: a box
// holds 16 bytes of each row -- the words of four consecutive stages -- so it
// is loaded once per group of four stages, and the transposer, which frees
// the slot after the group's last stage, has three of the four stages' scale
// blocks written before their operands land.  NVFP4 boxes (one stage's four
// words) stay in the stage.
template <int KIND, int TW>
struct Layout {
  static_assert(TW == 1 || (TW == 2 && KIND == 0), "two-slot tiles are MXFP8 only");
  static constexpr bool BOX_RING = KIND == 0;
  static constexpr int OFF_B = A_BYTES;                  // B box of slot h at OFF_B + h * B_BYTES
  static constexpr int BOXES_BYTES = (1 + TW) * SFBOX_BYTES;   // the A box, then the B box (slot h at + h * SFBOX_BYTES)
  static constexpr int OFF_SFA_BOX = A_BYTES + TW * B_BYTES;   // in the stage (NVFP4) or a ring slot (MXFP8, offset 0)
  static constexpr int OFF_SFB_BOX = OFF_SFA_BOX + SFBOX_BYTES;
  static constexpr int OFF_SFA_BLK = A_BYTES + TW * B_BYTES + (BOX_RING ? 0 : BOXES_BYTES);
  static constexpr int SRC_BYTES = KIND == 0 ? SFBLK_BYTES : SF256_BYTES;
  static constexpr int OFF_SFB_BLK = OFF_SFA_BLK + (KIND == 0 ? 1 : 2) * SRC_BYTES;   // slot h at + h * SRC_BYTES
  static constexpr int STAGE_BYTES = ((OFF_SFB_BLK + TW * (KIND == 0 ? 1 : 2) * SRC_BYTES) + 1023) / 1024 * 1024;
  static constexpr int SF_COLS_STAGE = KIND == 0 ? (TW == 1 ? 8 : 16) : 32;
  static constexpr int STAGES = KIND == 0 ? (TW == 1 ? 5 : 4) : 4;
  static constexpr int ACC = TW == 1 ? ACC_BUFS : 1;     // accumulators (of TW slots each)
  static constexpr int SF0 = ACC * TW * BN;              // first scale column
  static_assert(SF0 + STAGES * SF_COLS_STAGE <= TMEM_COLS, "tensor memory");
  static constexpr int STAGING = TW == 1 ? EPI_WARPS * STG_BYTES : 0;   // per-warp TMA store staging
  static constexpr int OFF_RING = STAGES * STAGE_BYTES + STAGING;       // 1024-byte aligned
  static constexpr int RING_BYTES = BOX_RING ? 2 * BOXES_BYTES : 0;
  static_assert(OFF_RING % 1024 == 0 && BOXES_BYTES % 1024 == 0, "TMA box destinations");
  static constexpr size_t SMEM = 1024 + size_t(OFF_RING) + size_t(RING_BYTES) + 1024;
  static_assert(SMEM <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
};
constexpr int MAX_STAGES = 5;

enum Kind : int { kMxf8 = 0, kNvf4 = 1 };

struct alignas(16) Ctrl {
  uint64_t full[MAX_STAGES];   // operand bytes landed
  uint64_t sfin[MAX_STAGES];   // scale boxes landed
  uint64_t sfrdy[MAX_STAGES];  // scale blocks written by the transposer
  uint64_t empty[MAX_STAGES];  // the stage's MMAs and scale copies are done
  uint64_t bxfull[2];          // MXFP8: a ring slot's scale boxes landed
  uint64_t bxempty[2];         // MXFP8: the transposer is done with a ring slot
  uint64_t acc_full[ACC_BUFS];
  uint64_t acc_empty[ACC_BUFS];
  uint64_t mma_done;
  uint64_t tq_full[TQ];
  uint64_t tq_empty[TQ];
  QTile tq[TQ];
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(Ctrl) <= 1024, "control block");

struct KParams {
  const int32_t* offsets;
  int E, R, K, N, NT, KB;
  uint16_t* out;
  const uint16_t* grad_out;   // null: forward only
  const int32_t* row_src;
  int topk;
  float* slots;
  const float* s_enc_x;       // NVFP4 tensor scales (device)
  const float* s_enc_w;
  int* status;
  int* sched;
  unsigned long long wait_ns;
};

__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);      // start address >> 4
  d |= uint64_t(1) << 16;                       // leading byte offset (unused for swizzled K-major)
  d |= uint64_t(1024 >> 4) << 32;               // stride byte offset: 8 rows x 128 B
  d |= uint64_t(1) << 46;                       // descriptor version for tcgen05
  d |= uint64_t(2) << 61;                       // swizzle mode: 128-byte
  return d;
}

// A 32-row x 16-byte scale block in shared memory for tcgen05.cp: no swizzle,
// 8-row x 16-byte core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sfblk(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(128 >> 4) << 16;
  d |= uint64_t(128 >> 4) << 32;
  d |= uint64_t(1) << 46;
  return d;
}

// A 128-row x 32-byte source for tcgen05.cp .128x256b: no swizzle, 8-row x
// 16-byte core matrices; the two 16-byte halves of a row group 128 bytes
// apart (leading byte offset), row groups 256 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t smem_desc_sf256(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(128 >> 4) << 16;
  d |= uint64_t(256 >> 4) << 32;
  d |= uint64_t(1) << 46;
  return d;
}

// Byte offset of 32-bit word slot s (0..7) of row r in such a source.
__device__ __forceinline__ uint32_t sf256_word(int r, int s) {
  return uint32_t((r >> 3) * 256 + (s >> 2) * 128 + (r & 7) * 16 + (s & 3) * 4);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {   // i is a compile-time constant
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Instruction descriptor of the block-scaled kinds: B scale id (bits 4-5),
// A and B formats (7-9, 10-12), both K-major, N >> 3 (17-22), scale format
// (23: 1 = E8M0, 0 = E4M3), M >> 4 (24-28), A scale id (29-30).
template <int KIND, int N>
__device__ __forceinline__ uint32_t bs_idesc(uint32_t sf_id) {
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "UMMA N");
  constexpr uint32_t fmt = KIND == kMxf8 ? 0u : 1u;          // E4M3 in mxf8f6f4 / E2M1 in mxf4nvf4
  constexpr uint32_t sfmt = KIND == kMxf8 ? 1u : 0u;
  return (sf_id << 4) | (fmt << 7) | (fmt << 10) | (uint32_t(N >> 3) << 17) | (sfmt << 23) |
         (uint32_t(BM >> 4) << 24) | (sf_id << 29);
}

template <int KIND>
__device__ __forceinline__ void bs_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  if (KIND == kMxf8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  }
}

// 128 rows x 256 bits of shared memory into tensor-memory lanes 0..127 (row
// r to lane r), 8 columns from taddr.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 32 rows x 128 bits of shared memory into tensor-memory lanes 32w + j of
// the 4 columns at taddr, for each lane quarter w.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int KIND, int MODE, int TW>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                       const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                       const __grid_constant__ CUtensorMap tmap_o, const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = Layout<KIND, TW>;
  Ctrl& c = *reinterpret_cast<Ctrl*>(base + size_t(L::OFF_RING) + size_t(L::RING_BYTES));
  const uint32_t stage0 = smem_u32(base);
  const uint32_t ring0 = stage0 + uint32_t(L::OFF_RING);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;

  if (tid == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(smem_u32(&c.full[s]), 1);
      mbar_init(smem_u32(&c.sfin[s]), 1);
      mbar_init(smem_u32(&c.sfrdy[s]), 1);
      mbar_init(smem_u32(&c.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&c.bxfull[b]), 1);
      mbar_init(smem_u32(&c.bxempty[b]), 1);
    }
    for (int b = 0; b < L::ACC; ++b) {
      mbar_init(smem_u32(&c.acc_full[b]), 1);
      // the four warps of the group that took the tile (TW = 2: both groups, one slot each)
      mbar_init(smem_u32(&c.acc_empty[b]), 4 * TW);
    }
    mbar_init(smem_u32(&c.mma_done), 1);
    for (int i = 0; i < TQ; ++i) {
      mbar_init(smem_u32(&c.tq_full[i]), 1);
      mbar_init(smem_u32(&c.tq_empty[i]), 3 + EPI_WARPS);   // producer, transposer, MMA thread, epilogue warps
    }
    c.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_sfa);
    tma_prefetch_desc(&tmap_sfb);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  pdl_begin();   // no global memory is touched above this line
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int issued_total = 0;
      int groups_issued = 0;   // MXFP8 scale-box loads, two ring slots in turn
      int stage = 0;
      uint32_t ph = 0;
      for (int qi = 0;; ++qi) {
        const int qs = qi % TQ;
        if (!mbar_wait(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), &c.abort, p.status, p.wait_ns)) break;
        const QTile tl = c.tq[qs];
        mbar_arrive(smem_u32(&c.tq_empty[qs]));
        if (tl.cur < 0) break;
        const int brow = tl.e * p.N + tl.n0;
        bool ok = true;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(smem_u32(&c.empty[stage]), ph ^ 1u, &c.abort, p.status, p.wait_ns)) { ok = false; break; }
          // a group's ring slot is free once the transposer is done with the
          // group two back (waited for before anything is issued, so that the
          // drain below counts every copy in flight)
          if (L::BOX_RING && (kb & 3) == 0 &&
              !mbar_wait(smem_u32(&c.bxempty[groups_issued & 1]), uint32_t((groups_issued >> 1) & 1) ^ 1u, &c.abort,
                         p.status, p.wait_ns)) { ok = false; break; }
          const uint32_t sa = stage0 + stage * L::STAGE_BYTES;
          const uint32_t full = smem_u32(&c.full[stage]);
          const uint32_t sfin = smem_u32(&c.sfin[stage]);
          mbar_arrive_expect_tx(full, A_BYTES + TW * B_BYTES);
          tma_load_2d(sa, &tmap_a, full, kb * ROWB, tl.row0);
          // B (and below its scales): one box of TW * 128 rows -- the tensor
          // maps' box height -- whose slot-h half lands at + h * B_BYTES
          tma_load_2d(sa + L::OFF_B, &tmap_b, full, kb * ROWB, brow);
          // 16 bytes of scales per row: four stages' words (MXFP8, into a
          // ring slot once per group) or this stage's four (NVFP4)
          if (L::BOX_RING) {
            if ((kb & 3) == 0) {
              const int b = groups_issued & 1;
              const uint32_t slot = ring0 + uint32_t(b * L::BOXES_BYTES);
              const uint32_t bx = smem_u32(&c.bxfull[b]);
              mbar_arrive_expect_tx(bx, L::BOXES_BYTES);
              tma_load_2d(slot, &tmap_sfa, bx, 16 * (kb >> 2), tl.row0);
              tma_load_2d(slot + SFBOX_BYTES, &tmap_sfb, bx, 16 * (kb >> 2), brow);
              ++groups_issued;
            }
          } else {
            mbar_arrive_expect_tx(sfin, (1 + TW) * SFBOX_BYTES);
            tma_load_2d(sa + L::OFF_SFA_BOX, &tmap_sfa, sfin, 16 * kb, tl.row0);
            tma_load_2d(sa + L::OFF_SFB_BOX, &tmap_sfb, sfin, 16 * kb, brow);
          }
          ++issued_total;
          if (++stage == L::STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
      }
      // let every copy this thread started land before the CTA can exit
      for (int s = 0; s < L::STAGES; ++s) {
        const int n = (issued_total - s + L::STAGES - 1) / L::STAGES;
        if (n > 0) {
          mbar_wait_drain(smem_u32(&c.full[s]), uint32_t(n - 1) & 1u, p.wait_ns / 4);
          if (!L::BOX_RING) mbar_wait_drain(smem_u32(&c.sfin[s]), uint32_t(n - 1) & 1u, p.wait_ns / 4);
        }
      }
      if (L::BOX_RING) {
        for (int b = 0; b < 2; ++b) {
          const int n = (groups_issued - b + 1) / 2;
          if (n > 0) mbar_wait_drain(smem_u32(&c.bxfull[b]), uint32_t(n - 1) & 1u, p.wait_ns / 4);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      for (int qi = 0;; ++qi) {
        const int qs = qi % TQ;
        if (!mbar_wait(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), &c.abort, p.status, p.wait_ns)) break;
        const int cur = c.tq[qs].cur;
        mbar_arrive(smem_u32(&c.tq_empty[qs]));
        if (cur < 0) break;
        if (!mbar_wait(smem_u32(&c.acc_empty[acc]), aph ^ 1u, &c.abort, p.status, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * TW * BN);   // slot h at + h * BN
        bool ok = true;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(smem_u32(&c.full[stage]), ph, &c.abort, p.status, p.wait_ns)) { ok = false; break; }
          if (!mbar_wait(smem_u32(&c.sfrdy[stage]), ph, &c.abort, p.status, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = stage0 + stage * L::STAGE_BYTES;
          const uint32_t sfc = tmem_base + uint32_t(L::SF0 + stage * L::SF_COLS_STAGE);
          // scale sources -> tensor memory (ordered before the MMAs this thread issues next)
          if (KIND == kMxf8) {
            tmem_cp_32x128b_x4(sfc, smem_desc_sfblk(sa + L::OFF_SFA_BLK));
#pragma unroll
            for (int h = 0; h < TW; ++h)
              tmem_cp_32x128b_x4(sfc + 4u + 4u * uint32_t(h), smem_desc_sfblk(sa + L::OFF_SFB_BLK + h * SFBLK_BYTES));
          } else {
            tmem_cp_128x256b(sfc, smem_desc_sf256(sa + L::OFF_SFA_BLK));
            tmem_cp_128x256b(sfc + 8u, smem_desc_sf256(sa + L::OFF_SFA_BLK + SF256_BYTES));
            tmem_cp_128x256b(sfc + 16u, smem_desc_sf256(sa + L::OFF_SFB_BLK));
            tmem_cp_128x256b(sfc + 24u, smem_desc_sf256(sa + L::OFF_SFB_BLK + SF256_BYTES));
          }
          const uint64_t adesc = smem_desc_k128(sa);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // 32 bytes of each row per MMA: 32 E4M3 or 64 E2M1 values.  MXFP8:
            // byte kk of the stage's word (scale id); NVFP4: the word of MMA kk,
            // for tile row 32c + j at column 4 kk + c (A) or 16 + 4 kk + c (B)
            // of the stage's scale columns
            const uint32_t sfid = KIND == kMxf8 ? uint32_t(kk) : 0u;
            const uint32_t sfa = KIND == kMxf8 ? sfc : sfc + 4u * uint32_t(kk);
            // one MMA over the tile's TW slots: B rows 0 .. TW*128-1 (one box),
            // their scales in the columns from sfc + 4 (MXFP8) on, the
            // accumulators of the slots side by side
            const uint32_t sfb = KIND == kMxf8 ? sfc + 4u : sfc + 16u + 4u * uint32_t(kk);
            const uint64_t bdesc = smem_desc_k128(sa + L::OFF_B);
            bs_mma<KIND>(d_tmem, adesc + uint64_t(kk * 2), bdesc + uint64_t(kk * 2), bs_idesc<KIND, TW * BN>(sfid),
                         sfa, sfb, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&c.empty[stage]));
          if (++stage == L::STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(smem_u32(&c.acc_full[acc]));
        if (++acc == L::ACC) { acc = 0; aph ^= 1u; }
      }
      tc_commit(smem_u32(&c.mma_done));
      mbar_wait_drain(smem_u32(&c.mma_done), 0, p.wait_ns / 4);
    }
  } else if (warp == SF_WARP) {
    // -------------------------------------------------- scale transposer
    // Box row t holds the 16 scale bytes of tile row t (four 32-bit words).
    // MXFP8: block word (j, c) = this stage's word of tile row 32c + j, lane j
    //        writing block row j (one .32x128b.warpx4 copy per operand).
    // NVFP4: source h (of each operand) holds, in every 32-row quarter q,
    //        row 32q + j = at slot 4k' + c the word of MMA 2h + k' of tile row
    //        32c + j, so tensor-memory lane 32q + j, column 8h + 4k' + c holds
    //        the scale of tile row 32c + j for that MMA in every lane quarter,
    //        as the replicating .32x128b.warpx4 copy lays it out.  Lane j owns
    //        tile rows j, 32 + j, 64 + j, 96 + j.
    // MXFP8: the boxes of a group of four stages sit in ring slot g % 2; the
    // stage's block area is free once the stage's previous MMAs are done
    // (the producer's wait, on the same barrier), which is usually long
    // before the stage's operands land.
    int stage = 0;
    uint32_t ph = 0;
    int groups_done = 0;
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      if (!warp_wait(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), &c.abort, p.status, lane, p.wait_ns)) break;
      const int cur = c.tq[qs].cur;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.tq_empty[qs]));
      if (cur < 0) break;
      bool ok = true;
      for (int kb = 0; kb < p.KB; ++kb) {
        uint32_t boxes;
        if (L::BOX_RING) {
          const int b = groups_done & 1;
          if ((kb & 3) == 0 &&
              !warp_wait(smem_u32(&c.bxfull[b]), uint32_t((groups_done >> 1) & 1), &c.abort, p.status, lane,
                         p.wait_ns)) { ok = false; break; }
          if (!warp_wait(smem_u32(&c.empty[stage]), ph ^ 1u, &c.abort, p.status, lane, p.wait_ns)) { ok = false; break; }
          boxes = ring0 + uint32_t(b * L::BOXES_BYTES);
        } else {
          if (!warp_wait(smem_u32(&c.sfin[stage]), ph, &c.abort, p.status, lane, p.wait_ns)) { ok = false; break; }
          boxes = stage0 + stage * L::STAGE_BYTES + L::OFF_SFA_BOX;
        }
        const uint32_t sa = stage0 + stage * L::STAGE_BYTES;
#pragma unroll
        for (int op = 0; op < 1 + TW; ++op) {
          // op 0: A; op 1 + h: B of slot h
          const uint32_t box = boxes + (op == 0 ? 0u : uint32_t(SFBOX_BYTES + (op - 1) * SFBOX_BYTES));
          const uint32_t blk = sa + (op == 0 ? L::OFF_SFA_BLK : L::OFF_SFB_BLK + (op - 1) * L::SRC_BYTES);
          uint4 r[4];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) r[cc] = lds_v4(box + uint32_t((32 * cc + lane) * 16));
          if (KIND == kMxf8) {
            // this stage's word is word kb % 4 of the row's 16 bytes
            const int w = kb & 3;
            uint4 o;
            o.x = w == 0 ? r[0].x : w == 1 ? r[0].y : w == 2 ? r[0].z : r[0].w;
            o.y = w == 0 ? r[1].x : w == 1 ? r[1].y : w == 2 ? r[1].z : r[1].w;
            o.z = w == 0 ? r[2].x : w == 1 ? r[2].y : w == 2 ? r[2].z : r[2].w;
            o.w = w == 0 ? r[3].x : w == 1 ? r[3].y : w == 2 ? r[3].z : r[3].w;
            sts_v4(blk + uint32_t(lane * 16), o);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int kk = 2 * h + k2;
                const uint4 o = make_uint4(word_of(r[0], kk), word_of(r[1], kk), word_of(r[2], kk), word_of(r[3], kk));
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                  sts_v4(blk + uint32_t(h * SF256_BYTES) + sf256_word(32 * qq + lane, 4 * k2), o);
              }
          }
        }
        fence_proxy_async_smem();   // the generic-proxy block writes, before the tensor core's copy reads them
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c.sfrdy[stage]));
        if (L::BOX_RING && ((kb & 3) == 3 || kb == p.KB - 1)) {
          // every lane has read the group's boxes (the barrier above): the slot can be reloaded
          if (lane == 0) mbar_arrive(smem_u32(&c.bxempty[groups_done & 1]));
          ++groups_done;
        }
        if (++stage == L::STAGES) { stage = 0; ph ^= 1u; }
      }
      if (!ok) break;
    }
  } else if (warp == SCHED_WARP) {
    // -------------------------------------------------- tile scheduler
    ExpertTables tb;
    int units_heavy = 0, units_light = 0;
    const bool bad = build_tables<BM, HEAVY_MT>(tb, p.offsets, E, p.R, lane, units_heavy, units_light);
    if (bad && lane == 0) record_error(p.status, DMOE_ERR_ROUTING);
    const int units = units_heavy + units_light;
    const int total_tiles = bad ? 0 : units * p.NT;
    int tile = int(blockIdx.x);
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      const int cur = tile < total_tiles ? tile : -1;
      int nxt = 0;
      if (cur >= 0 && lane == 0) nxt = int(gridDim.x) + atomicAdd(p.sched, 1);
      QTile q{};
      q.cur = -1;
      if (cur >= 0) q = decode_tile_warp<BM, TW * BN>(cur, tb, E, p.NT, units_heavy, units, lane);
      if (!warp_wait(smem_u32(&c.tq_empty[qs]), uint32_t((qi / TQ) & 1) ^ 1u, &c.abort, p.status, lane, p.wait_ns))
        break;
      if (lane == 0) {
        c.tq[qs] = q;
        mbar_arrive(smem_u32(&c.tq_full[qs]));
      }
      if (cur < 0) break;
      tile = __shfl_sync(0xffffffffu, nxt, 0);
    }
  } else {
    // -------------------------------------------------- epilogue (2 groups of 4 warps)
    // TW = 1: group g takes the CTA's tiles g, g+2, g+4, ...; tile i sits in
    // accumulator i % 3.  TW = 2: both groups take every tile, group g its
    // slot g; each warp first drains its 32 rows x 128 columns into registers
    // as bf16 (the values it stores and dots), then frees the accumulator, so
    // the next tile's MMAs wait only for that drain.  Every epilogue warp reads
    // every queue entry (to see the end marker).  Warp w reads TMEM lanes
    // 32*(w%4)..+31.  Same staging, stores and fixed in-slot tree as the bf16
    // single-CTA kernel.
    const int q = warp & 3;
    const int grp = (warp - EPI_WARP0) >> 2;
    const int k4 = lane & 3;
    const uint64_t pol_keep = policy_evict_last();
    const uint32_t stg = stage0 + uint32_t(L::STAGES * L::STAGE_BYTES + (warp - EPI_WARP0) * STG_BYTES);   // TW = 1
    float alpha = 1.0f;
    if (KIND == kNvf4) alpha = __frcp_rn(__fmul_rn(__ldg(p.s_enc_x), __ldg(p.s_enc_w)));
    int acc = 0;
    uint32_t aph = 0;
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      if (!warp_wait(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), &c.abort, p.status, lane, p.wait_ns)) break;
      const QTile tl = c.tq[qs];
      const int cur = tl.cur;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.tq_empty[qs]));
      if (cur < 0) break;
      if (TW == 1 && (qi & 1) != grp) {
        if (++acc == L::ACC) { acc = 0; aph ^= 1u; }
        continue;
      }
      const int col0 = tl.n0 + (TW == 2 ? grp * BN : 0);
      int rr[4], src[4];
      bool ok[4];
      // the rows whose 16-byte piece k4 this lane stores and dots: TW = 1,
      // rows 8i + lane/4 (the staging buffer's read-back layout); TW = 2,
      // rows 4 (lane/4) + i (after a quad transpose of the lane's own row, as
      // in the CTA-pair kernel)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rr[i] = tl.row0 + q * 32 + (TW == 2 ? (lane & ~3) + i : i * 8 + (lane >> 2));
        ok[i] = rr[i] < tl.row_end;
        src[i] = 0;
      }
      const bool full32 = tl.row0 + q * 32 + 32 <= tl.row_end;
      if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (ok[i]) {
            src[i] = p.row_src[rr[i]];
            if (unsigned(src[i]) >= unsigned(p.R)) {   // corrupt row_src: report, never index with it
              record_error(p.status, DMOE_ERR_ROUTING);
              ok[i] = false;
            }
          }
        }
      }
      if (TW == 2) {
        // grad_out of the rows the lane dots: chunk 0 before the accumulator
        // is ready, then one chunk ahead of use
        const uint16_t* gp[4] = {nullptr, nullptr, nullptr, nullptr};   // forward only: no grad_out
        if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            gp[i] = p.grad_out + size_t(ok[i] ? src[i] / p.topk : 0) * p.N + (ok[i] ? col0 : 0) + k4 * 8;
        }
        uint4 gc[4], gn[4];
        if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
          for (int i = 0; i < 4; ++i) gc[i] = ok[i] ? ldg_nc_v4_hint(gp[i], pol_keep) : make_uint4(0, 0, 0, 0);
        }
        if (!warp_wait(smem_u32(&c.acc_full[acc]), aph, &c.abort, p.status, lane, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t tcol = tmem_base + uint32_t(acc * TW * BN + grp * BN) + (uint32_t(q * 32) << 16);
        // drain: row `lane` of the warp's quarter, four chunks of 32 columns, as
        // bf16, each chunk quad-transposed at once (yb[ch][i] = piece k4 of row
        // 4 (lane/4) + i)
        uint4 yb[4][4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tcol + uint32_t(ch * 32), v);
          tmem_wait_ld();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            yb[ch][kk].x = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 0]), __uint_as_float(v[8 * kk + 1]));
            yb[ch][kk].y = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 2]), __uint_as_float(v[8 * kk + 3]));
            yb[ch][kk].z = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 4]), __uint_as_float(v[8 * kk + 5]));
            yb[ch][kk].w = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 6]), __uint_as_float(v[8 * kk + 7]));
          }
          quad_transpose(yb[ch], lane);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c.acc_empty[acc]));
        if (++acc == L::ACC) { acc = 0; aph ^= 1u; }
        float a[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) a[i][j] = 0.0f;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          if (MODE != int(GemmMode::kFwd) && ch + 1 < 4) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              gn[i] = ok[i] ? ldg_nc_v4_hint(gp[i] + (ch + 1) * 32, pol_keep) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ok[i]) {
              stg_v4(p.out + size_t(rr[i]) * p.N + col0 + ch * 32 + k4 * 8, yb[ch][i]);
              if (MODE != int(GemmMode::kFwd)) slot_accumulate8(a[i], gc[i], yb[ch][i]);
            }
          }
          if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
            for (int i = 0; i < 4; ++i) gc[i] = gn[i];
          }
        }
        if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float part = slot_tree(a[i]);
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 2));
            if (k4 == 0 && ok[i]) p.slots[size_t(col0 / SLOT) * p.R + rr[i]] = part;
          }
        }
        continue;
      }
      uint4 g[16];
      if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint16_t* gp = p.grad_out + size_t(ok[i] ? src[i] / p.topk : 0) * p.N + (ok[i] ? col0 : 0) + k4 * 8;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) g[ch * 4 + i] = ok[i] ? ldg_nc_v4_hint(gp + ch * 32, pol_keep) : make_uint4(0, 0, 0, 0);
        }
      }
      if (!warp_wait(smem_u32(&c.acc_full[acc]), aph, &c.abort, p.status, lane, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t tcol = tmem_base + uint32_t(acc * BN) + (uint32_t(q * 32) << 16);   // TW = 1
      float a[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) a[i][j] = 0.0f;
#pragma unroll
      for (int ch = 0; ch < SLOT / 32; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tcol + uint32_t(ch * 32), v);
        tmem_wait_ld();
        if (KIND == kNvf4) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__fmul_rn(__uint_as_float(v[j]), alpha));
        }
        if (lane == 0) bulk_wait_group_read<0>();   // the previous chunk's store has read the staging
        __syncwarp();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint4 y;
          y.x = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 0]), __uint_as_float(v[8 * kk + 1]));
          y.y = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 2]), __uint_as_float(v[8 * kk + 3]));
          y.z = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 4]), __uint_as_float(v[8 * kk + 5]));
          y.w = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 6]), __uint_as_float(v[8 * kk + 7]));
          sts_v4(stg + uint32_t(lane * 64 + ((kk ^ ((lane >> 1) & 3)) << 4)), y);
        }
        __syncwarp();
        if (full32) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmap_o, stg, col0 + ch * 32, tl.row0 + q * 32);
            bulk_commit_group();
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = i * 8 + (lane >> 2);
          const uint4 y = lds_v4(stg + uint32_t(row * 64 + ((k4 ^ ((row >> 1) & 3)) << 4)));
          if (ok[i]) {
            if (!full32) stg_v4(p.out + size_t(rr[i]) * p.N + col0 + ch * 32 + k4 * 8, y);
            if (MODE != int(GemmMode::kFwd)) slot_accumulate8(a[i], g[ch * 4 + i], y);
          }
        }
        __syncwarp();
      }
      if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float part = slot_tree(a[i]);
          part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
          part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 2));
          if (k4 == 0 && ok[i]) p.slots[size_t(col0 / SLOT) * p.R + rr[i]] = part;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.acc_empty[acc]));
      if (++acc == L::ACC) { acc = 0; aph ^= 1u; }
    }
    if (lane == 0) bulk_wait_group_all();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (tid == 0) {
    // every counter fetch of this CTA (made by its scheduler warp) has
    // returned before the barrier above; the last CTA to finish zeroes both
    // counters for the next launch on this stream
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == int(gridDim.x) - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
}

template <int KIND, int MODE, int TW>
cudaError_t launch_kind_mode(const CUtensorMap* maps, const KParams& kp, int grid, cudaStream_t stream) {
  using L = Layout<KIND, TW>;
  const cudaError_t e =
      ensure_kernel_smem(reinterpret_cast<const void*>(grouped_gemm_bs_kernel<KIND, MODE, TW>), int(L::SMEM));
  if (e != cudaSuccess) return e;
  return launch_chained(grouped_gemm_bs_kernel<KIND, MODE, TW>, dim3(grid), dim3(NUM_THREADS), L::SMEM, stream,
                        maps[0], maps[1], maps[2], maps[3], maps[4], kp);
}

}  // namespace

cudaError_t launch_grouped_gemm_block_scaled(const BlockScaledArgs& a, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  const bool nvf4 = a.kind == 1;
  const uint64_t kbytes = nvf4 ? uint64_t(a.K) / 2 : uint64_t(a.K);        // operand bytes per row
  const uint64_t sbytes = nvf4 ? uint64_t(a.K) / 16 : uint64_t(a.K) / 32;  // scale bytes per row
  CUtensorMap maps[5];
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (!make_tmap_2d(&maps[0], a.Xq, u8, uint64_t(a.R), kbytes, kbytes, ROWB, BM, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  // MXFP8 with an even number of slots: two-slot tiles, unless narrow tiles are asked for
  const int tw = (!nvf4 && (a.N / BN) % 2 == 0 && !a.narrow) ? 2 : 1;
  if (!make_tmap_2d(&maps[1], a.Wq, u8, uint64_t(a.E) * a.N, kbytes, kbytes, ROWB, BN * tw,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&maps[2], a.Xs, u8, uint64_t(a.R), sbytes, sbytes, 16, BM, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&maps[3], a.Ws, u8, uint64_t(a.E) * a.N, sbytes, sbytes, 16, BN * tw, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return cudaErrorInvalidValue;
  if (!make_tmap_bf16_store32(&maps[4], a.out, uint64_t(a.R), uint64_t(a.N))) return cudaErrorInvalidValue;
  KParams kp;
  kp.offsets = a.offsets;
  kp.E = a.E;
  kp.R = a.R;
  kp.K = a.K;
  kp.N = a.N;
  kp.NT = a.N / (BN * tw);
  kp.KB = int(kbytes / ROWB);
  kp.out = static_cast<uint16_t*>(a.out);
  kp.grad_out = static_cast<const uint16_t*>(a.grad_out);
  kp.row_src = a.row_src;
  kp.topk = a.topk;
  kp.slots = a.slots;
  kp.s_enc_x = a.s_enc_x;
  kp.s_enc_w = a.s_enc_w;
  kp.status = a.status;
  kp.sched = a.sched;
  kp.wait_ns = kWaitLimitNs;
  if (!kp.sched) return cudaErrorInvalidValue;
  const int grid = a.num_ctas > 0 ? a.num_ctas : device_sm_count();
  const bool fwd = a.grad_out == nullptr;
  if (!nvf4) {
    if (tw == 2)
      return fwd ? launch_kind_mode<kMxf8, int(GemmMode::kFwd), 2>(maps, kp, grid, stream)
                 : launch_kind_mode<kMxf8, int(GemmMode::kSlots), 2>(maps, kp, grid, stream);
    return fwd ? launch_kind_mode<kMxf8, int(GemmMode::kFwd), 1>(maps, kp, grid, stream)
               : launch_kind_mode<kMxf8, int(GemmMode::kSlots), 1>(maps, kp, grid, stream);
  }
  return fwd ? launch_kind_mode<kNvf4, int(GemmMode::kFwd), 1>(maps, kp, grid, stream)
             : launch_kind_mode<kNvf4, int(GemmMode::kSlots), 1>(maps, kp, grid, stream);
}

}  // namespace dmoe
