// Persistent grouped GEMM for GB300 (sm_103a) with the fused private-slot
// dprob epilogue.
//
// The operation follows "Trillion-Parameter Pretraining Goes Bitwise-
// Deterministic: NVIDIA Cuts the Determinism Tax to About 2%", section
// "Interpretation": in the grouped-GEMM epilogue every N-tile used to add its
// share of dprob[token] at one address, so the result depended on arrival
// order; here each N-tile writes its share into a private slot and a later
// pass combines the slots in a fixed order.  The slot width is fixed at 128
// output columns, independent of the MMA tile width, so the bits do not
// depend on the tile shape either.
//
// Design (one CTA per SM, persistent, warp-specialised, 352 threads):
//   warp 0  TMA producer: A tile [128 rows x 64 k] and B tile [256 n x 64 k]
//           per stage, 128-byte swizzle, 4-stage ring in shared memory.
//   warp 1  tcgen05.mma issuer (one thread): 128x256x16 bf16 MMAs, fp32
//           accumulators in tensor memory, double-buffered (2 x 256 columns).
//   warps 2-9  epilogue: tcgen05.ld of the accumulator, bf16 rounding into a
//           swizzled staging buffer, expert_out stores (a TMA tensor store per
//           32x32 chunk when all 32 rows belong to the expert, masked row
//           stores otherwise), and the per-slot dot products with grad_out in
//           the fixed tree (one warp per 32 rows x 128 columns = one private
//           slot).  The rows' grad_out slices are fetched before the
//           accumulator is ready.
//   warp 10 tile scheduler: claims tiles, decodes each into (expert, rows,
//           columns) a few tiles ahead of use and queues the decoded tile
//           for the other roles, so no role decodes on its critical path.
// Tiles (one m-tile x one n-tile of one expert) are ordered so that heavy and
// light experts' work interleaves (see decode_tile_warp) and handed out dynamically
// through a global counter: each output element is produced by exactly one
// tile with a fixed k order, so the result does not depend on which CTA runs
// it, on the order, or on the grid size.
// An M-tile may run past its expert's last row into the next expert's rows;
// those rows are computed but never stored.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int BM = 128;                  // rows per tile (UMMA M)
constexpr int BN = 256;                  // columns per tile (UMMA N)
constexpr int BK = 64;                   // k per stage: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;               // k per tcgen05.mma (kind::f16)
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int B_STAGE_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;  // 512 = all of tensor memory
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 8;                  // two per TMEM lane quarter
constexpr int SCHED_WARP = EPI_WARP0 + EPI_WARPS;
constexpr int NUM_THREADS = 32 * (SCHED_WARP + 1);
constexpr int SLOT = DMOE_SLOT_COLS;
constexpr int TQ = 4;                         // tile-queue depth (the scheduler runs <= 3 tiles ahead)
constexpr int HEAVY_MT = 3;                   // experts with >= 3 m-tiles reuse each weight slice 3+ times

// A decoded tile as the scheduler queues it: cur = tile index (-1 = no more
// tiles), e = expert, rows [row0, row_end) of that expert's range starting at
// row0 (the tile covers row0 .. row0 + BM - 1), columns n0 .. n0 + BN - 1.
struct QTile {
  int cur, e, row0, row_end, n0, pad0, pad1, pad2;
};

struct alignas(8) Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[ACC_BUFS];
  uint64_t acc_empty[ACC_BUFS];
  uint64_t mma_done;
  uint64_t tq_full[TQ];                  // tile queue: scheduler -> producer, MMA and epilogue
  uint64_t tq_empty[TQ];                 // slot consumed by the producer, the MMA thread and all epilogue warps
  QTile tq[TQ];
  uint32_t tmem_base;
  int abort;
  int bad;
  int off[DMOE_MAX_EXPERTS + 1];         // expert row offsets
  int hp[DMOE_MAX_EXPERTS + 1];          // exclusive prefix of m-tiles of heavy experts (0 for light ones)
  int cp[DMOE_MAX_EXPERTS + 1];          // exclusive prefix of m-tiles of light experts (0 for heavy ones)
};

constexpr int STG_BYTES = 32 * 64;             // per epilogue warp: 32 rows x 32 bf16
constexpr size_t kSmemBytes = 1024 + size_t(STAGES) * STAGE_BYTES + size_t(EPI_WARPS) * STG_BYTES + sizeof(Ctrl);
static_assert(kSmemBytes <= 232448, "dynamic shared memory above the 227 KB a CTA may use");

struct KParams {
  const int32_t* offsets;
  int E, R, K, N, NT, KB;
  uint16_t* out;
  const uint16_t* grad_out;
  const int32_t* row_src;
  int topk;
  float* slots;
  float* dprob;
  int* wflags;  // serialized writers: slots already added per (m-tile, row quarter); zero at launch
  int* status;
  int* sched;   // [0] next-tile counter, [1] finished-CTA counter; zero between launches
  unsigned long long wait_ns;   // limit of every pipeline wait
  int stall_test;               // test only: CTA 0 arms its first stage but never loads it
};

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);      // start address >> 4
  d |= uint64_t(1) << 16;                       // leading byte offset (unused for swizzled K-major)
  d |= uint64_t(1024 >> 4) << 32;               // stride byte offset: 8 rows x 128 B
  d |= uint64_t(1) << 46;                       // descriptor version for tcgen05
  d |= uint64_t(2) << 61;                       // swizzle mode: 128-byte
  return d;
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major, M=128, N=256.
constexpr uint32_t kIdesc = (1u << 4)                       // D format: f32
                            | (1u << 7)                     // A format: bf16
                            | (1u << 10)                    // B format: bf16
                            | (uint32_t(BN >> 3) << 17)     // N >> 3
                            | (uint32_t(BM >> 4) << 24);    // M >> 4

// Tile order.  A unit is one m-tile of one expert; its NT n-tiles are
// consecutive tiles (they share the X rows in L2).  Units of heavy experts
// (compute-bound: each weight slice serves >= HEAVY_MT m-tiles) and of light
// experts (bound by streaming their weights from HBM) are merged in
// proportion -- unit position p is heavy iff floor((p+1)H/U) > floor(pH/U) --
// so both the tensor cores and HBM stay busy; within each class units follow
// expert order, so an expert's weight slices are reused while resident.
// The order only decides when a tile runs, never what it computes.
//
// Decoded by the whole scheduler warp (called with all 32 lanes): the expert
// is the largest e < E with pre[e] <= u in the class's exclusive m-tile
// prefix, found with two ballots (every 32nd entry, then the 32 entries of
// that segment; E <= 1024) instead of a serial binary search.
__device__ __forceinline__ QTile decode_tile_warp(int t, const Ctrl& c, int E, int NT, int H, int U, int lane) {
  const int p = t / NT;
  const int n_tile = t - p * NT;
  const int i = int((long long)p * H / U);                   // heavy units before position p
  const bool heavy = (long long)(p + 1) * H / U > i;
  const int* pre = heavy ? c.hp : c.cp;
  const int u = heavy ? i : p - i;
  const int e1 = lane * 32;
  const unsigned m1 = __ballot_sync(0xffffffffu, e1 < E && pre[e1] <= u);   // lane 0 always (pre[0] = 0)
  const int seg = 31 - __clz(m1);
  const int e2 = seg * 32 + lane;
  const int v2 = e2 < E ? pre[e2] : 0x7fffffff;
  const unsigned m2 = __ballot_sync(0xffffffffu, v2 <= u);
  const int l2 = 31 - __clz(m2);
  const int e = seg * 32 + l2;
  const int pe = __shfl_sync(0xffffffffu, v2, l2);
  QTile q;
  q.cur = t;
  q.e = e;
  q.row0 = c.off[e] + (u - pe) * BM;
  q.row_end = c.off[e + 1];
  q.n0 = n_tile * BN;
  q.pad0 = q.pad1 = q.pad2 = 0;
  return q;
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_o, const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl& c = *reinterpret_cast<Ctrl*>(base + size_t(STAGES) * STAGE_BYTES + size_t(EPI_WARPS) * STG_BYTES);
  const uint32_t stage0 = smem_u32(base);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&c.full[s]), 1);
      mbar_init(smem_u32(&c.empty[s]), 1);
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(smem_u32(&c.acc_full[b]), 1);
      mbar_init(smem_u32(&c.acc_empty[b]), EPI_WARPS);
    }
    mbar_init(smem_u32(&c.mma_done), 1);
    for (int i = 0; i < TQ; ++i) {
      mbar_init(smem_u32(&c.tq_full[i]), 1);
      mbar_init(smem_u32(&c.tq_empty[i]), 2 + EPI_WARPS);   // producer, MMA thread, epilogue warps
    }
    c.abort = 0;
    c.bad = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  // Expert offsets -> shared memory, validated, and the m-tile prefix.
  pdl_begin();   // no global memory is touched above this line
  for (int e = tid; e <= E; e += NUM_THREADS) c.off[e] = p.offsets[e];
  __syncthreads();
  int bad = 0;
  for (int e = tid; e < E; e += NUM_THREADS) {
    int a = c.off[e], b = c.off[e + 1];
    if (b < a) bad = 1;
    const int mt = (b > a) ? (b - a + BM - 1) / BM : 0;
    c.hp[e + 1] = mt >= HEAVY_MT ? mt : 0;
    c.cp[e + 1] = mt >= HEAVY_MT ? 0 : mt;
  }
  if (tid == 0) {
    if (c.off[0] != 0 || c.off[E] != p.R) bad = 1;
    c.hp[0] = 0;
    c.cp[0] = 0;
  }
  bad = __syncthreads_or(bad);
  if (warp < 2) {
    // inclusive scans of hp[1..E] (warp 0) and cp[1..E] (warp 1) in chunks of 32
    int* pre = warp == 0 ? c.hp : c.cp;
    int carry = 0;
    for (int b0 = 1; b0 <= E; b0 += 32) {
      int i = b0 + lane;
      int v = (i <= E) ? pre[i] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += u;
      }
      if (i <= E) pre[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (bad && tid == 0) record_error(p.status, DMOE_ERR_ROUTING);
  const int units_heavy = c.hp[E];
  const int units = c.hp[E] + c.cp[E];
  const int total_tiles = bad ? 0 : units * p.NT;
  const uint32_t tmem_base = c.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      // stages are used round-robin, so stage s has been loaded
      // (issued_total - s + STAGES - 1) / STAGES times (minus the one skipped
      // by the stall test); no per-stage array in local memory
      int issued_total = 0;
      bool skipped_first = false;
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
          const uint32_t full = smem_u32(&c.full[stage]);
          const uint32_t sa = stage0 + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(full, STAGE_BYTES);
          if (p.stall_test && blockIdx.x == 0 && qi == 0 && kb == 0) {
            // expected bytes that never arrive: the MMA's wait on this stage
            // must run out and report DMOE_ERR_TIMEOUT (nothing is in flight)
            skipped_first = true;
          } else {
            tma_load_2d(sa, &tmap_a, full, kb * BK, tl.row0);
            tma_load_2d(sa + A_STAGE_BYTES, &tmap_b, full, kb * BK, brow);
          }
          ++issued_total;
          if (++stage == STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
      }
      // let every copy this thread started land before the CTA can exit
      for (int s = 0; s < STAGES; ++s) {
        const int n = (issued_total - s + STAGES - 1) / STAGES - ((s == 0 && skipped_first) ? 1 : 0);
        if (n > 0 && !(s == 0 && skipped_first))
          mbar_wait_drain(smem_u32(&c.full[s]), uint32_t(n - 1) & 1u, p.wait_ns / 4);
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
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(smem_u32(&c.full[stage]), ph, &c.abort, p.status, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = stage0 + stage * STAGE_BYTES;
          const uint64_t adesc = smem_desc_k128(sa);
          const uint64_t bdesc = smem_desc_k128(sa + A_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // advance 32 bytes (16 bf16) along k inside the swizzled row
            tc_mma_f16(d_tmem, adesc + uint64_t(kk * 2), bdesc + uint64_t(kk * 2), kIdesc,
                       (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&c.empty[stage]));
          if (++stage == STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(smem_u32(&c.acc_full[acc]));
        if (++acc == ACC_BUFS) { acc = 0; aph ^= 1u; }
      }
      // every MMA must be finished before tensor memory is released
      tc_commit(smem_u32(&c.mma_done));
      mbar_wait_drain(smem_u32(&c.mma_done), 0, p.wait_ns / 4);
    }
  } else if (warp == SCHED_WARP) {
    // -------------------------------------------------- tile scheduler (one warp)
    // Tiles are handed out dynamically (first tile = blockIdx.x, then a
    // global counter), so neighbouring tiles -- which share weight slices
    // and X rows in L2 -- run at nearly the same time on different SMs.
    // Which CTA computes a tile never changes its bits.  Each claimed tile
    // is decoded while its queue slot is still in use and queued as soon as
    // the slot frees, so the producer moves from one tile's last stage to
    // the next tile's first without a pause; the next claim is in flight
    // meanwhile.
    // The serialized control claims every tile from the counter, so a tile
    // is owned only by a CTA that is already running: its writers wait on
    // earlier-claimed tiles only, which always make progress.
    constexpr bool kClaimAll = MODE == int(GemmMode::kSerial);
    int tile = 0;
    if (lane == 0) tile = kClaimAll ? atomicAdd(p.sched, 1) : int(blockIdx.x);
    tile = __shfl_sync(0xffffffffu, tile, 0);
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      // the serialized control claims n-tile-major (every m-tile's n-tile 0,
      // then every n-tile 1, ...), so a writer's predecessor was claimed a
      // whole round earlier; queued tiles carry the usual unit-major index
      const int cur = tile >= total_tiles ? -1
                      : kClaimAll ? (tile % units) * p.NT + tile / units : tile;
      int nxt = 0;
      if (cur >= 0 && lane == 0) nxt = (kClaimAll ? 0 : int(gridDim.x)) + atomicAdd(p.sched, 1);
      QTile q{};
      q.cur = -1;
      if (cur >= 0) q = decode_tile_warp(cur, c, E, p.NT, units_heavy, units, lane);
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
    // -------------------------------------------------- epilogue (8 warps)
    // Warp w may only read TMEM lanes 32*(w%4)..+31; warps 2-5 take the first
    // 128 columns (one slot) of their lane quarter, warps 6-9 the second.
    // tcgen05.ld gives one row per thread; each 32x32 bf16 chunk goes through
    // a 2 KB swizzled shared-memory buffer so that four lanes cover 64
    // contiguous bytes of a row: the expert_out stores and the grad_out
    // gather then touch 8 rows per warp instruction instead of 32.
    const int q = warp & 3;
    const int h = (warp - EPI_WARP0) / 4;
    const int k4 = lane & 3;                     // 16-byte piece of a 64-byte chunk row
    // grad_out rows are gathered 8x per token and slot: ask L2 to keep them
    // while 2+ GB of weights stream past.
    const uint64_t pol_keep = policy_evict_last();
    const uint32_t stg = stage0 + uint32_t(STAGES * STAGE_BYTES + (warp - EPI_WARP0) * STG_BYTES);
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
      const int col0 = tl.n0 + h * SLOT;
      const bool active = col0 < p.N;           // warp-uniform: a half-width last N-tile
      // rows of this lane in the coalesced layout: q*32 + i*8 + lane/4, i = 0..3
      int rr[4], src[4];
      bool ok[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rr[i] = tl.row0 + q * 32 + i * 8 + (lane >> 2);
        ok[i] = active && rr[i] < tl.row_end;
        src[i] = 0;
      }
      // a warp whose 32 rows all belong to the expert writes each 32x32 chunk
      // with one TMA tensor store from the staging buffer; a ragged last
      // quarter (rows of the next expert follow) stores row by row instead
      const bool full32 = active && (tl.row0 + q * 32 + 32 <= tl.row_end);
      // Prefetch grad_out for all four rows before the accumulator is ready.
      uint4 g[16];
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
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint16_t* gp = p.grad_out + size_t(ok[i] ? src[i] / p.topk : 0) * p.N + (ok[i] ? col0 : 0) + k4 * 8;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) g[ch * 4 + i] = ok[i] ? ldg_nc_v4_hint(gp + ch * 32, pol_keep) : make_uint4(0, 0, 0, 0);
        }
      }
      if (!warp_wait(smem_u32(&c.acc_full[acc]), aph, &c.abort, p.status, lane, p.wait_ns)) break;
      tc_fence_after();
      if (active) {
        const uint32_t tcol = tmem_base + uint32_t(acc * BN + h * SLOT) + (uint32_t(q * 32) << 16);
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
          // the previous chunk's tensor store must have read the staging buffer
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
          // row `lane` of the chunk -> staging, piece kk at slot kk ^ ((row >> 1) & 3)
          // (the 64-byte swizzle of the output tensor map)
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
            fence_proxy_async_smem();   // the generic-proxy staging writes, before the TMA unit reads them
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
          float parts[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // part k4 of row rr[i]; combine the four parts as (L0 + L1) + (L2 + L3)
            float part = slot_tree(a[i]);
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 2));
            parts[i] = part;
            if (k4 == 0 && ok[i]) {
              if (MODE == int(GemmMode::kSlots))
                p.slots[size_t(col0 / SLOT) * p.R + rr[i]] = part;
              else if (MODE == int(GemmMode::kAtomic))
                atomicAdd(p.dprob + src[i], part);
            }
          }
          if (MODE == int(GemmMode::kSerial)) {
            // Serialized writers: slot s of these 32 rows is added into dprob
            // only after slots 0..s-1 have been, so dprob = ((P0 + P1) + P2) + ...
            // -- the fixed-order combine's bits -- but the tiles of one
            // m-tile wait on one another instead of writing in parallel.
            const int s = col0 / SLOT;
            int* ctr = p.wflags + size_t(cur / p.NT) * 4 + q;
            int go = 1;
            if (lane == 0) go = counter_wait(ctr, s, &c.abort, p.status, p.wait_ns) ? 1 : 0;
            go = __shfl_sync(0xffffffffu, go, 0);
            __syncwarp();
            if (!go) break;
            __threadfence();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (k4 == 0 && ok[i]) {
                float* d = p.dprob + src[i];
                __stcg(d, s == 0 ? parts[i] : __fadd_rn(__ldcg(d), parts[i]));
              }
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(ctr, s + 1);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.acc_empty[acc]));
      if (++acc == ACC_BUFS) { acc = 0; aph ^= 1u; }
    }
    // every tensor store of this warp has landed before the CTA can exit
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

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // resolved once; the initialisation of a function-local static is thread-safe
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

}  // namespace

// 2-D bf16 tensor [rows, cols] (cols contiguous), box [box_rows, 64], 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {uint32_t(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor of `dtype` [rows, cols] with row pitch `row_bytes` (a multiple of
// 16), box [box_rows, box_cols], with the given swizzle and L2 promotion.
bool make_tmap_2d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, uint64_t rows, uint64_t cols,
                  uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle,
                  CUtensorMapL2promotion promotion) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  promotion, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D bf16 output [rows, cols] (cols contiguous, cols % 8 == 0) for TMA stores of
// box [32, 32] (64-byte rows) from a 64-byte-swizzled staging buffer.
bool make_tmap_bf16_store32(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {32u, 32u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D fp32 tensor [rows, cols] (cols contiguous, cols % 4 == 0) for TMA stores of
// box [box_rows, 16] through a 64-byte-swizzled staging buffer.
bool make_tmap_f32_store(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {16u, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const KParams& kp,
                        int grid, cudaStream_t stream) {
  const cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(grouped_gemm_kernel<MODE>), int(kSmemBytes));
  if (e != cudaSuccess) return e;
  return launch_chained(grouped_gemm_kernel<MODE>, dim3(grid), dim3(NUM_THREADS), kSmemBytes, stream, ta, tb, to, kp);
}

}  // namespace

size_t serial_flag_bytes(long long R, int E) {
  // m-tiles <= R/BM + E (at most one partial tile per expert), four row quarters each
  return size_t(R / BM + E + 1) * 4 * sizeof(int);
}

cudaError_t launch_grouped_gemm_1sm(GemmMode mode, const GemmArgs& a, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  CUtensorMap ta, tb, to;
  if (!make_tmap_bf16(&ta, a.X, uint64_t(a.R), uint64_t(a.K), BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, uint64_t(a.E) * a.N, uint64_t(a.K), BN)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16_store32(&to, a.out, uint64_t(a.R), uint64_t(a.N))) return cudaErrorInvalidValue;
  KParams kp;
  kp.offsets = a.offsets;
  kp.E = a.E;
  kp.R = a.R;
  kp.K = a.K;
  kp.N = a.N;
  kp.NT = (a.N + BN - 1) / BN;
  kp.KB = (a.K + BK - 1) / BK;
  kp.out = static_cast<uint16_t*>(a.out);
  kp.grad_out = static_cast<const uint16_t*>(a.grad_out);
  kp.row_src = a.row_src;
  kp.topk = a.topk;
  kp.slots = a.slots;
  kp.dprob = a.dprob;
  kp.wflags = a.wflags;
  kp.status = a.status;
  kp.sched = a.sched;
  if (!kp.sched) return cudaErrorInvalidValue;
  kp.stall_test = (a.flags & DMOE_LAUNCH_TEST_STALL) ? 1 : 0;
  kp.wait_ns = kp.stall_test ? 200ull * 1000ull * 1000ull : kWaitLimitNs;   // a short limit for the test
  int grid = a.num_ctas > 0 ? a.num_ctas : device_sm_count();
  if (mode == GemmMode::kSerial && !kp.wflags) return cudaErrorInvalidValue;
  switch (mode) {
    case GemmMode::kFwd: return launch_mode<int(GemmMode::kFwd)>(ta, tb, to, kp, grid, stream);
    case GemmMode::kSlots: return launch_mode<int(GemmMode::kSlots)>(ta, tb, to, kp, grid, stream);
    case GemmMode::kAtomic: return launch_mode<int(GemmMode::kAtomic)>(ta, tb, to, kp, grid, stream);
    case GemmMode::kSerial: return launch_mode<int(GemmMode::kSerial)>(ta, tb, to, kp, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dmoe
