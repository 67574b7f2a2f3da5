// Grouped GEMM + private-slot dprob epilogue on CTA pairs (2-SM tensor-core
// MMA, tcgen05 .cta_group::2) for GB300 (sm_103a).
//
// Same operation, tile order, epilogue arithmetic and results as the
// single-CTA kernel in grouped_gemm.cu ("Trillion-Parameter Pretraining Goes
// Bitwise-Deterministic: NVIDIA Cuts the Determinism Tax to About 2%",
// section "Interpretation": per-N-tile private dprob slots, combined later in
// a fixed order).  What changes is how a tile is fed to the tensor cores:
//
// A cluster of two CTAs (two SMs) owns a 256-row x 256-column tile.  The even
// CTA ("leader") issues tcgen05.mma.cta_group::2 with M = 256: each CTA holds
// 128 of the A rows and 128 of the 256 B rows of every 64-wide k stage in its
// own shared memory, and receives its 128 rows of the fp32 accumulator in its
// own tensor memory.  Per SM and per MMA cycle this halves the B operand that
// shared memory must supply and that TMA must bring in, which is what limits
// a single-CTA 128x256 tile on this part, and a stage shrinks to 32 KB so
// seven fit: the kernel keeps nothing else in shared memory (the expert
// tables live in the scheduler warp's registers, and the epilogue transposes
// through warp shuffles instead of a staging buffer).  Both CTAs load their halves with TMA and signal the leader's
// stage barrier; the leader's MMA commits free the stage in both CTAs
// (multicast) and publish finished accumulators to both epilogues.
//
// Roles per CTA (352 threads): warp 0 TMA producer; warp 1 tensor-memory
// owner and, in the leader, the single MMA-issuing thread (in the other CTA,
// a forwarder that turns its epilogue's local releases into one
// cluster-scope arrival each); warps 2-9 the epilogue (identical to the
// single-CTA kernel, on this CTA's 128 rows); warp 10, in the leader only,
// the tile scheduler: it takes tiles from the global counter, decodes each
// into (expert, rows, columns) a few tiles ahead of use and queues the
// decoded tile in both CTAs (the other CTA's copy through distributed shared
// memory), so no role decodes on its critical path.
// Every wait is bounded; a timeout in either CTA aborts both.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tile_sched.cuh"

namespace dmoe {

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);

namespace {

constexpr int BM = 128;                  // rows per CTA
constexpr int PM = 256;                  // rows per CTA pair (UMMA M)
constexpr int BN = 256;                  // columns per tile (UMMA N)
constexpr int BNH = BN / 2;              // B rows held by each CTA
constexpr int BK = 64;                   // k per stage: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int STAGES = 7;
constexpr int A_STAGE_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_STAGE_BYTES = BNH * BK * 2;    // 16 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 8;
constexpr int SCHED_WARP = EPI_WARP0 + EPI_WARPS;
constexpr int NUM_THREADS = 32 * (SCHED_WARP + 1);
constexpr int SLOT = DMOE_SLOT_COLS;
constexpr int TQ = 4;
constexpr int HEAVY_MT = 2;              // pair m-tiles (256 rows) per expert that make it compute-bound

struct alignas(16) Ctrl {
  uint64_t full[STAGES];                 // leader: both CTAs' halves of a stage landed
  uint64_t empty[STAGES];                // each CTA: the pair's MMAs are done with the stage
  uint64_t acc_full[ACC_BUFS];           // each CTA: accumulator ready
  uint64_t acc_empty[ACC_BUFS];          // leader: both CTAs' epilogues drained the accumulator
  uint64_t mma_done;
  uint64_t tq_full[TQ];                  // each CTA: decoded tile published by the leader's scheduler
  uint64_t tq_empty[TQ];                 // leader: every consumer of both CTAs read the slot
  uint64_t tq_read[TQ];                  // other CTA: its epilogue warps read the slot
  uint64_t acc_read[ACC_BUFS];           // other CTA: its epilogue warps drained the accumulator
  QTile tq[TQ];
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + size_t(STAGES) * STAGE_BYTES + sizeof(Ctrl);
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
  int* status;
  int* sched;
  unsigned long long wait_ns;
  int stall_test;
};

__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(1) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// kind::f16: fp32 D, bf16 A and B, both K-major, M = 256 (the pair), N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                            (uint32_t(PM >> 4) << 24);

// Bounded wait that also raises the other CTA's abort flag when it gives up.
// CLUSTER = true for barriers the other CTA arrives on after writing this
// CTA's shared memory or reading its own tensor memory (acquire at cluster
// scope); the per-stage barriers, completed by TMA bytes and tensor-core
// commits, use the CTA-scope wait.
template <bool CLUSTER>
__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, Ctrl& c, const KParams& p,
                                      uint32_t peer_abort) {
  const bool ok = CLUSTER ? mbar_wait_cluster(bar, parity, &c.abort, p.status, p.wait_ns)
                          : mbar_wait(bar, parity, &c.abort, p.status, p.wait_ns);
  if (ok) return true;
  st_cluster_s32(peer_abort, 1);
  return false;
}

template <bool CLUSTER>
__device__ __forceinline__ bool pwarp_wait(uint32_t bar, uint32_t parity, Ctrl& c, const KParams& p,
                                           uint32_t peer_abort, int lane) {
  int ok = 1;
  if (lane == 0) ok = pwait<CLUSTER>(bar, parity, c, p, peer_abort) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl& c = *reinterpret_cast<Ctrl*>(base + size_t(STAGES) * STAGE_BYTES);
  const uint32_t stage0 = smem_u32(base);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int E = p.E;
  const uint32_t rank = cluster_ctarank();       // 0 = leader (issues the MMAs)
  const bool leader = rank == 0;
  const uint32_t peer = rank ^ 1u;
  const uint32_t peer_abort = mapa_shared(smem_u32(&c.abort), peer);

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&c.full[s]), 1);                 // leader's producer arms it for both CTAs' bytes
      mbar_init(smem_u32(&c.empty[s]), 1);                // one multicast commit per use
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      mbar_init(smem_u32(&c.acc_full[b]), 1);
      mbar_init(smem_u32(&c.acc_empty[b]), EPI_WARPS + 1);  // leader: its epilogue warps + the other CTA's forwarder
      mbar_init(smem_u32(&c.acc_read[b]), EPI_WARPS);
    }
    mbar_init(smem_u32(&c.mma_done), 1);
    for (int i = 0; i < TQ; ++i) {
      mbar_init(smem_u32(&c.tq_full[i]), 1);
      // leader: its producer, MMA thread and epilogue warps + the other CTA's producer and forwarder
      mbar_init(smem_u32(&c.tq_empty[i]), 2 + EPI_WARPS + 2);
      mbar_init(smem_u32(&c.tq_read[i]), EPI_WARPS);
    }
    c.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&c.tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  pdl_begin();   // no global memory is touched above this line
  tc_fence_before();
  // both CTAs' barriers are initialised before either touches the other's
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int n_pairs = int(gridDim.x) / 2;
  const int pair_id = int(blockIdx.x) / 2;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t ph = 0;
      bool in_flight = false;
      int armed_total = 0;         // leader: stages armed so far (round-robin over STAGES)
      for (int qi = 0;; ++qi) {
        const int qs = qi % TQ;
        if (!pwait<true>(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), c, p, peer_abort)) break;
        const QTile tl = c.tq[qs];
        if (leader) mbar_arrive(smem_u32(&c.tq_empty[qs]));
        else mbar_arrive_cluster(mapa_shared(smem_u32(&c.tq_empty[qs]), peer));
        if (tl.cur < 0) break;
        const int arow = tl.row0 + int(rank) * BM;
        const int brow = tl.e * p.N + tl.n0 + int(rank) * BNH;
        bool ok = true;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!pwait<false>(smem_u32(&c.empty[stage]), ph ^ 1u, c, p, peer_abort)) { ok = false; break; }
          const uint32_t full_leader = mapa_shared(smem_u32(&c.full[stage]), 0);
          const uint32_t sa = stage0 + stage * STAGE_BYTES;
          // The leader arms the stage for both CTAs' bytes; the other CTA's
          // copies may land first (the tx count dips below zero), but the
          // phase cannot complete before the leader's arrival.
          if (leader) {
            mbar_arrive_expect_tx(smem_u32(&c.full[stage]), 2 * STAGE_BYTES);
            ++armed_total;
          }
          if (p.stall_test && blockIdx.x == 0 && qi == 0 && kb == 0) {
            // bytes that never arrive: the leader's MMA wait must run out
          } else {
            tma_load_2d_pair(sa, &tmap_a, full_leader, kb * BK, arow);
            tma_load_2d_pair(sa + A_STAGE_BYTES, &tmap_b, full_leader, kb * BK, brow);
            in_flight = true;
          }
          if (++stage == STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
      }
      if (leader) {
        // every armed stage completes only when both CTAs' copies landed
        for (int s = 0; s < STAGES; ++s) {
          const int n = (armed_total - s + STAGES - 1) / STAGES;
          if (n > 0) mbar_wait_drain(smem_u32(&c.full[s]), uint32_t(n - 1) & 1u, p.wait_ns / 4);
        }
      } else if (c.abort && in_flight) {
        // on the unwind path the other CTA may stop consuming: give copies this
        // CTA started time to land before it can exit
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && !leader) {
      // ------------------------------------------------ forwarder (other CTA)
      // Its epilogue warps release tile slots and accumulators on local
      // barriers; this thread passes each completion on to the leader with a
      // single cluster-scope arrival, off the epilogue's critical path.
      int acc = 0;
      uint32_t aph = 0;
      for (int qi = 0;; ++qi) {
        const int qs = qi % TQ;
        const uint32_t qph = uint32_t((qi / TQ) & 1);
        if (!pwait<true>(smem_u32(&c.tq_full[qs]), qph, c, p, peer_abort)) break;
        const int cur = c.tq[qs].cur;
        if (!pwait<false>(smem_u32(&c.tq_read[qs]), qph, c, p, peer_abort)) break;
        mbar_arrive_cluster(mapa_shared(smem_u32(&c.tq_empty[qs]), peer));
        if (cur < 0) break;
        if (!pwait<false>(smem_u32(&c.acc_read[acc]), aph, c, p, peer_abort)) break;
        mbar_arrive_cluster(mapa_shared(smem_u32(&c.acc_empty[acc]), peer));
        if (++acc == ACC_BUFS) { acc = 0; aph ^= 1u; }
      }
    }
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer (leader only)
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      for (int qi = 0;; ++qi) {
        const int qs = qi % TQ;
        if (!pwait<false>(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), c, p, peer_abort)) break;
        const int cur = c.tq[qs].cur;
        mbar_arrive(smem_u32(&c.tq_empty[qs]));
        if (cur < 0) break;
        if (!pwait<true>(smem_u32(&c.acc_empty[acc]), aph ^ 1u, c, p, peer_abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!pwait<false>(smem_u32(&c.full[stage]), ph, c, p, peer_abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = stage0 + stage * STAGE_BYTES;
          const uint64_t adesc = smem_desc_k128(sa);
          const uint64_t bdesc = smem_desc_k128(sa + A_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            tc_mma_pair_f16(d_tmem, adesc + uint64_t(kk * 2), bdesc + uint64_t(kk * 2), kIdesc,
                            (kb | kk) != 0 ? 1u : 0u);
          tc_commit_pair_mc(smem_u32(&c.empty[stage]), uint16_t(0x3));
          if (++stage == STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair_mc(smem_u32(&c.acc_full[acc]), uint16_t(0x3));
        if (++acc == ACC_BUFS) { acc = 0; aph ^= 1u; }
      }
      tc_commit_pair(smem_u32(&c.mma_done));
      mbar_wait_drain(smem_u32(&c.mma_done), 0, p.wait_ns / 4);
    }
  } else if (warp == SCHED_WARP) {
    if (leader) {
      // ------------------------------------------------ tile scheduler (leader, one warp)
      // First tile = the pair index, then the global counter.  Each claimed
      // tile is decoded while its queue slot is still in use and published
      // to both CTAs as soon as every consumer of both has released the
      // slot; the next claim is in flight meanwhile.
      ExpertTables tb;
      int units_heavy = 0, units_light = 0;
      const bool bad = build_tables<PM, HEAVY_MT>(tb, p.offsets, E, p.R, lane, units_heavy, units_light);
      if (bad && lane == 0) record_error(p.status, DMOE_ERR_ROUTING);
      const int units = units_heavy + units_light;
      const int total_tiles = bad ? 0 : units * p.NT;
      int tile = 0;
      if (lane == 0) tile = pair_id;
      tile = __shfl_sync(0xffffffffu, tile, 0);
      for (int qi = 0;; ++qi) {
        const int qs = qi % TQ;
        const int cur = tile < total_tiles ? tile : -1;
        int nxt = 0;
        if (cur >= 0 && lane == 0) nxt = n_pairs + atomicAdd(p.sched, 1);
        QTile q{};
        q.cur = -1;
        if (cur >= 0) q = decode_tile_warp<PM, BN>(cur, tb, E, p.NT, units_heavy, units, lane);
        if (!pwarp_wait<true>(smem_u32(&c.tq_empty[qs]), uint32_t((qi / TQ) & 1) ^ 1u, c, p, peer_abort, lane))
          break;
        if (lane == 0) {
          c.tq[qs] = q;
          // the other CTA's copy: eight words through distributed shared
          // memory, made visible by the release of the arrival that follows
          const uint32_t dst = mapa_shared(smem_u32(&c.tq[qs]), peer);
          st_cluster_s32(dst + 0, q.cur);
          st_cluster_s32(dst + 4, q.e);
          st_cluster_s32(dst + 8, q.row0);
          st_cluster_s32(dst + 12, q.row_end);
          st_cluster_s32(dst + 16, q.n0);
          mbar_arrive(smem_u32(&c.tq_full[qs]));
          mbar_arrive_cluster(mapa_shared(smem_u32(&c.tq_full[qs]), peer));
        }
        if (cur < 0) break;
        tile = __shfl_sync(0xffffffffu, nxt, 0);
      }
    }
  } else {
    // -------------------------------------------------- epilogue (8 warps, both CTAs)
    const int q = warp & 3;
    const int h = (warp - EPI_WARP0) / 4;
    const int k4 = lane & 3;
    const uint64_t pol_keep = policy_evict_last();
    int acc = 0;
    uint32_t aph = 0;
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      if (!pwarp_wait<true>(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), c, p, peer_abort, lane)) break;
      const QTile tl = c.tq[qs];
      const int cur = tl.cur;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(leader ? &c.tq_empty[qs] : &c.tq_read[qs]));
      }
      if (cur < 0) break;
      const int col0 = tl.n0 + h * SLOT;
      const bool active = col0 < p.N;
      const int row_cta = tl.row0 + int(rank) * BM;
      // after the quad transpose lane 4a + k4 holds piece k4 of rows 4a + i
      // (i = 0..3) of this warp's 32: a store instruction covers 64
      // contiguous bytes of each of eight rows
      int rr[4], src[4];
      bool ok[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rr[i] = row_cta + q * 32 + (lane & ~3) + i;
        ok[i] = active && rr[i] < tl.row_end;
        src[i] = 0;
      }
      uint4 g[16];
      if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (ok[i]) {
            src[i] = p.row_src[rr[i]];
            if (unsigned(src[i]) >= unsigned(p.R)) {
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
      if (!pwarp_wait<false>(smem_u32(&c.acc_full[acc]), aph, c, p, peer_abort, lane)) break;
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
          // row `lane` of the chunk as four 16-byte pieces of bf16
          uint4 y[4];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            y[kk].x = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 0]), __uint_as_float(v[8 * kk + 1]));
            y[kk].y = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 2]), __uint_as_float(v[8 * kk + 3]));
            y[kk].z = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 4]), __uint_as_float(v[8 * kk + 5]));
            y[kk].w = pack_bf16x2_rn(__uint_as_float(v[8 * kk + 6]), __uint_as_float(v[8 * kk + 7]));
          }
          quad_transpose(y, lane);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ok[i]) {
              stg_v4(p.out + size_t(rr[i]) * p.N + col0 + ch * 32 + k4 * 8, y[i]);
              if (MODE != int(GemmMode::kFwd)) slot_accumulate8(a[i], g[ch * 4 + i], y[i]);
            }
          }
        }
        if (MODE != int(GemmMode::kFwd)) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float part = slot_tree(a[i]);
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 1));
            part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, 2));
            if (k4 == 0 && ok[i]) {
              if (MODE == int(GemmMode::kSlots))
                p.slots[size_t(col0 / SLOT) * p.R + rr[i]] = part;
              else
                atomicAdd(p.dprob + src[i], part);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(leader ? &c.acc_empty[acc] : &c.acc_read[acc]));
      }
      if (++acc == ACC_BUFS) { acc = 0; aph ^= 1u; }
    }
  }

  // No CTA leaves (or frees tensor memory) while the other may still touch
  // its shared memory or the leader's MMAs may still write its accumulators.
  __syncthreads();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == int(gridDim.x) - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
}

template <int MODE>
cudaError_t launch_pair_mode(const CUtensorMap& ta, const CUtensorMap& tb, const KParams& kp, int grid,
                             cudaStream_t stream) {
  const cudaError_t e =
      ensure_kernel_smem(reinterpret_cast<const void*>(grouped_gemm_pair_kernel<MODE>), int(kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE>, ta, tb, kp);
}

// Largest even CTA count whose pairs can all be resident at once (per device).
template <int MODE>
int compute_resident_pair_ctas() {
  if (ensure_kernel_smem(reinterpret_cast<const void*>(grouped_gemm_pair_kernel<MODE>), int(kSmemBytes)) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(device_sm_count() & ~1), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_pair_kernel<MODE>, &cfg) != cudaSuccess || clusters < 1)
    clusters = device_sm_count() / 2;
  return 2 * clusters;
}

template <int MODE>
int resident_pair_ctas() {
  const int n = cached_per_device(reinterpret_cast<const void*>(grouped_gemm_pair_kernel<MODE>),
                                  compute_resident_pair_ctas<MODE>);
  return n > 0 ? n : 2;
}

template <int MODE>
cudaError_t launch_pairs(const GemmArgs& a, cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, a.X, uint64_t(a.R), uint64_t(a.K), BM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, a.W, uint64_t(a.E) * a.N, uint64_t(a.K), BNH)) return cudaErrorInvalidValue;
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
  kp.status = a.status;
  kp.sched = a.sched;
  if (!kp.sched) return cudaErrorInvalidValue;
  kp.stall_test = (a.flags & DMOE_LAUNCH_TEST_STALL) ? 1 : 0;
  kp.wait_ns = kp.stall_test ? 200ull * 1000ull * 1000ull : kWaitLimitNs;
  const int resident = resident_pair_ctas<MODE>();
  int grid = a.num_ctas > 0 ? a.num_ctas : resident;
  grid = grid < resident ? grid : resident;    // every pair resident: no pair waits on a queued one
  grid &= ~1;
  if (grid < 2) grid = 2;
  return launch_pair_mode<MODE>(ta, tb, kp, grid, stream);
}

}  // namespace

// Both kernels give the same bits; the choice is about speed only.  CTA
// pairs halve the operand traffic per SM but work on 256-row tiles, which
// waste more rows when experts are small: without reading the (device-side)
// offsets, pick pairs when the mean expert has at least kPairMinMeanRows rows.
constexpr long long kPairMinMeanRows = 512;

cudaError_t launch_grouped_gemm(GemmMode mode, const GemmArgs& a, cudaStream_t stream) {
  bool pairs;
  if (mode == GemmMode::kSerial) pairs = false;   // the serialized control has one kernel
  else if (a.flags & DMOE_LAUNCH_SINGLE_CTA) pairs = false;
  else if (a.flags & DMOE_LAUNCH_CTA_PAIRS) pairs = true;
  else pairs = (long long)a.R >= kPairMinMeanRows * a.E;
  if (!pairs) return launch_grouped_gemm_1sm(mode, a, stream);
  if (a.R == 0) return cudaSuccess;
  switch (mode) {
    case GemmMode::kFwd: return launch_pairs<int(GemmMode::kFwd)>(a, stream);
    case GemmMode::kSlots: return launch_pairs<int(GemmMode::kSlots)>(a, stream);
    case GemmMode::kAtomic: return launch_pairs<int(GemmMode::kAtomic)>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dmoe
