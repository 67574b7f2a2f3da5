// Deterministic grouped-GEMM weight gradient for GB300 (sm_103a):
//
//   dW[e, n, c] (+)= sum over expert e's rows r (ascending blocks of 64) of dY[r, n] * X[r, c]
//
// the gradient of the FFN-out projection's weight W[e] [N, K] for
// expert_out = X_e W_e^T.  A weight-gradient path is one of the workloads whose
// determinism overhead the pages measure ("Trillion-Parameter Pretraining Goes
// Bitwise-Deterministic: NVIDIA Cuts the Determinism Tax to About 2%", section
// "Synopsis"; "NVIDIA fait passer le déterminisme bit à bit de Megatron Core à
// 2432 GPU ...", section "Optimisation pour le Nemotron à mille milliards de
// paramètres").  The usual nondeterminism of such a kernel comes from split-K
// partial sums added atomically; here every output tile is reduced by one CTA
// over all of its expert's rows in ascending order, so no two writers meet and
// the bits do not depend on the grid, the stream or the schedule.
//
// The reduction runs over rows, so both operands are read "MN-major": the
// 128 n-values of a dY tile and the 256 c-values of an X tile are contiguous in
// memory.  TMA loads boxes of 64 rows x 64 elements (128 bytes, 128-byte
// swizzle) and the shared-memory descriptors describe that layout: 64-element
// boxes LBO = 8 KB apart along M/N, 8-row groups SBO = 1 KB apart along the
// reduction, 2 KB per 16-row MMA step.
//
// Design (one CTA per SM, persistent, warp-specialised, 352 threads):
//   warp 0     TMA producer: per stage dY [64 r x 128 n] and X [64 r x 256 c].
//   warp 1     tcgen05.mma issuer (lane 0): 128x256x16 MMAs, fp32 in tensor
//              memory (2 x 256 columns).  In a tile's last stage only the
//              16-row steps holding the expert's rows are issued, and the whole
//              warp first zeroes the rows of the last step that belong to the
//              next expert, so no row is ever counted twice.
//   warps 2-9  epilogue: tensor memory -> registers -> swizzled shared memory ->
//              TMA tensor stores of dW (add-reduce stores in accumulate mode).
//   warp 10    tile scheduler: claims tiles and decodes each into (expert,
//              rows, n and c offsets) a few tiles ahead of use, so the
//              producer goes from one tile's last row block to the next
//              tile's first without a pause (light experts' tiles are only one
//              or two row blocks long).
// Tiles (one 128 x 256 block of one expert's dW) of experts with many rows come
// first, then the rest, each class in expert order, handed out dynamically.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace dmoe {

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
bool make_tmap_f32_store(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);

namespace {

constexpr int BM = 128;                  // dW rows (n) per tile = UMMA M
constexpr int BN = 256;                  // dW columns (c) per tile = UMMA N
constexpr int BK = 64;                   // reduction rows per stage
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int BOX_BYTES = BK * 128;      // 64 rows x 64 bf16
constexpr int A_STAGE_BYTES = (BM / 64) * BOX_BYTES;
constexpr int B_STAGE_BYTES = (BN / 64) * BOX_BYTES;
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int BOXES = STAGE_BYTES / BOX_BYTES;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 8;
constexpr int SCHED_WARP = EPI_WARP0 + EPI_WARPS;
constexpr int NUM_THREADS = 32 * (SCHED_WARP + 1);
constexpr int TQ = 4;
constexpr int HEAVY_KB = 16;             // experts with >= 16 row blocks (1024 rows) go first
constexpr int STG_BYTES = 32 * 64;       // per epilogue warp: 32 rows x 16 fp32

// A decoded tile as the scheduler queues it (cur = -1: no more tiles).
struct alignas(16) WTile {
  int cur, e, row0, rows, n0, c0, pad0, pad1;
};

struct alignas(16) Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[ACC_BUFS];
  uint64_t acc_empty[ACC_BUFS];
  uint64_t mma_done;
  uint64_t tq_full[TQ];
  uint64_t tq_empty[TQ];
  WTile tq[TQ];
  uint32_t tmem_base;
  int abort;
  int off[DMOE_MAX_EXPERTS + 1];
  int hp[DMOE_MAX_EXPERTS + 1];          // exclusive prefix count of heavy experts
  int lp[DMOE_MAX_EXPERTS + 1];          // exclusive prefix count of the other experts
};

constexpr size_t kSmemBytes = 1024 + size_t(STAGES) * STAGE_BYTES + size_t(EPI_WARPS) * STG_BYTES + sizeof(Ctrl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct KParams {
  const int32_t* offsets;
  int E, R, K, N, NTn, NTc;
  float* dW;
  int accumulate;
  int* status;
  int* sched;
  unsigned long long wait_ns;
};

// Descriptor of an MN-major operand tile written by TMA as 64-element boxes
// with 128-byte swizzling: boxes BOX_BYTES apart (leading byte offset), 8-row
// groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t smem_desc_mn128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(BOX_BYTES >> 4) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// kind::f16, fp32 D, bf16 A and B, both MN-major (bits 15, 16), M=128, N=256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                            (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

// Tile t: heavy experts' tiles first (expert order), then the others; inside
// an expert, the n-tile varies fastest.  Only the timing depends on it.
// Decoded by the whole scheduler warp: the expert is the largest e < E whose
// class prefix count is <= u (two ballots over the shared tables, E <= 1024).
__device__ __forceinline__ WTile decode_tile_warp(int t, const Ctrl& c, int E, int NTn, int NTc, int heavy_tiles,
                                                  int lane) {
  const int per = NTn * NTc;
  const bool heavy = t < heavy_tiles;
  const int u = heavy ? t / per : (t - heavy_tiles) / per;
  const int j = heavy ? t % per : (t - heavy_tiles) % per;
  const int* pre = heavy ? c.hp : c.lp;
  const int e1 = lane * 32;
  const unsigned m1 = __ballot_sync(0xffffffffu, e1 < E && pre[e1] <= u);   // lane 0 always (pre[0] = 0)
  const int seg = 31 - __clz(m1);
  const int e2 = seg * 32 + lane;
  const unsigned m2 = __ballot_sync(0xffffffffu, e2 < E && pre[e2] <= u);
  const int e = seg * 32 + (31 - __clz(m2));
  WTile tl;
  tl.cur = t;
  tl.e = e;
  tl.row0 = c.off[e];
  tl.rows = c.off[e + 1] - c.off[e];
  tl.n0 = (j % NTn) * BM;
  tl.c0 = (j / NTn) * BN;
  tl.pad0 = tl.pad1 = 0;
  return tl;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_wgrad_kernel(const __grid_constant__ CUtensorMap tmap_dy, const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_dw, const KParams p) {
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
      mbar_init(smem_u32(&c.tq_empty[i]), 2 + EPI_WARPS);   // producer, MMA warp, epilogue warps
    }
    c.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_dy);
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_dw);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  pdl_begin();   // no global memory is touched above this line
  for (int e = tid; e <= E; e += NUM_THREADS) c.off[e] = p.offsets[e];
  __syncthreads();
  int bad = 0;
  for (int e = tid; e < E; e += NUM_THREADS) {
    const int a = c.off[e], b = c.off[e + 1];
    if (b < a) bad = 1;
    const bool heavy = (b - a) >= HEAVY_KB * BK;
    c.hp[e + 1] = heavy ? 1 : 0;
    c.lp[e + 1] = heavy ? 0 : 1;
  }
  if (tid == 0) {
    if (c.off[0] != 0 || c.off[E] != p.R) bad = 1;
    c.hp[0] = 0;
    c.lp[0] = 0;
  }
  bad = __syncthreads_or(bad);
  if (warp < 2) {
    int* pre = warp == 0 ? c.hp : c.lp;
    int carry = 0;
    for (int b0 = 1; b0 <= E; b0 += 32) {
      const int i = b0 + lane;
      int v = (i <= E) ? pre[i] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, d);
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
  const int per = p.NTn * p.NTc;
  const int heavy_tiles = c.hp[E] * per;
  const int total_tiles = bad ? 0 : E * per;
  const uint32_t tmem_base = c.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int issued_total = 0;
      int stage = 0;
      uint32_t ph = 0;
      for (int qi = 0;; ++qi) {
        const int qs = qi % TQ;
        if (!mbar_wait(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), &c.abort, p.status, p.wait_ns)) break;
        const WTile tl = c.tq[qs];
        mbar_arrive(smem_u32(&c.tq_empty[qs]));
        if (tl.cur < 0) break;
        const int KB = (tl.rows + BK - 1) / BK;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&c.empty[stage]), ph ^ 1u, &c.abort, p.status, p.wait_ns)) { ok = false; break; }
          const uint32_t full = smem_u32(&c.full[stage]);
          const uint32_t sa = stage0 + stage * STAGE_BYTES;
          const int y = tl.row0 + kb * BK;   // rows past R are filled with zeros by the TMA unit
          mbar_arrive_expect_tx(full, STAGE_BYTES);
#pragma unroll
          for (int b = 0; b < BM / 64; ++b)
            tma_load_2d(sa + b * BOX_BYTES, &tmap_dy, full, tl.n0 + b * 64, y);
#pragma unroll
          for (int b = 0; b < BN / 64; ++b)   // boxes at c >= K are filled with zeros
            tma_load_2d(sa + A_STAGE_BYTES + b * BOX_BYTES, &tmap_x, full, tl.c0 + b * 64, y);
          ++issued_total;
          if (++stage == STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
      }
      // let every copy this thread started land before the CTA can exit
      for (int s = 0; s < STAGES; ++s) {
        const int n = (issued_total - s + STAGES - 1) / STAGES;
        if (n > 0) mbar_wait_drain(smem_u32(&c.full[s]), uint32_t(n - 1) & 1u, p.wait_ns / 4);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------- MMA issuer (whole warp)
    int stage = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t aph = 0;
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      if (!warp_wait(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), &c.abort, p.status, lane, p.wait_ns)) break;
      const WTile tl = c.tq[qs];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.tq_empty[qs]));
      if (tl.cur < 0) break;
      const int KB = (tl.rows + BK - 1) / BK;
      if (KB == 0) continue;   // an expert without rows: the epilogue writes zeros
      if (!warp_wait(smem_u32(&c.acc_empty[acc]), aph ^ 1u, &c.abort, p.status, lane, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!warp_wait(smem_u32(&c.full[stage]), ph, &c.abort, p.status, lane, p.wait_ns)) { ok = false; break; }
        const uint32_t sa = stage0 + stage * STAGE_BYTES;
        const int valid = min(tl.rows - kb * BK, BK);
        const int groups = (valid + UMMA_K - 1) / UMMA_K;   // 16-row MMA steps holding the expert's rows
        const int pad_end = groups * UMMA_K;
        if (valid < pad_end) {
          // Rows valid..pad_end-1 of the last 16-row step belong to the next
          // expert (or lie past R): zero them in every box (a row is one
          // 128-byte line of a box; the swizzle only permutes 16-byte pieces
          // inside it).  Steps past pad_end are not issued at all.
          const int words = (pad_end - valid) * 8;
          for (int i = lane; i < BOXES * words; i += 32) {
            const int b = i / words;
            const int w = i - b * words;
            sts_v4(sa + uint32_t(b * BOX_BYTES + valid * 128 + w * 16), make_uint4(0u, 0u, 0u, 0u));
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint64_t adesc = smem_desc_mn128(sa);
          const uint64_t bdesc = smem_desc_mn128(sa + A_STAGE_BYTES);
          for (int kk = 0; kk < groups; ++kk) {
            // 16 rows = two 8-row groups = 2 KB further along the reduction
            tc_mma_f16(d_tmem, adesc + uint64_t(kk * 128), bdesc + uint64_t(kk * 128), kIdesc,
                       (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&c.empty[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; ph ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(smem_u32(&c.acc_full[acc]));
      __syncwarp();
      if (++acc == ACC_BUFS) { acc = 0; aph ^= 1u; }
    }
    if (lane == 0) {
      // every MMA must be finished before tensor memory is released
      tc_commit(smem_u32(&c.mma_done));
      mbar_wait_drain(smem_u32(&c.mma_done), 0, p.wait_ns / 4);
    }
    __syncwarp();
  } else if (warp == SCHED_WARP) {
    // -------------------------------------------------- tile scheduler (one warp)
    // first tile = blockIdx.x, then the global counter; each claimed tile is
    // decoded while its queue slot is still in use and queued as soon as it
    // frees, with the next claim in flight meanwhile
    int tile = int(blockIdx.x);
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      const int cur = tile < total_tiles ? tile : -1;
      int nxt = 0;
      if (cur >= 0 && lane == 0) nxt = int(gridDim.x) + atomicAdd(p.sched, 1);
      WTile q{};
      q.cur = -1;
      if (cur >= 0) q = decode_tile_warp(cur, c, E, p.NTn, p.NTc, heavy_tiles, lane);
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
    // Warp w reads TMEM lanes 32*(w%4)..+31 (dW rows n0 + 32q ..); warps 2-5
    // take columns 0..127 of the tile, warps 6-9 columns 128..255.  Each
    // 32-row x 16-column fp32 piece is written to a 2 KB staging buffer in the
    // TMA unit's 64-byte-swizzled layout (piece kk of row r at kk ^ ((r/2)%4),
    // which also keeps the shared-memory writes free of bank conflicts) and
    // sent to dW by one TMA tensor store -- an add-reduce in accumulate mode,
    // one fp32 addition per element.  Columns past K are clipped by the TMA
    // unit.
    const int q = warp & 3;
    const int h = (warp - EPI_WARP0) / 4;
    const uint32_t stg = stage0 + uint32_t(STAGES * STAGE_BYTES + (warp - EPI_WARP0) * STG_BYTES);
    int acc = 0;
    uint32_t aph = 0;
    for (int qi = 0;; ++qi) {
      const int qs = qi % TQ;
      if (!warp_wait(smem_u32(&c.tq_full[qs]), uint32_t((qi / TQ) & 1), &c.abort, p.status, lane, p.wait_ns)) break;
      const WTile tl = c.tq[qs];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.tq_empty[qs]));
      if (tl.cur < 0) break;
      const int col0 = tl.c0 + h * 128;
      float* dw_rows = p.dW + (size_t(tl.e) * p.N + tl.n0 + q * 32) * size_t(p.K);
      if (tl.rows == 0) {
        // an expert without rows: dW[e] = 0 (left as it is when accumulating)
        if (!p.accumulate) {
          for (int r = 0; r < 32; ++r) {
            const int cc = col0 + lane * 4;
            if (cc < p.K) stg_v4(dw_rows + size_t(r) * p.K + cc, make_uint4(0u, 0u, 0u, 0u));
          }
        }
        continue;
      }
      if (!warp_wait(smem_u32(&c.acc_full[acc]), aph, &c.abort, p.status, lane, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t tcol = tmem_base + uint32_t(acc * BN + h * 128) + (uint32_t(q * 32) << 16);
      const int grow = tl.e * p.N + tl.n0 + q * 32;   // row of dW viewed as [E*N, K]
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tcol + uint32_t(ch * 32), v);
        tmem_wait_ld();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int cc = col0 + ch * 32 + half * 16;
          if (lane == 0) bulk_wait_group_read<0>();   // the previous box has left the staging buffer
          __syncwarp();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int j = half * 16 + kk * 4;
            sts_v4(stg + uint32_t(lane * 64 + ((kk ^ ((lane >> 1) & 3)) << 4)),
                   make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && cc < p.K) {
            if (p.accumulate)
              tma_reduce_add_2d(&tmap_dw, stg, cc, grow);
            else
              tma_store_2d(&tmap_dw, stg, cc, grow);
            bulk_commit_group();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&c.acc_empty[acc]));
      if (++acc == ACC_BUFS) { acc = 0; aph ^= 1u; }
    }
    if (lane == 0) bulk_wait_group_all();   // every store has landed before the CTA exits
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (tid == 0) {
    // every counter fetch of this CTA (made by its scheduler warp) has
    // returned before the barrier above; the last CTA to finish zeroes the
    // tile counters for the next launch
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == int(gridDim.x) - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
}

}  // namespace

cudaError_t launch_grouped_wgrad(const WgradArgs& a, cudaStream_t stream) {
  const size_t dw_bytes = size_t(a.E) * a.N * a.K * sizeof(float);
  if (a.R == 0) {   // no rows anywhere: every dW[e] is zero
    return a.accumulate ? cudaSuccess : cudaMemsetAsync(a.dW, 0, dw_bytes, stream);
  }
  CUtensorMap tdy, tx, tdw;
  if (!make_tmap_bf16(&tdy, a.dY, uint64_t(a.R), uint64_t(a.N), BK)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tx, a.X, uint64_t(a.R), uint64_t(a.K), BK)) return cudaErrorInvalidValue;
  if (!make_tmap_f32_store(&tdw, a.dW, uint64_t(a.E) * a.N, uint64_t(a.K), 32)) return cudaErrorInvalidValue;
  KParams kp;
  kp.offsets = a.offsets;
  kp.E = a.E;
  kp.R = a.R;
  kp.K = a.K;
  kp.N = a.N;
  kp.NTn = a.N / BM;
  kp.NTc = (a.K + BN - 1) / BN;
  kp.dW = a.dW;
  kp.accumulate = a.accumulate ? 1 : 0;
  kp.status = a.status;
  kp.sched = a.sched;
  kp.wait_ns = kWaitLimitNs;
  if (!kp.sched) return cudaErrorInvalidValue;
  const cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(grouped_wgrad_kernel), int(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = a.num_ctas > 0 ? a.num_ctas : device_sm_count();
  return launch_chained(grouped_wgrad_kernel, dim3(grid), dim3(NUM_THREADS), kSmemBytes, stream, tdy, tx, tdw, kp);
}

}  // namespace dmoe
