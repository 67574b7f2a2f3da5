// Chunk-wise tensor fingerprint on the GPU.
//
// "NVIDIA fait passer le déterminisme bit à bit de Megatron Core à 2432 GPU
// ...", section "Méthodologie de débogage du non-déterminisme": fingerprints are
// computed on the GPU, with shape, dtype and element count recorded, and
// order-sensitive data is fingerprinted chunk by chunk.
//
// Positional mode (raw bits): for chunk c, acc_c = sum over its 32-bit words
// w_i (global word index i, zero-padded tail) of fmix32(w_i ^ i*0x9E3779B9),
// mod 2^64, and the chunk hash is sm64(acc_c ^ (c << 32) ^ chunk_length).
// The sum is an integer sum mod 2^64, associative and commutative, so the
// block partials may land in any order: the bits never depend on scheduling.
// fmix32 is MurmurHash3's finalizer, sm64 splitmix64's output function.
//
// Xor mode: xor of the chunk's elements widened to 64 bits, the reduction
// torch.hash_tensor uses, also order-independent.
//
// One launch: each chunk is hashed by a cluster of eight CTAs, one part of
// the chunk each; the parts' sums meet in distributed shared memory and the
// cluster's first CTA finalizes the chunk -- no atomics, no zero-fill.  The
// clusters are persistent (as many as fit) and loop over the chunks.
// The pass is HBM-bound: 16-byte loads, about a dozen integer ops per word.
#include <algorithm>
#include <mutex>

#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int kUnroll = 8;                 // 16-byte loads in flight per thread
// CTA size: 1024 threads cut the latency of one-chunk buffers; 128 threads
// (more CTAs and clusters resident) stream large buffers faster.
constexpr int kThreadsFew = 1024;
constexpr int kThreadsMany = 128;
constexpr size_t kFewChunks = 8;
constexpr uint32_t kCluster = 8;           // CTAs (parts) per chunk, one cluster

__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  return h;
}

__host__ __device__ __forceinline__ uint64_t sm64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ uint64_t word_term(uint32_t w, uint64_t i) {
  return fmix32(w ^ (uint32_t(i) * 0x9E3779B9u));
}

template <int kThreads>
__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v) {
  __shared__ uint64_t ws[kThreads / 32];
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_down_sync(0xffffffffu, v, d);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) ws[warp] = v;
  __syncthreads();
  uint64_t t = 0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kThreads / 32; ++w) t += ws[w];
  return t;
}

template <int kThreads>
__device__ __forceinline__ uint64_t block_xor_u64(uint64_t v) {
  __shared__ uint64_t ws[kThreads / 32];
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v ^= __shfl_down_sync(0xffffffffu, v, d);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) ws[warp] = v;
  __syncthreads();
  uint64_t t = 0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kThreads / 32; ++w) t ^= ws[w];
  return t;
}

// Grid: persistent clusters of kCluster CTAs; cluster k hashes chunks k,
// k + nclusters, ...; CTA r hashes bytes [c*chunk + r*part, ...) of chunk c.
// VEC: data is 16-byte aligned.
template <bool VEC, int kThreads>
__global__ void __launch_bounds__(kThreads)
fp_positional_kernel(const uint8_t* __restrict__ data, size_t nbytes, size_t chunk_bytes, size_t part_bytes,
                     unsigned long long* __restrict__ out, size_t nchunks) {
  __shared__ unsigned long long part_sum[2];   // double-buffered by chunk parity: one cluster barrier per chunk
  pdl_begin();
  const uint32_t rank = cluster_ctarank();
  const size_t nclusters = gridDim.x / kCluster;
  int it = 0;
  for (size_t c = blockIdx.x / kCluster; c < nchunks; c += nclusters, ++it) {
  const size_t chunk_end = min(nbytes, (c + 1) * chunk_bytes);
  const size_t b0 = min(chunk_end, c * chunk_bytes + size_t(rank) * part_bytes);
  const size_t b1 = min(chunk_end, b0 + part_bytes);
  uint64_t sum = 0;
  // 16-byte groups fully inside [b0, b1), kUnroll of them in flight per thread
  const size_t nfull = (b1 - b0) / 16;
  for (size_t v0 = threadIdx.x; v0 < nfull; v0 += size_t(kThreads) * kUnroll) {
    uint32_t w[kUnroll][4];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t v = v0 + size_t(u) * kThreads;
      if (v >= nfull) continue;
      const size_t off = b0 + v * 16;
      if (VEC) {
        const uint4 q = ldg_nc_v4(data + off);
        w[u][0] = q.x; w[u][1] = q.y; w[u][2] = q.z; w[u][3] = q.w;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          w[u][k] = uint32_t(data[off + 4 * k]) | (uint32_t(data[off + 4 * k + 1]) << 8) |
                    (uint32_t(data[off + 4 * k + 2]) << 16) | (uint32_t(data[off + 4 * k + 3]) << 24);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t v = v0 + size_t(u) * kThreads;
      if (v >= nfull) continue;
      const uint64_t i0 = (b0 + v * 16) / 4;
#pragma unroll
      for (int k = 0; k < 4; ++k) sum += word_term(w[u][k], i0 + k);
    }
  }
  // ragged tail (only at the very end of the buffer): words with 4i < b1
  if (threadIdx.x == 0) {
    for (size_t off = b0 + nfull * 16; off < b1; off += 4) {
      uint32_t w = 0;
      for (int k = 0; k < 4; ++k)
        if (off + k < b1) w |= uint32_t(data[off + k]) << (8 * k);
      sum += word_term(w, off / 4);
    }
  }
  const uint64_t t = block_sum_u64<kThreads>(sum);
  if (threadIdx.x == 0) part_sum[it & 1] = t;
  cluster_sync_all();   // also keeps block_sum's scratch from being reused early
  if (rank == 0 && threadIdx.x == 0) {
    uint64_t acc = 0;
    for (uint32_t r = 0; r < kCluster; ++r)
      acc += ld_shared_cluster_u64(mapa_shared(smem_u32(&part_sum[it & 1]), r));
    const size_t len = chunk_end - c * chunk_bytes;
    out[c] = sm64(acc ^ (uint64_t(c) << 32) ^ uint64_t(len));
  }
  }
  cluster_sync_all();   // no CTA leaves while the first one still reads its sums
}

// xor_kind: 0 unsigned, 1 signed, 2 float16, 3 bfloat16, 4 float32, 5 float64
template <int ES>
__device__ __forceinline__ uint64_t widen(const uint8_t* p, int kind) {
  if (ES == 1) {
    uint8_t u = *p;
    return kind == 1 ? uint64_t(int64_t(int8_t(u))) : uint64_t(u);
  } else if (ES == 2) {
    uint16_t u = *reinterpret_cast<const uint16_t*>(p);
    if (kind == 1) return uint64_t(int64_t(int16_t(u)));
    if (kind == 2) return uint64_t(__double_as_longlong(double(__half2float(__ushort_as_half(u)))));
    if (kind == 3) return uint64_t(__double_as_longlong(double(__uint_as_float(uint32_t(u) << 16))));
    return uint64_t(u);
  } else if (ES == 4) {
    uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    if (kind == 1) return uint64_t(int64_t(int32_t(u)));
    if (kind == 4) return uint64_t(__double_as_longlong(double(__uint_as_float(u))));
    return uint64_t(u);
  } else {
    return *reinterpret_cast<const uint64_t*>(p);
  }
}

template <int ES, int kThreads>
__global__ void __launch_bounds__(kThreads)
fp_xor_kernel(const uint8_t* __restrict__ data, size_t nbytes, size_t chunk_bytes, size_t part_bytes, int kind,
              unsigned long long* __restrict__ out, size_t nchunks) {
  __shared__ unsigned long long part_x[2];
  pdl_begin();
  const uint32_t rank = cluster_ctarank();
  const size_t nclusters = gridDim.x / kCluster;
  int it = 0;
  for (size_t c = blockIdx.x / kCluster; c < nchunks; c += nclusters, ++it) {
  const size_t chunk_end = min(nbytes, (c + 1) * chunk_bytes);
  const size_t b0 = min(chunk_end, c * chunk_bytes + size_t(rank) * part_bytes);
  const size_t b1 = min(chunk_end, b0 + part_bytes);
  uint64_t x = 0;
  for (size_t off = b0 + size_t(threadIdx.x) * ES; off < b1; off += size_t(kThreads) * ES)
    x ^= widen<ES>(data + off, kind);
  const uint64_t t = block_xor_u64<kThreads>(x);
  if (threadIdx.x == 0) part_x[it & 1] = t;
  cluster_sync_all();
  if (rank == 0 && threadIdx.x == 0) {
    uint64_t acc = 0;
    for (uint32_t r = 0; r < kCluster; ++r) acc ^= ld_shared_cluster_u64(mapa_shared(smem_u32(&part_x[it & 1]), r));
    out[c] = acc;
  }
  }
  cluster_sync_all();
}

// Clusters are persistent: as many as can be resident at once (capped by the
// number of chunks), each looping over chunks.
template <int kThreads, typename K, typename... Args>
cudaError_t launch_clustered(K kernel, size_t nchunks, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // resident clusters of this kernel on this device (queried once per device)
  static cudaLaunchConfig_t occ_cfg;
  static cudaLaunchAttribute occ_attr;
  static K occ_kernel;
  static std::mutex occ_mu;
  int max_clusters;
  {
    std::lock_guard<std::mutex> lock(occ_mu);
    occ_cfg = cfg;
    occ_attr = attr[0];
    occ_cfg.attrs = &occ_attr;
    occ_cfg.numAttrs = 1;
    occ_kernel = kernel;
    max_clusters = cached_per_device(reinterpret_cast<const void*>(kernel), []() {
      int n = 0;
      return cudaOccupancyMaxActiveClusters(&n, occ_kernel, &occ_cfg) == cudaSuccess ? n : 0;
    });
  }
  if (max_clusters <= 0) max_clusters = 1;
  const size_t clusters = nchunks < size_t(max_clusters) ? nchunks : size_t(max_clusters);
  cfg.gridDim = dim3(unsigned(clusters * kCluster));
  return cudaLaunchKernelEx(&cfg, kernel, args..., nchunks);
}

}  // namespace

cudaError_t launch_fingerprint(const void* data, size_t nbytes, int elem_size, int xor_kind, size_t chunk_bytes,
                               int mode, uint64_t* chunk_hash, cudaStream_t stream) {
  const size_t nchunks = (nbytes + chunk_bytes - 1) / chunk_bytes;
  if (nchunks == 0) return cudaSuccess;
  if (nchunks * kCluster > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  // parts are 16-byte multiples so that part starts keep the chunk's alignment
  const size_t part = ((chunk_bytes + kCluster - 1) / kCluster + 15) / 16 * 16;
  auto* out = reinterpret_cast<unsigned long long*>(chunk_hash);
  const uint8_t* d = static_cast<const uint8_t*>(data);
  const bool few = nchunks <= kFewChunks;
  if (mode == 0) {
    const bool vec = (reinterpret_cast<uintptr_t>(d) & 15) == 0;
    if (few)
      return vec ? launch_clustered<kThreadsFew>(fp_positional_kernel<true, kThreadsFew>, nchunks, stream, d, nbytes,
                                                 chunk_bytes, part, out)
                 : launch_clustered<kThreadsFew>(fp_positional_kernel<false, kThreadsFew>, nchunks, stream, d, nbytes,
                                                 chunk_bytes, part, out);
    return vec ? launch_clustered<kThreadsMany>(fp_positional_kernel<true, kThreadsMany>, nchunks, stream, d, nbytes,
                                                chunk_bytes, part, out)
               : launch_clustered<kThreadsMany>(fp_positional_kernel<false, kThreadsMany>, nchunks, stream, d, nbytes,
                                                chunk_bytes, part, out);
  }
  switch (elem_size) {
#define DMOE_FP_XOR(ES)                                                                                        \
  case ES:                                                                                                     \
    return few ? launch_clustered<kThreadsFew>(fp_xor_kernel<ES, kThreadsFew>, nchunks, stream, d, nbytes,     \
                                               chunk_bytes, part, xor_kind, out)                               \
               : launch_clustered<kThreadsMany>(fp_xor_kernel<ES, kThreadsMany>, nchunks, stream, d, nbytes,   \
                                                chunk_bytes, part, xor_kind, out);
    DMOE_FP_XOR(1)
    DMOE_FP_XOR(2)
    DMOE_FP_XOR(4)
    DMOE_FP_XOR(8)
#undef DMOE_FP_XOR
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dmoe
