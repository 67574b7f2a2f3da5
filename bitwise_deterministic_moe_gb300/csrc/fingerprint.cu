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
// The pass is HBM-bound: 16-byte loads, about a dozen integer ops per word.
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int kThreads = 256;
constexpr size_t kPartBytes = 16 * 1024;   // bytes of one chunk handled by one CTA

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

// 1-D grid, block = chunk * parts + part.  VEC: data is 16-byte aligned.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
fp_positional_kernel(const uint8_t* __restrict__ data, size_t nbytes, size_t chunk_bytes, unsigned parts,
                     unsigned long long* __restrict__ acc) {
  pdl_begin();
  const size_t c = blockIdx.x / parts;
  const size_t b0 = c * chunk_bytes + size_t(blockIdx.x % parts) * kPartBytes;
  const size_t chunk_end = min(nbytes, (c + 1) * chunk_bytes);
  if (b0 >= chunk_end) return;
  const size_t b1 = min(chunk_end, b0 + kPartBytes);
  uint64_t sum = 0;
  // 16-byte groups fully inside [b0, b1)
  const size_t nfull = (b1 - b0) / 16;
  for (size_t v = threadIdx.x; v < nfull; v += kThreads) {
    const size_t off = b0 + v * 16;
    uint32_t w[4];
    if (VEC) {
      const uint4 q = ldg_nc_v4(data + off);
      w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        w[k] = uint32_t(data[off + 4 * k]) | (uint32_t(data[off + 4 * k + 1]) << 8) |
               (uint32_t(data[off + 4 * k + 2]) << 16) | (uint32_t(data[off + 4 * k + 3]) << 24);
    }
    const uint64_t i0 = off / 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) sum += word_term(w[k], i0 + k);
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
  const uint64_t t = block_sum_u64(sum);
  if (threadIdx.x == 0 && t != 0) atomicAdd(acc + c, (unsigned long long)t);
}

__global__ void fp_finalize_kernel(unsigned long long* __restrict__ acc, size_t nchunks, size_t nbytes,
                                   size_t chunk_bytes) {
  pdl_begin();
  const size_t c = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= nchunks) return;
  const size_t len = min(chunk_bytes, nbytes - c * chunk_bytes);
  acc[c] = sm64(acc[c] ^ (uint64_t(c) << 32) ^ uint64_t(len));
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

template <int ES>
__global__ void __launch_bounds__(kThreads)
fp_xor_kernel(const uint8_t* __restrict__ data, size_t nbytes, size_t chunk_bytes, unsigned parts, int kind,
              unsigned long long* __restrict__ acc) {
  pdl_begin();
  const size_t c = blockIdx.x / parts;
  const size_t b0 = c * chunk_bytes + size_t(blockIdx.x % parts) * kPartBytes;
  const size_t chunk_end = min(nbytes, (c + 1) * chunk_bytes);
  if (b0 >= chunk_end) return;
  const size_t b1 = min(chunk_end, b0 + kPartBytes);
  uint64_t x = 0;
  for (size_t off = b0 + size_t(threadIdx.x) * ES; off < b1; off += size_t(kThreads) * ES)
    x ^= widen<ES>(data + off, kind);
  const uint64_t t = block_xor_u64(x);
  if (threadIdx.x == 0 && t != 0) atomicXor(acc + c, (unsigned long long)t);
}

}  // namespace

cudaError_t launch_fingerprint(const void* data, size_t nbytes, int elem_size, int xor_kind, size_t chunk_bytes,
                               int mode, uint64_t* chunk_hash, cudaStream_t stream) {
  const size_t nchunks = (nbytes + chunk_bytes - 1) / chunk_bytes;
  if (nchunks == 0) return cudaSuccess;
  const size_t parts = (std::min(chunk_bytes, nbytes) + kPartBytes - 1) / kPartBytes;
  if (nchunks * parts > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(chunk_hash, 0, nchunks * sizeof(uint64_t), stream);
  if (e != cudaSuccess) return e;
  auto* acc = reinterpret_cast<unsigned long long*>(chunk_hash);
  const uint8_t* d = static_cast<const uint8_t*>(data);
  const unsigned grid = unsigned(nchunks * parts);
  const unsigned np = unsigned(parts);
  if (mode == 0) {
    if ((reinterpret_cast<uintptr_t>(d) & 15) == 0)
      e = launch_chained(fp_positional_kernel<true>, dim3(grid), dim3(kThreads), 0, stream, d, nbytes, chunk_bytes, np, acc);
    else
      e = launch_chained(fp_positional_kernel<false>, dim3(grid), dim3(kThreads), 0, stream, d, nbytes, chunk_bytes, np, acc);
    if (e != cudaSuccess) return e;
    return launch_chained(fp_finalize_kernel, dim3(unsigned((nchunks + 255) / 256)), dim3(256), 0, stream, acc, nchunks,
                          nbytes, chunk_bytes);
  }
  switch (elem_size) {
    case 1: return launch_chained(fp_xor_kernel<1>, dim3(grid), dim3(kThreads), 0, stream, d, nbytes, chunk_bytes, np, xor_kind, acc);
    case 2: return launch_chained(fp_xor_kernel<2>, dim3(grid), dim3(kThreads), 0, stream, d, nbytes, chunk_bytes, np, xor_kind, acc);
    case 4: return launch_chained(fp_xor_kernel<4>, dim3(grid), dim3(kThreads), 0, stream, d, nbytes, chunk_bytes, np, xor_kind, acc);
    case 8: return launch_chained(fp_xor_kernel<8>, dim3(grid), dim3(kThreads), 0, stream, d, nbytes, chunk_bytes, np, xor_kind, acc);
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dmoe
