// Block-scaled low-precision encodings of bf16 tensors: MXFP8 and NVFP4.
//
// The pages fingerprint the encoded values and the scale buffers of MXFP8 and
// NVFP4 tensors ("NVIDIA fait passer le déterminisme bit à bit de Megatron Core
// à 2432 GPU ...", section "Méthodologie de débogage du non-déterminisme"), so
// both encoders must produce identical bytes on every run.  Every output byte
// is a function of its own block (plus, for NVFP4, the tensor's maximum, an
// order-independent reduction), computed by one thread with conversions that
// round to nearest even: nothing depends on the grid or on scheduling.
//
// MXFP8 (OCP Microscaling Formats v1.0): a block of 32 consecutive values of a
// row shares the E8M0 scale X = 2^s, s = floor(log2(amax)) - 8 (8 = the E4M3
// maximum exponent), s >= -127; elements are E4M3(v / X), saturating at 448.
// A block holding a NaN or an infinity gets scale 0xFF and elements 0x7F.
//
// NVFP4: 16-value blocks, E4M3 block scale and an fp32 tensor scale, all in
// binary32 in this order: S_enc = 2688 / amax_tensor (1 if amax is 0);
// s_b = E4M3((amax_b / 6) * S_enc); q_i = E2M1((x_i * S_enc) / value(s_b)),
// 0 when s_b is 0; two E2M1 codes per byte, element 2i in the low nibble.
//
// Both passes are HBM-bound: 16-byte loads, one thread per block.  The NVFP4
// encode pass divides by the block scale through one correctly rounded
// reciprocal per block and a two-fma correction per element (block_scale.cuh),
// on the packed fp32x2 pipe, instead of sixteen divisions.
#include "block_scale.cuh"
#include "common.cuh"
#include "internal.h"

namespace dmoe {
namespace {

constexpr int kThreads = 256;

// two fp32 -> packed E4M3 pair (lo in bits 0..7), nearest even, saturating
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// eight fp32 -> four bytes of packed E2M1 pairs (element 2i in the low nibble)
__device__ __forceinline__ uint32_t pack_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  f[0] = bf16lo(q.x); f[1] = bf16hi(q.x);
  f[2] = bf16lo(q.y); f[3] = bf16hi(q.y);
  f[4] = bf16lo(q.z); f[5] = bf16hi(q.z);
  f[6] = bf16lo(q.w); f[7] = bf16hi(q.w);
}

// value of a non-negative E4M3 code (exponent bias 7, 3 fraction bits), exactly
__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
  const int e = (c >> 3) & 0xF;
  const int m = c & 0x7;
  if (e == 0) return float(m) * 0.001953125f;                       // m * 2^-9
  return float(8 + m) * __uint_as_float(uint32_t(127 + e - 10) << 23);   // (8 + m) * 2^(e-10)
}

// floor(log2(a)) of a positive finite fp32 (normal or subnormal), exactly
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t u = __float_as_uint(a);
  const int e = int((u >> 23) & 0xFF);
  if (e > 0) return e - 127;
  return (31 - __clz(int(u & 0x7FFFFF))) - 149;
}

__global__ void __launch_bounds__(kThreads)
mxfp8_kernel(const uint4* __restrict__ x, long long nblocks, uint4* __restrict__ vals, uint8_t* __restrict__ scales) {
  pdl_begin();
  for (long long b = blockIdx.x * (long long)kThreads + threadIdx.x; b < nblocks;
       b += (long long)gridDim.x * kThreads) {
    float f[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float t[8];
      unpack8(ldg_nc_v4(x + b * 4 + i), t);
#pragma unroll
      for (int j = 0; j < 8; ++j) f[i * 8 + j] = t[j];
    }
    float amax = 0.f;
    bool finite = true;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float a = fabsf(f[j]);
      finite = finite && (a <= 3.402823466e38f);   // false for NaN and infinity
      amax = fmaxf(amax, a);
    }
    uint4 o0, o1;
    uint8_t sc;
    if (!finite) {
      o0 = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      o1 = o0;
      sc = 0xFF;
    } else {
      int s = amax > 0.f ? floor_log2(amax) - 8 : -127;
      if (s < -127) s = -127;
      sc = uint8_t(s + 127);
      const float inv = __uint_as_float(uint32_t(127 - s) << 23);   // 2^-s, a normal fp32 for s in [-127, 119]
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t lo = pack_e4m3x2(__fmul_rn(f[4 * k], inv), __fmul_rn(f[4 * k + 1], inv));
        const uint32_t hi = pack_e4m3x2(__fmul_rn(f[4 * k + 2], inv), __fmul_rn(f[4 * k + 3], inv));
        w[k] = lo | (hi << 16);
      }
      o0 = make_uint4(w[0], w[1], w[2], w[3]);
      o1 = make_uint4(w[4], w[5], w[6], w[7]);
    }
    vals[b * 2] = o0;
    vals[b * 2 + 1] = o1;
    scales[b] = sc;
  }
}

// max |x| over the tensor as fp32 bits (non-negative floats order like their bits)
__global__ void __launch_bounds__(kThreads)
amax_kernel(const uint4* __restrict__ x, long long nvec, unsigned int* __restrict__ amax_bits) {
  pdl_begin();
  float m = 0.f;
  const long long stride = (long long)gridDim.x * kThreads;
  for (long long i0 = blockIdx.x * (long long)kThreads + threadIdx.x; i0 < nvec; i0 += stride * 8) {
    uint4 q[8];   // eight 16-byte loads in flight per thread
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const long long i = i0 + u * stride;
      q[u] = i < nvec ? ldg_nc_v4(x + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float t[8];
      unpack8(q[u], t);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(t[j]));
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax_bits, __float_as_uint(m));
}

// |x| maximum of eight packed bf16 pairs, as fp32 (max of non-negative values is exact in bf16)
__device__ __forceinline__ float block_amax16(const uint4& p0, const uint4& p1) {
  const uint32_t w[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(w[i] & 0x7FFF7FFFu));
  return fmaxf(bf16lo(m), bf16hi(m));
}

__global__ void __launch_bounds__(kThreads)
nvfp4_kernel(const uint4* __restrict__ x, long long nblocks, const unsigned int* __restrict__ amax_bits,
             uint2* __restrict__ packed, uint8_t* __restrict__ scales, float* __restrict__ s_enc_out) {
  pdl_begin();
  const float amax_t = __uint_as_float(*amax_bits);
  const float s_enc = amax_t > 0.f ? __fdiv_rn(2688.0f, amax_t) : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *s_enc_out = s_enc;
  const float2 s_enc2 = make_float2(s_enc, s_enc);
  const long long stride = (long long)gridDim.x * kThreads;
  for (long long b0 = blockIdx.x * (long long)kThreads + threadIdx.x; b0 < nblocks; b0 += stride * 2) {
    // two blocks per thread per round: four 16-byte loads in flight
    uint4 in[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long b = b0 + u * stride;
      in[u][0] = b < nblocks ? ldg_nc_v4(x + b * 2) : make_uint4(0u, 0u, 0u, 0u);
      in[u][1] = b < nblocks ? ldg_nc_v4(x + b * 2 + 1) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long b = b0 + u * stride;
      if (b >= nblocks) break;
      const float amax = block_amax16(in[u][0], in[u][1]);
      const float dec = __fmul_rn(__fdiv_rn(amax, 6.0f), s_enc);
      const uint8_t sb = uint8_t(pack_e4m3x2(dec, 0.f) & 0xFF);
      uint2 out = make_uint2(0u, 0u);   // a zero scale encodes every element as +0
      if (sb != 0) {
        const float sv = e4m3_to_float(sb);
        const float y = __frcp_rn(sv);
        const float2 nb = make_float2(-sv, -sv);
        const float2 y2 = make_float2(y, y);
        const uint32_t w[8] = {in[u][0].x, in[u][0].y, in[u][0].z, in[u][0].w,
                               in[u][1].x, in[u][1].y, in[u][1].z, in[u][1].w};
        float h[2][8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 a = __fmul2_rn(make_float2(bf16lo(w[i]), bf16hi(w[i])), s_enc2);
          const float2 q = div2_by_block_scale(a, nb, y2);
          h[i >> 2][2 * (i & 3)] = q.x;
          h[i >> 2][2 * (i & 3) + 1] = q.y;
        }
        out = make_uint2(pack_e2m1x8(h[0]), pack_e2m1x8(h[1]));
      }
      packed[b] = out;
      scales[b] = sb;
    }
  }
}

int grid_for(long long work) {
  const long long cap = (long long)device_sm_count() * 8;
  const long long g = (work + kThreads - 1) / kThreads;
  return int(g < 1 ? 1 : (g < cap ? g : cap));
}

}  // namespace

cudaError_t launch_quantize_mxfp8(const void* x, long long n, void* vals, void* scales, cudaStream_t stream) {
  const long long nblocks = n / 32;
  if (nblocks == 0) return cudaSuccess;
  return launch_chained(mxfp8_kernel, dim3(grid_for(nblocks)), dim3(kThreads), 0, stream, static_cast<const uint4*>(x),
                        nblocks, static_cast<uint4*>(vals), static_cast<uint8_t*>(scales));
}

cudaError_t launch_quantize_nvfp4(const void* x, long long n, void* packed, void* scales, float* s_enc,
                                  unsigned int* amax_scratch, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax_scratch, 0, sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  const long long nvec = n / 8;
  if (nvec > 0) {
    e = launch_chained(amax_kernel, dim3(grid_for(nvec)), dim3(kThreads), 0, stream, static_cast<const uint4*>(x), nvec,
                       amax_scratch);
    if (e != cudaSuccess) return e;
  }
  const long long nblocks = n / 16;
  return launch_chained(nvfp4_kernel, dim3(grid_for(nblocks)), dim3(kThreads), 0, stream,
                        static_cast<const uint4*>(x), nblocks, static_cast<const unsigned int*>(amax_scratch),
                        static_cast<uint2*>(packed), static_cast<uint8_t*>(scales), s_enc);
}

}  // namespace dmoe
