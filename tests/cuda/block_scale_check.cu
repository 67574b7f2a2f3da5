// Exhaustive check of the NVFP4 block-scale division (block_scale.cuh) against
// the compiler's correctly rounded binary32 division: for every positive
// finite E4M3 scale value s and every binary32 significand, dividends a of
// both signs in the six binades that put a / s between 2^-3 and 2^3 (every
// E2M1 rounding boundary and the saturation at 6 lie there) must give
// bit-identical quotients.  Test infrastructure only: built and run by the GPU
// tests, never linked into the library.
#include <cstdint>
#include <cuda_runtime.h>

#include "block_scale.cuh"

namespace {

__device__ float e4m3_value(int c) {
  const int e = (c >> 3) & 0xF;
  const int m = c & 0x7;
  if (e == 0) return float(m) * 0.001953125f;                     // m * 2^-9
  return float(8 + m) * __uint_as_float(uint32_t(127 + e - 10) << 23);
}

__global__ void check_kernel(unsigned long long* mismatches, unsigned long long* first) {
  const int code = 1 + int(blockIdx.y);                          // 1 .. 126
  const float s = e4m3_value(code);
  const float y = __frcp_rn(s);
  const float2 nb = make_float2(-s, -s);
  const float2 y2 = make_float2(y, y);
  const int eb = ilogbf(s);
  const uint32_t n = 1u << 23;
  for (uint32_t m = blockIdx.x * blockDim.x + threadIdx.x; m < n; m += gridDim.x * blockDim.x) {
    for (int j = -2; j <= 3; ++j) {
      const float a = __uint_as_float((uint32_t(127 + eb + j) << 23) | m);
      const float2 q = dmoe::div2_by_block_scale(make_float2(a, -a), nb, y2);
      const float ref = __fdiv_rn(a, s);
      if (__float_as_uint(q.x) != __float_as_uint(ref) || __float_as_uint(q.y) != __float_as_uint(-ref)) {
        atomicAdd(mismatches, 1ull);
        atomicCAS(first, ~0ull, (unsigned long long)code << 40 | (unsigned long long)(j + 8) << 32 | m);
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // signed zeros keep their sign
    const float2 z = dmoe::div2_by_block_scale(make_float2(0.0f, -0.0f), nb, y2);
    if (__float_as_uint(z.x) != 0u || __float_as_uint(z.y) != 0x80000000u) atomicAdd(mismatches, 1ull);
  }
}

}  // namespace

// Returns a cudaError_t; *mismatches = failing cases, *first = the first one
// found (code << 40 | (binade + 8) << 32 | significand), all ones if none.
extern "C" int block_scale_check(unsigned long long* mismatches, unsigned long long* first) {
  unsigned long long* d = nullptr;
  cudaError_t e = cudaMalloc(&d, 2 * sizeof(unsigned long long));
  if (e != cudaSuccess) return int(e);
  const unsigned long long init[2] = {0ull, ~0ull};
  e = cudaMemcpy(d, init, sizeof(init), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    check_kernel<<<dim3(2048, 126), 256>>>(d, d + 1);
    e = cudaGetLastError();
  }
  unsigned long long h[2] = {0ull, 0ull};
  if (e == cudaSuccess) e = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  *mismatches = h[0];
  *first = h[1];
  return int(e);
}
