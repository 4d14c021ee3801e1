// fp32 -> three bf16 slices (x = hi + mid + lo exactly, for normal x), the
// operand format of the split-bf16 tcgen05 GEMMs.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace kfac {

constexpr int kSlices = 3;

// x -> slices, each carrying the remainder of the previous ones
__device__ __forceinline__ void split_value(float x, __nv_bfloat16 (&s)[kSlices]) {
  float r = x;
#pragma unroll
  for (int k = 0; k < kSlices; ++k) {
    s[k] = __float2bfloat16_rn(r);
    r = r - __bfloat162float(s[k]);
  }
}

// eight consecutive values -> one 16-byte store per slice (dst 16-byte
// aligned); the first NP slices are written
template <int NP = kSlices>
__device__ __forceinline__ void split8_store(const float (&x)[8], uint16_t* dst, long long slice_stride) {
  uint32_t w[kSlices][4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat16 a[kSlices], b[kSlices];
    split_value(x[2 * e], a);
    split_value(x[2 * e + 1], b);
#pragma unroll
    for (int k = 0; k < kSlices; ++k) {
      __nv_bfloat162 p;
      p.x = a[k];
      p.y = b[k];
      w[k][e] = *reinterpret_cast<const uint32_t*>(&p);
    }
  }
#pragma unroll
  for (int k = 0; k < NP; ++k)
    *reinterpret_cast<uint4*>(dst + k * slice_stride) = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
}

}  // namespace kfac
