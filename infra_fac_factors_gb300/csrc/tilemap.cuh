// Upper-tile work units of a d x d symmetric factor (host and device).
//
// The factor is cut into 128-row blocks.  Row block i covers rows
// [128 i, 128 i + 128) and, because the factor is symmetric, only the columns
// [128 i, d) are computed (the upper tiles; SPD-KFAC §III-A counts a factor by
// its upper triangle).  Those columns are cut into chunks of at most 256, one
// work unit each: unit = (row block i, first column j0, width w).  Units are
// numbered row block by row block, left to right.
#pragma once
#include <math.h>
#include <stdint.h>

namespace kfac {

constexpr int kTileM = 128;  // rows per unit (tcgen05 M)
constexpr int kTileN = 256;  // max columns per unit (tcgen05 N)

__host__ __device__ inline int64_t units_in_row_block(int64_t d, int64_t i) {
  return (d - kTileM * i + kTileN - 1) / kTileN;
}

__host__ __device__ inline int64_t factor_units(int64_t d) {
  const int64_t T = (d + kTileM - 1) / kTileM;
  int64_t n = 0;
  for (int64_t i = 0; i < T; ++i) n += units_in_row_block(d, i);
  return n;
}

// Unit t (0 <= t < factor_units(d)) -> (i, j0, w).
__host__ __device__ inline void factor_unit(int64_t d, int64_t t, int& i, int64_t& j0, int& w) {
  const int64_t T = (d + kTileM - 1) / kTileM;
  for (int64_t r = 0; r < T; ++r) {
    const int64_t n = units_in_row_block(d, r);
    if (t < n) {
      i = (int)r;
      j0 = kTileM * r + kTileN * t;
      const int64_t rem = d - j0;
      w = (int)(rem < kTileN ? rem : kTileN);
      return;
    }
    t -= n;
  }
  i = -1;
  j0 = 0;
  w = 0;
}

// The same map in constant time (32-bit; t < 2^31).  Row blocks 2k and 2k + 1
// hold n0 - k and n1 - k units (n0 = ceil(d / 256), n1 = floor((d + 127) / 256);
// a row block past the factor's last one holds none), so the units of the
// first k pairs of row blocks number C(k) = k (n0 + n1) - k (k - 1), and the
// pair of unit t is the largest k with C(k) <= t (a quadratic, inverted with
// one fp32 square root and corrected by +-1).
__host__ __device__ inline void factor_unit_fast(int d, int t, int& i, int& j0, int& w) {
  const int n0 = (d + 255) / 256, n1 = (d + 127) / 256, s = n0 + n1;
  auto C = [&](int k) { return k * s - k * (k - 1); };
  const float disc = (float)(s + 1) * (float)(s + 1) - 4.0f * (float)t;  // rounding is corrected below
  int k = (int)(((float)(s + 1) - sqrtf(disc > 0.f ? disc : 0.f)) * 0.5f);
  if (k < 0) k = 0;
  while (k > 0 && C(k) > t) --k;
  while (C(k + 1) <= t && k + 1 <= n0) ++k;
  const int rem = t - C(k);
  int r, u;
  if (rem < n0 - k) {
    r = 2 * k;
    u = rem;
  } else {
    r = 2 * k + 1;
    u = rem - (n0 - k);
  }
  i = r;
  j0 = kTileM * r + kTileN * u;
  const int left = d - j0;
  w = left < kTileN ? left : kTileN;
}

}  // namespace kfac
