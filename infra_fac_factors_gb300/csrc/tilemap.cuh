// Upper-tile work units of a d x d symmetric factor (host and device).
//
// The factor is cut into 128-row blocks; because it is symmetric only the
// upper tiles are stored (element (r, c) with c >= 128 floor(r / 128); SPD-KFAC
// §III-A counts a factor by its upper triangle).  The tensor-core SYRK runs
// in CTA pairs that share the column operand, so the units come in pairs:
// row blocks 2s and 2s + 1 ("pair s") both take the columns [256 s, d), cut
// into chunks of at most 256 (n0 - s chunks, n0 = ceil(d / 256)).  Unit
// 2 v + rank of pair-chunk v is (row block 2s + rank, first column j0,
// width w).  Of a unit, only the columns >= 128 i of an existing row block
// i are stored: row block 2s + 1's first chunk starts with its lower tile
// (2s + 1, 2s), which is computed and dropped, and with an odd number of row
// blocks the last pair's second unit is a stand-in that stores nothing.
// Pair-chunks are numbered pair by pair, left to right.
#pragma once
#include <math.h>
#include <stdint.h>

namespace kfac {

constexpr int kTileM = 128;  // rows per unit (tcgen05 M)
constexpr int kTileN = 256;  // max columns per unit (tcgen05 N)

__host__ __device__ inline int64_t pair_chunks(int64_t d) {
  const int64_t n0 = (d + kTileN - 1) / kTileN;
  return n0 * (n0 + 1) / 2;
}

__host__ __device__ inline int64_t factor_units(int64_t d) { return 2 * pair_chunks(d); }

// Unit t (0 <= t < factor_units(d)) -> (i, j0, w), by enumeration.
__host__ __device__ inline void factor_unit(int64_t d, int64_t t, int& i, int64_t& j0, int& w) {
  const int64_t n0 = (d + kTileN - 1) / kTileN;
  int64_t v = t / 2;
  for (int64_t s = 0; s < n0; ++s) {
    if (v < n0 - s) {
      i = (int)(2 * s + t % 2);
      j0 = kTileN * (s + v);
      const int64_t rem = d - j0;
      w = (int)(rem < kTileN ? rem : kTileN);
      return;
    }
    v -= n0 - s;
  }
  i = -1;
  j0 = 0;
  w = 0;
}

// The same map in constant time (32-bit; t < 2^31).  The pairs before s hold
// C(s) = s n0 - s (s - 1) / 2 pair-chunks; the pair of pair-chunk v is the
// largest s with C(s) <= v (a quadratic, inverted with one fp32 square root
// and corrected by +-1).
__host__ __device__ inline void factor_unit_fast(int d, int t, int& i, int& j0, int& w) {
  const int n0 = (d + kTileN - 1) / kTileN;
  const int v = t >> 1;
  auto C = [&](int s) { return s * n0 - s * (s - 1) / 2; };
  const float b = 2.0f * (float)n0 + 1.0f;
  const float disc = b * b - 8.0f * (float)v;  // rounding is corrected below
  int s = (int)((b - sqrtf(disc > 0.f ? disc : 0.f)) * 0.5f);
  if (s < 0) s = 0;
  if (s > n0 - 1) s = n0 - 1;
  while (s > 0 && C(s) > v) --s;
  while (s + 1 < n0 && C(s + 1) <= v) ++s;
  i = 2 * s + (t & 1);
  j0 = kTileN * (s + (v - C(s)));
  const int left = d - j0;
  w = left < kTileN ? left : kTileN;
}

}  // namespace kfac
