// Probe vectors of the inverse's a-posteriori residual checks (host and
// device; no CUDA dependence, so that host tests can include it).
//
// fp32 pass (four probes, every matrix):
//   v_p(i) = s(i) H4[p][c(i)],   p = 0..3,  H4[p][b] = (-1)^popcount(p & b),
// with a sign s(i) and a class c(i) in 0..3 from the splitmix64 finaliser
// of i.  Each v_p alone has independent +-1 entries (a Rademacher vector, so
// E||E v_p||^2 = ||E||_F^2).  Together, sum_p v_p(i) v_p(j) / 4 is
// s(i) s(j) when c(i) = c(j) and zero otherwise: the mean of the four squared
// norms is a sum over the pairs of equal class.  The classes are hashed, not
// i mod 4, so that no periodic structure of the residual can fall into one
// class (that would leave the four probes one projection apart, chi-square
// with one degree of freedom instead of four).  The structure lets D v_p be
// formed from one sum of s(j) D_ij per class of j.
//
// Newton-step decision (sixteen probes, flagged matrices only): independent
// signs, sixteen bits of one hash of i.
#pragma once
#include <stdint.h>

namespace kfac {

__host__ __device__ inline uint64_t probe_mix(uint64_t z) {  // splitmix64 finaliser
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
// s(i) (bit 0 of the hash) and c(i) (bits 1-2)
__host__ __device__ inline float probe_base_sign(long long i) {
  return (probe_mix((uint64_t)i) & 1ull) ? 1.f : -1.f;
}
__host__ __device__ inline int probe_class(long long i) { return (int)((probe_mix((uint64_t)i) >> 1) & 3ull); }
__host__ __device__ inline float hadamard4(int p, int b) {
  const int pb = p & b & 3;
  return ((pb ^ (pb >> 1)) & 1) ? -1.f : 1.f;
}
__host__ __device__ inline float probe4(long long i, int p) { return probe_base_sign(i) * hadamard4(p, probe_class(i)); }
// the Newton-step decision's probes: bit p of one hash of i, apart from the
// stream above (offset 2^40); probe16_bits(i) gives all sixteen at once
constexpr int kProbes16 = 16;
__host__ __device__ inline uint32_t probe16_bits(long long i) {
  return (uint32_t)(probe_mix((uint64_t)i + (1ull << 40)) & 0xFFFFull);
}
__host__ __device__ inline float probe16(long long i, int p) { return ((probe16_bits(i) >> p) & 1u) ? 1.f : -1.f; }

}  // namespace kfac
