// Host/device interface of the split-bf16 tcgen05 GEMM (gemm_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace kfac {

constexpr int kGtMaxProbs = 96;  // problems per launch (kernel parameter space)
constexpr int kSplitMax = 384;   // matrices per split launch (64 B each in parameter space)

// One problem C = alpha * A B^T.  a / b: bf16 slices [3][rows][ld].
struct GtOperand {
  const uint16_t* a;
  const uint16_t* b;
  long long M, N, K, lda, ldb;
  void* out;                   // fp32 [M][ldc], or bf16 slices [3][M][ldc] when out_split
  long long ldc, out_slice_stride;
  int out_split;
  float alpha;
  int flag_idx;                // index into the launch's flags (see launch_gemm_tc), or -1
  float* w;                    // fp32 [M][ldw] weights: w -= lr * C (fp32 output only), or null
  long long ldw;
  float lr;
};

struct GtProb {
  void* out;
  float* w;
  long long ldc, out_slice_stride, tile_begin, ldw;
  int M, N, K, tiles_n, out_split, flag_idx;
  float alpha, lr;
};

// fp32 src [rows][ld_src] -> bf16 dst slices: slice k at dst + k * slice_stride.
// When `probe` is set, the same pass adds src * z into probe[rows][kProbeN]
// (z: the Rademacher probes of probe8 in gemm_tc.cu, bit offset probe_shift:
// 0 for the right probes, 8 for the left ones).
struct SplitItem {
  const float* src;
  uint16_t* dst;
  long long rows, cols, ld_src, ld_dst, slice_stride, item_begin;
  float* probe;
  int probe_shift;
  int flag_idx;
};
struct SplitParams {
  SplitItem items[kSplitMax];
  const int* flags;
  long long total_items;
  int n;
  int planes;
};

// Probes of the preconditioning check: eight Rademacher vectors on each side.
// Entry k of the probes at index i (8 g + e):
//   z_k(i) = H8[k][e ^ t(g)] * (sign from bit e + shift of probe_hash(g)),
// H8 the 8 x 8 Sylvester-Hadamard matrix, shift 0 for the right probes and 8
// for the left ones, and t(g) a 3-bit class offset per group of eight (bits
// 16-18 of the hash for the right probes, 19-21 for the left).  Each z_k is a
// Rademacher vector; the mean of the 8 x 8 bilinear forms keeps the pairs
// of equal class, and the class offset stops a residual concentrated on
// every eighth index from falling into one class.  Since
// H8[k][e ^ t] = H8[k][e] H8[k][t], a group's eight projections are its
// 8-point Walsh-Hadamard transform with probe k's result times H8[k][t].
constexpr int kProbeN = 8;

// sign (+1 / -1) of probe k at index i: bit k + shift of a 32-bit integer
// hash of i (the "lowbias32" mixing function: xor-shift / multiply rounds)
__host__ __device__ __forceinline__ uint32_t probe_hash(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352dU;
  x ^= x >> 15;
  x *= 0x846ca68bU;
  x ^= x >> 16;
  return x;
}

// t(g) of the probes with bit offset `shift` (0 or 8), from probe_hash(g)
__host__ __device__ __forceinline__ int probe_class_offset(uint32_t hash, int shift) {
  return (int)((hash >> (16 + 3 * (shift / 8))) & 7u);
}
// H8[k][b] = (-1)^popcount(k & b)
__host__ __device__ __forceinline__ float hadamard8(int k, int b) {
  const int kb = k & b & 7;
  return ((kb ^ (kb >> 1) ^ (kb >> 2)) & 1) ? -1.f : 1.f;
}

// `planes` bf16 slices per fp32 value (2 or 3).  Items whose flag_idx >= 0 run
// only when flags[flag_idx] != 0 (flags may be null: every item runs).
// compact: small blocks, one per chunk of rows, that fit beside a GEMM block
// on one SM (for a split that overlaps the GEMMs of other matrices).
int launch_split(const SplitItem* items, int n, int planes, const int* flags, cudaStream_t stream,
                 bool compact = false);
// ns = operand slices read per product: 3 (six MMAs per multiply-add, all 24
// bits) or 2 (three MMAs: hi*hi + hi*mid + mid*hi, 16 bits).  Split outputs
// are written with ns slices.  Problems whose flag_idx >= 0 run only when
// flags[flag_idx] != 0.  pairs: CTA pairs sharing B through TMA multicast.
// A problem with w applies w -= lr * C in the epilogue (fp32 output only).
int launch_gemm_tc(const GtOperand* ops, int n, int ns, const int* flags, cudaStream_t stream,
                   bool pairs = true);  // sorts by K
int launch_gemm_tc_sorted(const GtOperand* ops, int n, int ns, const int* flags, cudaStream_t stream,
                          bool pairs = true);

}  // namespace kfac
