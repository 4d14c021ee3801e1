// Host/device interface of the split-bf16 tcgen05 GEMM (gemm_tc.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace kfac {

constexpr int kGtMaxProbs = 96;  // problems per launch (kernel parameter space)
constexpr int kSplitMax = 384;   // matrices per split launch (64 B each in parameter space)

// One problem C = alpha * A B^T.  a / b: bf16 slices [NS][rows][ld].
struct GtOperand {
  const uint16_t* a;
  const uint16_t* b;
  long long M, N, K, lda, ldb;
  void* out;                   // fp32 [M][ldc], or bf16 slices [NS][M][ldc] when out_split
  long long ldc, out_slice_stride;
  int out_split;
  float alpha;
};

struct GtProb {
  void* out;
  long long ldc, out_slice_stride, tile_begin;
  int M, N, K, tiles_n, out_split;
  float alpha;
};

// fp32 src [rows][ld_src] -> bf16 dst slices: slice k at dst + k * slice_stride.
struct SplitItem {
  const float* src;
  uint16_t* dst;
  long long rows, cols, ld_src, ld_dst, slice_stride, item_begin;
};
struct SplitParams {
  SplitItem items[kSplitMax];
  long long total_items;
  int n;
};

// Three bf16 slices per fp32 value (see gemm_tc.cu).
int launch_split(const SplitItem* items, int n, cudaStream_t stream);
int launch_gemm_tc(const GtOperand* ops, int n, cudaStream_t stream);         // sorts by K
int launch_gemm_tc_sorted(const GtOperand* ops, int n, cudaStream_t stream);  // as given

}  // namespace kfac
