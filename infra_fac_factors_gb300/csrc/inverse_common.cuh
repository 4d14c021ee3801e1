// Shared pieces of the batched damped inverse (inverse.cu: fp64 CUDA-core
// pass and host orchestration; inverse_tc.cu: fp32 tensor-core pass).
#pragma once
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace kfac {

constexpr int kInvMaxGroup = 256;
constexpr float kAutoKappa = 3e5f;
constexpr double kAutoResidual = 2.5e-4;
constexpr int kProbes = 4;

struct InvMat {
  const float* D;
  float* X;
  long long ld_in, ld_out;
  long long off_buf;     // byte offset of the fp64 L/W buffers in the workspace
  long long off_rowsum;  // float index of this matrix's row sums
  long long off_probe;   // double index of this matrix's probe vectors w, y
  long long row_off;     // first row of this matrix in the stacked fp32 work buffers
  int d, T;
};

struct InvState {
  int info32, info64, failed, use64;
  float min_piv, kappa;
  float xnorm2, est_res;  // ||X||_F^2 and the estimated residual of the fp32 pass
};

// Rademacher probe entry v_p(i) in {-1, +1} (splitmix64 finaliser of (i, p)).
__device__ __forceinline__ double probe_sign(long long i, int p) {
  unsigned long long z = (unsigned long long)(i * kProbes + p) + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (z & 1ull) ? 1.0 : -1.0;
}

struct InvSetup {
  InvMat mats[kInvMaxGroup];
  int n, mode;
  long long rowsum_total, probe_total;
};

struct InvCtx {
  uint8_t* ws;
  const InvMat* mats;
  InvState* st;
  float* rowsum;
  float2* probe;    // per matrix: w[kProbes][n_pad] then y[kProbes][n_pad], double-float (hi, lo)
  int* flagged;     // indices of the matrices the fp64 pass inverts
  int* nflagged;    // their count
  uint8_t* region;  // work buffers of the passes (fp32 tensor-core or fp64)
  float gamma_extra;
  int pass64;       // 0: fp32 pass, 1: fp64 pass
  int want_rowsum;  // fp32 pass of AUTO: record norms and probes
};

// ------------------------------------------------------------------ double-float sums
// (hi, lo) += x with the exact rounding error of hi + x carried in lo
// (Knuth's TwoSum); products of fp32 values by (whi + wlo) keep their exact
// error through an FMA.  About 48 significant bits with fp32 instructions
// only (fp64 throughput on this part is a small fraction of fp32).
__device__ __forceinline__ void df_add(float& hi, float& lo, float x) {
  const float s = hi + x;
  const float bb = s - hi;
  const float e = (hi - (s - bb)) + (x - bb);
  hi = s;
  lo += e;
}
__device__ __forceinline__ void df_add_prod(float& hi, float& lo, float x, float whi, float wlo) {
  const float p = x * whi;
  const float pe = fmaf(x, whi, -p);  // exact error of the product
  df_add(hi, lo, p);
  lo += fmaf(x, wlo, pe);
}
__device__ __forceinline__ double df_value(float hi, float lo) { return (double)hi + (double)lo; }
__device__ __forceinline__ float2 df_pack(float hi, float lo) {
  const float s = hi + lo;  // renormalise so that |lo| <= ulp(hi) / 2
  return make_float2(s, lo - (s - hi));
}

// fp64 pass: compact per-matrix buffers in the work region
template <typename T>
__device__ __forceinline__ T* lbuf(const InvCtx& c, const InvMat& m) {
  return reinterpret_cast<T*>(c.region + m.off_buf);
}
template <typename T>
__device__ __forceinline__ T* wbuf(const InvCtx& c, const InvMat& m) {
  return lbuf<T>(c, m) + (long long)m.T * 128 * m.T * 128;
}

// Whether matrix `mi` takes part in the current pass (and has not failed in it).
__device__ __forceinline__ bool inv_active(const InvCtx& c, int mi, bool need_ok) {
  const InvState& s = c.st[mi];
  if (c.pass64 ? !s.use64 : s.use64) return false;
  if (need_ok && s.failed) return false;
  return true;
}

__host__ __device__ inline long long tri(long long t) { return t * (t + 1) / 2; }
// largest r with r(r+1)/2 <= q
__device__ __forceinline__ int tri_root(long long q) {
  int r = (int)((sqrt(8.0 * (double)q + 1.0) - 1.0) * 0.5);
  while (tri(r + 1) <= q) ++r;
  while (tri(r) > q) --r;
  return r;
}

template <typename T>
__device__ __forceinline__ T dev_sqrt(T v);
template <>
__device__ __forceinline__ float dev_sqrt<float>(float v) { return __fsqrt_rn(v); }
template <>
__device__ __forceinline__ double dev_sqrt<double>(double v) { return sqrt(v); }
template <typename T>
__device__ __forceinline__ T dev_rcp(T v);
template <>
__device__ __forceinline__ float dev_rcp<float>(float v) { return __frcp_rn(v); }
template <>
__device__ __forceinline__ double dev_rcp<double>(double v) { return 1.0 / v; }

constexpr int kDiagPitch = 129;
template <typename T>
constexpr int diag_smem_bytes() {
  return 128 * kDiagPitch * (int)sizeof(T);
}

// Cholesky factor and inverse of one 128 x 128 diagonal block held in shared
// memory (`a`, pitch kDiagPitch, lower triangle valid, upper triangle zero),
// 128 threads.  On return `a` holds Winv = L^-1 (lower, zeros above) and the
// result is -1, or the block column of the first non-positive pivot.
// `min_piv` receives the smallest pivot among the first `valid` columns.
template <typename T>
__device__ int block_chol_inv(T* a, int valid, T& min_piv) {
  const int t = threadIdx.x;
  // Cholesky, right-looking; column j is scaled by 1/sqrt(pivot) one iteration
  // later, when no thread reads it any more, so each column costs one barrier.
  int fail = -1;
  min_piv = T(3.0e38);
  T prev_rs = T(0);
  for (int j = 0; j < 128; ++j) {
    const T piv = a[j * kDiagPitch + j];
    if (!(piv > T(0))) {  // also catches NaN
      fail = j;
      break;
    }
    if (j < valid && piv < min_piv) min_piv = piv;
    if (j > 0) {
      const int r = j + t;  // rows j .. 127 of column j-1
      if (r < 128) a[r * kDiagPitch + (j - 1)] *= prev_rs;
      if (t == 0) a[(j - 1) * kDiagPitch + (j - 1)] = dev_sqrt<T>(a[(j - 1) * kDiagPitch + (j - 1)]);
    }
    const T ip = dev_rcp<T>(piv);
    prev_rs = dev_rcp<T>(dev_sqrt<T>(piv));
    const int col = t;
    if (col > j) {
      const T f = a[col * kDiagPitch + j] * ip;
      for (int r = col; r < 128; ++r) a[r * kDiagPitch + col] -= a[r * kDiagPitch + j] * f;
    }
    __syncthreads();
  }
  if (fail >= 0) return fail;
  // last column: only its diagonal is left
  if (t == 0) a[127 * kDiagPitch + 127] = dev_sqrt<T>(a[127 * kDiagPitch + 127]);
  __syncthreads();
  // In-place inverse of the lower-triangular block, column by column from the
  // right: W_jj = 1/L_jj, W_rj = -(sum_{j<s<=r} W_rs L_sj) / L_jj.
  for (int j = 127; j >= 0; --j) {
    const T ljj = a[j * kDiagPitch + j];
    T s = T(0);
    const int r = t;
    if (r > j)
      for (int q = j + 1; q <= r; ++q) s += a[r * kDiagPitch + q] * a[q * kDiagPitch + j];
    __syncthreads();
    if (r > j) a[r * kDiagPitch + j] = -s / ljj;
    if (r == j) a[j * kDiagPitch + j] = dev_rcp<T>(ljj);
    __syncthreads();
  }
  return -1;
}

// the fp32 tensor-core pass (inverse_tc.cu)
struct TcLayout {
  long long R_tot, LD;         // stacked rows of all matrices, common leading dimension
  size_t acc, u, p, lp, winv;  // byte offsets inside the work region
  size_t bytes;
};
TcLayout tc_layout(int n, const int* T);
int run_tc_pass(const InvCtx& ctx, const InvMat* host_mats, int n, int Tmax, const int* Ts, const TcLayout& L,
                cudaStream_t stream);

}  // namespace kfac
