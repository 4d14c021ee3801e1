// Shared pieces of the batched damped inverse (inverse.cu: fp64 CUDA-core
// pass and host orchestration; inverse_tc.cu: fp32 tensor-core pass).
#pragma once
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "probes.cuh"

namespace kfac {

constexpr int kInvMaxGroup = 256;
constexpr float kAutoKappa = 3e5f;
constexpr double kAutoResidual = 2.5e-4;
constexpr int kProbes = 4;
// AUTO: a matrix whose Gershgorin discs bound its condition number by this
// ratio runs the fp32 pass with 16-bit operands (two bf16 slices, three MMAs
// per multiply-add).  Emulated on the host, two slices left a residual
// ||X D - I||_F / sqrt(d) of about 3e-6 times the condition number
// (2e-7 at 1, 1e-5 at 4, 1.2e-3 at 4e3); at 16 that is under 5e-5, five times
// below the residual bar that sends a matrix to the fp64 pass.
constexpr float kSlices16Kappa = 16.f;

struct InvMat {
  const float* D;
  float* X;
  long long ld_in, ld_out;
  long long off_buf;     // byte offset of the fp64 L/W buffers in the workspace
  long long off_rowsum;  // float index of this matrix's row sums
  long long off_probe;   // double index of this matrix's probe vectors w, y
  long long row_off;     // first row of this matrix in the stacked fp32 work buffers
  long long off_gpart;   // float index of this matrix's partial off-diagonal row sums (T x T x 128)
  long long off_ref;     // byte offset of the refinement buffers in the work region (AUTO)
  int d, T;
};

struct InvState {
  int info32, info64, failed, use64;
  float min_piv, kappa;
  float xnorm2, est_res;  // ||X||_F^2 and the estimated residual of the fp32 pass
  int slices;             // bf16 slices per operand in the fp32 pass: 3 (24-bit) or 2 (16-bit)
  // AUTO's Gershgorin bound, gathered over the row blocks (tc_route_kernel):
  // ordered bits of the smallest disc end and of the largest, a non-finite
  // flag and the number of row blocks done
  unsigned glo, ghi;
  int gbad, gdone;
  int refine;   // AUTO sent it away from the fp32 pass and its fp32 factorisation succeeded
  int refined;  // its inverse came from the tensor-core Newton step (refine.cu)
};

static_assert(kProbes == 4, "the fp32 pass's probes are the four rows of H4 (probes.cuh)");
// v_p(i) of the fp32 pass's residual check (probes.cuh)
__device__ __forceinline__ double probe_sign(long long i, int p) { return (double)probe4(i, p); }

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
  float* gpart;     // AUTO: per matrix, partial sums of |D_rc| (c != r) over each 128-column block
  float2* wpart;    // AUTO: per matrix, the same blocks' double-float partial sums of (D v_p)_r
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

// ljj = sqrt(piv) and inv = 1 / ljj of a Cholesky pivot; fp32 through the
// reciprocal square root (a few ulp, far inside the fp32 pass's error budget)
__device__ __forceinline__ void pivot_scale(float piv, float& ljj, float& inv) {
  inv = rsqrtf(piv);
  ljj = piv * inv;
}
__device__ __forceinline__ void pivot_scale(double piv, double& ljj, double& inv) {
  ljj = sqrt(piv);
  inv = 1.0 / ljj;
}

constexpr int kDiagPitch = 129;
template <typename T>
constexpr int diag_smem_bytes() {
  return 128 * kDiagPitch * (int)sizeof(T);
}

// Per-thread share of one warp's product tile, accumulated in registers:
// rows (lane / 16) * RH + i (i < RH) and columns 2 * (lane % 16) + e (e < 2) of
// C += A B, with A(r, q) = A[r * lda + q] and B(q, c) = B[q * bq + c * bc],
// q in [0, K).  Both operands are in shared memory; with the 129-element
// pitch of the diagonal block the reads are free of bank conflicts.
template <typename T, int RH>
__device__ __forceinline__ void warp_tile_mm(T (&acc)[RH][2], const T* A, int lda, const T* B, int bq, int bc,
                                             int K) {
  const int lane = threadIdx.x % 32;
  const T* a0 = A + (lane / 16) * RH * lda;
  const T* b0 = B + 2 * (lane % 16) * bc;
#pragma unroll 4
  for (int q = 0; q < K; ++q) {  // K is a multiple of 32
    const T b_0 = b0[q * bq], b_1 = b0[q * bq + bc];
#pragma unroll
    for (int i = 0; i < RH; ++i) {
      const T av = a0[i * lda + q];
      acc[i][0] += av * b_0;
      acc[i][1] += av * b_1;
    }
  }
}

template <typename T, int RH>
__device__ __forceinline__ void zero_tile(T (&acc)[RH][2]) {
#pragma unroll
  for (int i = 0; i < RH; ++i) acc[i][0] = acc[i][1] = T(0);
}

// Cholesky factor and inverse of one 128 x 128 diagonal block held in shared
// memory (`a`, pitch kDiagPitch, lower triangle valid, upper triangle zero),
// called by all threads of a 256-thread block.  On return `a` holds
// Winv = L^-1 (lower, zeros above) and the result is -1, or the column of the
// first non-positive (or NaN) pivot, in which case `a` is partly overwritten.
// `min_piv` receives the smallest pivot among the first `valid` columns.
//
// Blocked by 32 columns.  For each panel one warp factors the 32 x 32
// diagonal block in registers (lane i holds row i; columns travel by warp
// shuffles) and inverts it (lane c forms column c of the inverse); then all
// warps solve the rows below against that inverse and subtract the panel's
// contribution from the trailing lower triangle.  The inverse of the whole
// block is then assembled in place from the four diagonal inverses, block
// column by block column from the right:  W_ij = -(sum_{j<k<=i} W_ik L_kj) W_jj.
template <typename T>
__device__ int block_chol_inv(T* a, int valid, T& min_piv) {
  constexpr int P = kDiagPitch;
  __shared__ T wd[4][32][33];  // inverses of the four 32 x 32 diagonal factors
  __shared__ T dinv[128];      // 1 / L_jj
  __shared__ T tmp[96][33];    // partial products of the assembly step
  __shared__ T colbuf[32];     // pivot, then column j of L, during the 32 x 32 factorisation
  __shared__ int s_fail;
  __shared__ T s_minpiv;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, nwarps = blockDim.x / 32;
  if (tid == 0) {
    s_fail = -1;
    s_minpiv = T(3.0e38);
  }
  __syncthreads();
  for (int p = 0; p < 4; ++p) {
    const int p0 = 32 * p;
    if (warp == 0) {
      T x[32];  // row p0 + lane of the diagonal block
#pragma unroll
      for (int c = 0; c < 32; ++c) x[c] = (c <= lane) ? a[(p0 + lane) * P + p0 + c] : T(0);
      int fail = -1;  // uniform over the warp: every pivot is a broadcast
      T mp = T(3.0e38);
      // Step j: the pivot and then the scaled column j travel through shared
      // memory (one store per lane, broadcast loads that issue back to back),
      // not through a chain of 32 shuffles.
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (lane == j) colbuf[j] = x[j];
        __syncwarp();
        const T piv = colbuf[j];
        __syncwarp();
        if (fail < 0 && !(piv > T(0))) fail = j;
        if (fail < 0) {
          if (p0 + j < valid && piv < mp) mp = piv;
          T ljj, inv;
          pivot_scale(piv, ljj, inv);
          if (lane > j) x[j] *= inv;
          if (lane == j) {
            x[j] = ljj;
            dinv[p0 + j] = inv;
          }
          colbuf[lane] = x[j];  // column j of L (zero above the diagonal)
          __syncwarp();
#pragma unroll
          for (int c = j + 1; c < 32; ++c) {
            const T lcj = colbuf[c];
            if (lane >= c) x[c] -= x[j] * lcj;
          }
          __syncwarp();
        }
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) a[(p0 + lane) * P + p0 + c] = (c <= lane) ? x[c] : T(0);
      __syncwarp();
      if (lane == 0) {
        if (fail >= 0) s_fail = p0 + fail;
        if (mp < s_minpiv) s_minpiv = mp;
      }
      if (fail < 0) {
        // column `lane` of the inverse, forward substitution against e_lane
        T w[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) w[r] = (r == lane) ? T(1) : T(0);
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          w[q] *= dinv[p0 + q];
#pragma unroll
          for (int r = q + 1; r < 32; ++r) w[r] -= a[(p0 + r) * P + p0 + q] * w[q];
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) wd[p][r][lane] = w[r];
      }
    }
    __syncthreads();
    if (s_fail >= 0) return s_fail;
    const int nbt = 3 - p;  // 32-row blocks below the panel
    if (nbt == 0) break;
    // rows below the panel: L(r, panel) = A(r, panel) W_pp^T, 16-row items,
    // each warp reads and then overwrites only its own rows
    for (int it = warp; it < 2 * nbt; it += nwarps) {
      const int r0 = p0 + 32 + 16 * it;
      T acc[8][2];
      zero_tile(acc);
      warp_tile_mm<T, 8>(acc, a + r0 * P + p0, P, &wd[p][0][0], 1, 33, 32);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        T* row = a + (r0 + (lane / 16) * 8 + i) * P + p0 + 2 * (lane % 16);
        row[0] = acc[i][0];
        row[1] = acc[i][1];
      }
    }
    __syncthreads();
    // trailing lower triangle: A(r, c) -= L(r, panel) L(c, panel)^T, 32 x 32 tiles
    for (int it = warp; it < nbt * (nbt + 1) / 2; it += nwarps) {
      int bi = 0;
      while ((bi + 1) * (bi + 2) / 2 <= it) ++bi;
      const int bj = it - bi * (bi + 1) / 2;
      const int r0 = p0 + 32 + 32 * bi, c0 = p0 + 32 + 32 * bj;
      T acc[16][2];
      zero_tile(acc);
      warp_tile_mm<T, 16>(acc, a + r0 * P + p0, P, a + c0 * P + p0, 1, P, 32);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = (lane / 16) * 16 + i, c = 2 * (lane % 16);
        T* row = a + (r0 + r) * P + c0 + c;
        if (bi != bj || c <= r) row[0] -= acc[i][0];
        if (bi != bj || c + 1 <= r) row[1] -= acc[i][1];
      }
    }
    __syncthreads();
  }
  min_piv = s_minpiv;
  // the diagonal factors are no longer read: put their inverses in their place
  for (int e = tid; e < 4 * 32 * 32; e += blockDim.x) {
    const int p = e / 1024, r = (e / 32) % 32, c = e % 32;
    a[(32 * p + r) * P + 32 * p + c] = (c <= r) ? wd[p][r][c] : T(0);
  }
  __syncthreads();
  for (int j = 2; j >= 0; --j) {
    const int rb = 32 * (j + 1);   // first row below the diagonal block j
    const int items = 2 * (3 - j);  // 16-row items
    for (int it = warp; it < items; it += nwarps) {
      const int r0 = rb + 16 * it, i = r0 / 32;
      T acc[8][2];
      zero_tile(acc);
      // sum over k in (j, i] of W_ik L_kj; W_ik sits in a already (k > j)
      warp_tile_mm<T, 8>(acc, a + r0 * P + rb, P, a + rb * P + 32 * j, P, 1, 32 * (i - j));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        T* row = &tmp[r0 - rb + (lane / 16) * 8 + q][2 * (lane % 16)];
        row[0] = acc[q][0];
        row[1] = acc[q][1];
      }
    }
    __syncthreads();  // every L_kj of this block column has been read
    for (int it = warp; it < items; it += nwarps) {
      const int r0 = rb + 16 * it;
      T acc[8][2];
      zero_tile(acc);
      warp_tile_mm<T, 8>(acc, &tmp[r0 - rb][0], 33, &wd[j][0][0], 33, 1, 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        T* row = a + (r0 + (lane / 16) * 8 + q) * P + 32 * j + 2 * (lane % 16);
        row[0] = -acc[q][0];
        row[1] = -acc[q][1];
      }
    }
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
// refine.cu: bytes of one matrix's refinement buffers (np = 128 T), and the pass
size_t refine_bytes(long long np);
int run_refine_pass(const InvCtx& ctx, int n, int Tmax, cudaStream_t stream);
// inverse_tc.cu: the fp32 pass on tensor cores (with AUTO's residual probes)
int run_tc_pass(const InvCtx& ctx, const InvMat* host_mats, int n, int Tmax, const int* Ts, const TcLayout& L,
                cudaStream_t stream);

}  // namespace kfac
