// Batched inverse of damped SPD factors through a Cholesky decomposition
// (SPD-KFAC §IV: the inverse is computed through a Cholesky decomposition;
// §III-B: the damped inverses (A + lambda I)^-1, (G + lambda I)^-1).
//
// Algorithm, per matrix (size d, T = ceil(d/128) block rows, n_pad = 128 T,
// padded with the identity so every tile operation is full size: the padded
// matrix is diag(D, I) and its inverse diag(D^-1, I)).  Right-looking blocked
// sweep over the 128-wide block columns k = 0..T-1, Cholesky fused with the
// blocked forward substitution L W = I (W = L^-1):
//   diag(k)   L_kk = chol(A_kk), Winv_k = L_kk^-1 in shared memory (= W_kk)
//   panel(k)  L_rk = A_rk Winv_k^T   for r > k;   W_kc = Winv_k C_kc  for c < k
//   update(k) A_rc -= L_rk L_ck^T    for r >= c > k  (Schur complement)
//             C_rc  = [c<k] C_rc - L_rk W_kc  for r > k >= c  (block row r of L W = I)
// then X = W^T W, formed for the upper tiles and mirrored: X is exactly symmetric.
//
// Two passes run these steps:
//   * fp32 on tcgen05 tensor cores (inverse_tc.cu): every tile product with
//     three-slice bf16 operands, drained per k-step into fp32;
//   * fp64 on CUDA cores (this file), for the matrices that neither the
//     fp32 pass nor the Newton step after it settles (refine = AUTO) or for
//     all of them (refine = ALWAYS).
//
// refine = AUTO: the fp32 pass measures its own residual.  With kProbes
// Rademacher vectors v (+-1 entries), w = D v and then y = X w are formed in
// double-float arithmetic (fp32 pairs, ~48 bits), so ||y - v||^2 averaged over
// the probes is an unbiased estimate of ||X D - I||_F^2 (inverse_tc.cu: w
// from the partial sums tc_load_kernel leaves per tile, added up by
// tc_route_kernel; y in tc_probe_kernel).  Matrices whose estimated
// residual ||X D - I||_F / sqrt(d) exceeds 2.5e-4 (four times below the 1e-3
// target), whose ||D||_1 / min L_jj^2 exceeds 3e5 (a guard on the relative
// error), or whose fp32 factorisation failed, are flagged.  A flagged matrix
// whose factorisation succeeded first gets up to two Newton steps on the
// tensor cores (refine.cu); what is still flagged after them is redone in
// fp64, and the fp64 kernels of the other matrices exit at once.
#include <math.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "inverse_common.cuh"
#include "launch.h"
#include "simt.cuh"

namespace kfac {

// ------------------------------------------------------------------ setup
__global__ void inv_setup_kernel(const __grid_constant__ InvSetup prm, InvCtx c) {
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nth = (long long)gridDim.x * blockDim.x;
  const bool all64 = prm.mode == KFAC_REFINE_ALWAYS;
  for (long long e = tid; e < prm.n; e += nth) {
    const_cast<InvMat*>(c.mats)[e] = prm.mats[e];
    InvState s;
    s.info32 = 0;
    s.info64 = 0;
    s.failed = 0;
    s.use64 = all64 ? 1 : 0;
    s.min_piv = 3.0e38f;
    s.kappa = 0.f;
    s.xnorm2 = 0.f;
    s.est_res = 0.f;
    s.slices = 3;
    s.glo = 0xffffffffu;
    s.ghi = 0u;
    s.gbad = 0;
    s.gdone = 0;
    s.refine = 0;
    s.refined = 0;
    c.st[e] = s;
    c.flagged[e] = (int)e;
  }
  if (tid == 0) *c.nflagged = all64 ? prm.n : 0;
  for (long long e = tid; e < prm.rowsum_total; e += nth) c.rowsum[e] = 0.f;
  for (long long e = tid; e < prm.probe_total; e += nth) c.probe[e] = make_float2(0.f, 0.f);
}

// The fp64 pass kernels run a persistent 1-D grid over the matrices in the
// flagged list (tiles of one matrix spread over the grid), so that when the
// fp32 pass routes nothing to fp64 every launch ends at once.

// ------------------------------------------------------------------ fp64 pass: load D into the L-buffer
template <typename T>
__global__ void __launch_bounds__(256) inv_load_kernel(InvCtx c) {
  __shared__ float sub[32][33];
  const int nf = *c.nflagged;
  const int lx = threadIdx.x % 32, ly = threadIdx.x / 32;  // 32 x 8
  for (int f = 0; f < nf; ++f) {
    const int mi = c.flagged[f];
    const InvMat m = c.mats[mi];
    const long long np = (long long)m.T * 128;
    T* L = lbuf<T>(c, m);
    for (long long q = blockIdx.x; q < tri(m.T); q += gridDim.x) {
      const int R = tri_root(q), C = (int)(q - tri(R));  // lower tile (R, C), R >= C
      for (int sb = 0; sb < 16; ++sb) {
        const int bm = (sb / 4) * 32, bn = (sb % 4) * 32;  // sub-block rows (mm) / cols (nn) of the L tile
        // read D[C*128 + bn + y][R*128 + bm + x] (coalesced along x), store sub[y][x]
        for (int y = ly; y < 32; y += 8) {
          const long long gc = (long long)C * 128 + bn + y;   // D row   = L column
          const long long gr = (long long)R * 128 + bm + lx;  // D column = L row
          float v = 0.f;
          if (gc < m.d && gr < m.d && gr >= gc) v = m.D[gc * m.ld_in + gr];
          sub[y][lx] = v;
        }
        __syncthreads();
        for (int y = ly; y < 32; y += 8) {
          const long long gr = (long long)R * 128 + bm + y;
          const long long gc = (long long)C * 128 + bn + lx;
          T out;
          if (gr >= m.d || gc >= m.d)
            out = (gr == gc) ? T(1) : T(0);
          else if (gr < gc)
            out = T(0);
          else
            out = (T)sub[lx][y] + ((gr == gc) ? (T)c.gamma_extra : T(0));
          L[gr * np + gc] = out;
        }
        __syncthreads();
      }
    }
  }
}

// ------------------------------------------------------------------ fp64 pass: diagonal block
template <typename T>
__global__ void __launch_bounds__(256, 1) inv_diag_kernel(InvCtx c, int k) {
  extern __shared__ __align__(16) uint8_t diag_smem[];
  T* a = reinterpret_cast<T*>(diag_smem);
  const int nf = *c.nflagged;
  const int t = threadIdx.x;
  for (int f = blockIdx.x; f < nf; f += gridDim.x) {
    const int mi = c.flagged[f];
    const InvMat m = c.mats[mi];
    if (k >= m.T || c.st[mi].failed) continue;
    const long long np = (long long)m.T * 128;
    const T* src = lbuf<T>(c, m) + (long long)k * 128 * np + (long long)k * 128;
    for (int e = t; e < 128 * 128; e += blockDim.x) {
      const int r = e / 128, col = e % 128;
      a[r * kDiagPitch + col] = (col <= r) ? src[(long long)r * np + col] : T(0);
    }
    __syncthreads();
    T min_piv;
    const int fail = block_chol_inv<T>(a, m.d - k * 128, min_piv);
    if (fail >= 0) {
      if (t == 0) {
        c.st[mi].failed = 1;
        c.st[mi].info64 = k * 128 + fail + 1;
      }
    } else {
      T* dst = wbuf<T>(c, m) + (long long)k * 128 * np + (long long)k * 128;
      for (int e = t; e < 128 * 128; e += blockDim.x) {
        const int r = e / 128, col = e % 128;
        dst[(long long)r * np + col] = (col <= r) ? a[r * kDiagPitch + col] : T(0);
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ tile epilogues
template <typename T>
__device__ __forceinline__ void tile_store(T* dst, long long ld, const T (&acc)[4][8], int mode) {
  // mode 0: dst = acc, 1: dst -= acc, 2: dst = -acc (simt_tile_df's thread layout)
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    T* row = dst + (long long)(ty * 4 + a) * ld + tx * 8;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (mode == 0)
        row[b] = acc[a][b];
      else if (mode == 1)
        row[b] -= acc[a][b];
      else
        row[b] = -acc[a][b];
    }
  }
}

// ------------------------------------------------------------------ fp64 pass: panel
template <typename T>
__global__ void __launch_bounds__(kDfThreads) inv_panel_kernel(InvCtx c, int k) {
  __shared__ __align__(16) T smem[simt_smem_bytes<T>() / sizeof(T)];
  const int nf = *c.nflagged;
  for (int f = 0; f < nf; ++f) {
    const int mi = c.flagged[f];
    const InvMat m = c.mats[mi];
    if (k >= m.T || c.st[mi].failed) continue;
    const int nr = m.T - 1 - k;
    const long long np = (long long)m.T * 128;
    T* L = lbuf<T>(c, m);
    T* W = wbuf<T>(c, m);
    const T* winv = W + (long long)k * 128 * np + (long long)k * 128;
    for (int q = blockIdx.x; q < nr + k; q += gridDim.x) {
      T acc[4][8];
      if (q < nr) {
        const int r = k + 1 + q;
        T* Lrk = L + (long long)r * 128 * np + (long long)k * 128;
        Opnd<T> A{Lrk, np, 1, 128};
        Opnd<T> B{winv, np, 1, 128};
        simt_tile_df(acc, A, B, 128, smem);
        tile_store(Lrk, np, acc, 0);
      } else {
        const int cc = q - nr;
        T* Ckc = W + (long long)k * 128 * np + (long long)cc * 128;
        Opnd<T> A{winv, np, 1, 128};
        Opnd<T> B{Ckc, 1, np, 128};
        simt_tile_df(acc, A, B, 128, smem);
        tile_store(Ckc, np, acc, 0);
      }
    }
  }
}

// ------------------------------------------------------------------ fp64 pass: trailing update
// part 0: every job; part 1: the jobs step k + 1 reads (block row k + 1 of W
// and of L, block column k + 1 of L: m.T jobs); part 2: the others.
template <typename T>
__global__ void __launch_bounds__(kDfThreads) inv_update_kernel(InvCtx c, int k, int part) {
  __shared__ __align__(16) T smem[simt_smem_bytes<T>() / sizeof(T)];
  const int nf = *c.nflagged;
  for (int f = 0; f < nf; ++f) {
    const int mi = c.flagged[f];
    const InvMat m = c.mats[mi];
    if (k + 1 >= m.T || c.st[mi].failed) continue;
    const long long np = (long long)m.T * 128;
    T* L = lbuf<T>(c, m);
    T* W = wbuf<T>(c, m);
    const long long njobs = part == 1 ? m.T : tri(m.T) - tri(k + 1);
    for (long long q = blockIdx.x; q < njobs; q += gridDim.x) {
      int r, cc;
      if (part == 1) {
        r = q <= k + 1 ? k + 1 : (int)q;
        cc = q <= k + 1 ? (int)q : k + 1;
      } else {
        const long long qq = q + tri(k + 1);
        r = tri_root(qq);
        cc = (int)(qq - tri(r));
        if (part == 2 && (r == k + 1 || cc == k + 1)) continue;
      }
      const T* Lrk = L + (long long)r * 128 * np + (long long)k * 128;
      T acc[4][8];
      Opnd<T> A{Lrk, np, 1, 128};
      if (cc > k) {
        Opnd<T> B{L + (long long)cc * 128 * np + (long long)k * 128, np, 1, 128};
        simt_tile_df(acc, A, B, 128, smem);
        tile_store(L + (long long)r * 128 * np + (long long)cc * 128, np, acc, 1);
      } else {
        Opnd<T> B{W + (long long)k * 128 * np + (long long)cc * 128, 1, np, 128};
        simt_tile_df(acc, A, B, 128, smem);
        tile_store(W + (long long)r * 128 * np + (long long)cc * 128, np, acc, cc == k ? 2 : 1);
      }
    }
  }
}

// ------------------------------------------------------------------ fp64 pass: X = W^T W
template <typename T>
__global__ void __launch_bounds__(kDfThreads) inv_lauum_kernel(InvCtx c) {
  __shared__ __align__(16) T smem[simt_smem_bytes<T>() / sizeof(T)];
  const int nf = *c.nflagged;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  for (int f = 0; f < nf; ++f) {
    const int mi = c.flagged[f];
    const InvMat m = c.mats[mi];
    if (c.st[mi].failed) continue;
    const long long np = (long long)m.T * 128;
    const T* W = wbuf<T>(c, m);
    // Jobs come longest first (K = np - 128 j falls with j); CTA b takes job b
    // of even rounds and job G - 1 - b of odd ones, so that long and short
    // jobs pair up on each CTA.
    const long long G = gridDim.x, njobs = tri(m.T);
    for (long long round = 0; round * G < njobs; ++round) {
      const long long q = round * G + ((round & 1) ? G - 1 - blockIdx.x : blockIdx.x);
      if (q >= njobs) continue;
      const int j = tri_root(q);
      const int i = (int)(q - tri(j));  // i <= j
      T acc[4][8];
      Opnd<T> A{W + (long long)j * 128 * np + (long long)i * 128, 1, np, 128};
      Opnd<T> B{W + (long long)j * 128 * np + (long long)j * 128, 1, np, 128};
      simt_tile_df(acc, A, B, (int)(np - (long long)j * 128), smem);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int mm = ty * 4 + a;
        const long long row = (long long)i * 128 + mm;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int nn = tx * 8 + b;
          const long long col = (long long)j * 128 + nn;
          if (row >= m.d || col >= m.d || (i == j && mm > nn)) continue;
          const float v = (float)acc[a][b];
          m.X[row * m.ld_out + col] = v;
          m.X[col * m.ld_out + row] = v;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ AUTO decision
__global__ void __launch_bounds__(128) inv_flag_kernel(InvCtx c) {
  const int mi = blockIdx.x;
  const InvMat m = c.mats[mi];
  __shared__ float red[128];
  __shared__ double red2[128];
  const long long np = (long long)m.T * 128;
  const float2* y = c.probe + m.off_probe + (long long)kProbes * np;
  float mx = 0.f;
  double e2 = 0.0;  // sum over probes of ||X (D v) - v||^2
  for (int r = threadIdx.x; r < m.d; r += 128) {
    mx = fmaxf(mx, c.rowsum[m.off_rowsum + r]);
#pragma unroll
    for (int p = 0; p < kProbes; ++p) {
      const float2 yv = y[p * np + r];
      const double e = df_value(yv.x, yv.y) - probe_sign(r, p);
      e2 += e * e;
    }
  }
  red[threadIdx.x] = mx;
  red2[threadIdx.x] = e2;
  __syncthreads();
  for (int s = 64; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + s]);
      red2[threadIdx.x] += red2[threadIdx.x + s];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    InvState& s = c.st[mi];
    const float norm1 = red[0];
    const float kappa = s.min_piv > 0.f ? norm1 / s.min_piv : 3.0e38f;
    // E||(XD - I) v||^2 = ||XD - I||_F^2 for Rademacher v
    const double est = sqrt(red2[0] / kProbes / (double)m.d);
    s.kappa = kappa;
    s.est_res = (float)est;
    s.use64 = (s.failed || !(kappa <= kAutoKappa) || !(est <= kAutoResidual)) ? 1 : 0;
    if (s.use64) {
      s.failed = 0;  // the fp64 pass starts afresh
      c.flagged[atomicAdd(c.nflagged, 1)] = mi;
    }
  }
}

__global__ void inv_finish_kernel(InvCtx c, int n, int* info, int* route) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const InvState s = c.st[i];
  info[i] = s.use64 ? s.info64 : s.info32;
  if (route) route[i] = s.use64 ? 1 : s.refined ? 3 : (s.slices == 2 ? 2 : 0);
}

// ------------------------------------------------------------------ host side
struct InvLayout {
  size_t mats_off, st_off, flag_off, rowsum_off, probe_off, gpart_off, wpart_off, region_off, total;
  TcLayout tc;
};

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

static InvLayout inv_layout(int n, const kfac_inverse_args* args, int refine, long long* rowsum_total,
                            long long* probe_total, InvMat* mats /* may be null */) {
  InvLayout L;
  L.mats_off = 0;
  L.st_off = align256(sizeof(InvMat) * (size_t)n);
  L.flag_off = L.st_off + align256(sizeof(InvState) * (size_t)n);
  L.rowsum_off = L.flag_off + align256(sizeof(int) * (size_t)(n + 1));
  long long rs = 0, gp = 0;
  int Ts[kInvMaxGroup];
  for (int i = 0; i < n; ++i) {
    Ts[i] = (int)((args[i].d + 127) / 128);
    if (mats) {
      mats[i].off_rowsum = rs;
      mats[i].off_probe = 2 * kProbes * rs;
      mats[i].row_off = rs;
      mats[i].off_gpart = gp;
    }
    rs += (long long)Ts[i] * 128;
    gp += (long long)Ts[i] * Ts[i] * 128;
  }
  *rowsum_total = rs;
  *probe_total = 2 * kProbes * rs;
  L.probe_off = L.rowsum_off + align256(sizeof(float) * (size_t)rs);
  L.gpart_off = L.probe_off + align256(sizeof(float2) * (size_t)(2 * kProbes * rs));
  const size_t gpart_bytes = refine == KFAC_REFINE_AUTO ? align256(sizeof(float) * (size_t)gp) : 0;
  L.wpart_off = L.gpart_off + gpart_bytes;
  const size_t wpart_bytes = refine == KFAC_REFINE_AUTO ? align256(sizeof(float2) * (size_t)gp * kProbes) : 0;
  L.region_off = L.wpart_off + wpart_bytes;
  // the fp32 tensor-core pass and the fp64 pass run one after the other and
  // share the work region
  size_t fp64 = 0;
  if (refine != KFAC_REFINE_NONE)
    for (int i = 0; i < n; ++i) {
      const size_t np = (size_t)Ts[i] * 128;
      if (mats) mats[i].off_buf = (long long)fp64;
      fp64 += align256(2 * np * np * sizeof(double));
    }
  L.tc = tc_layout(n, Ts);
  const size_t fp32 = refine != KFAC_REFINE_ALWAYS ? L.tc.bytes : 0;
  // AUTO: the tensor-core Newton step (refine.cu) runs between the fp32 pass
  // and the fp64 pass, on the same region, with its own per-matrix buffers
  size_t ref = 0;
  if (refine == KFAC_REFINE_AUTO)
    for (int i = 0; i < n; ++i) {
      if (mats) mats[i].off_ref = (long long)ref;
      ref += align256(refine_bytes((long long)Ts[i] * 128));
    }
  size_t region = fp64 > fp32 ? fp64 : fp32;
  if (ref > region) region = ref;
  L.total = L.region_off + region;
  return L;
}

size_t inverse_workspace(int n, const kfac_inverse_args* args, int refine) {
  // groups of kInvMaxGroup run one after the other and reuse the workspace
  size_t best = 0;
  for (int base = 0; base < n; base += kInvMaxGroup) {
    const int cnt = n - base < kInvMaxGroup ? n - base : kInvMaxGroup;
    long long rs, pt;
    const InvLayout L = inv_layout(cnt, args + base, refine, &rs, &pt, nullptr);
    if (L.total > best) best = L.total;
  }
  return best;
}

static int run_fp64_pass(const InvCtx& ctx, int Tmax, cudaStream_t stream, bool lookahead = true) {
  const int dsm = diag_smem_bytes<double>();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (!ensure_smem_attr(dev, (const void*)inv_diag_kernel<double>, dsm)) return KFAC_ERR_CUDA;
  inv_load_kernel<double><<<sms, 256, 0, stream>>>(ctx);
  count_launch();
  // Look-ahead: step k's chain (diagonal block, panel, and the part of the
  // trailing update that step k + 1 reads) runs on the high-priority stream;
  // the rest of the update runs on the caller's stream, one job per CTA so
  // that SMs come free for the chain, beside the next steps' chain.
  cudaStream_t chain = nullptr;
  cudaEvent_t ev[4];
  const bool split = lookahead && Tmax > 2 && fp64_chain_stream(dev, stream, &chain, ev);
  if (split) {
    if (cudaEventRecord(ev[0], stream) != cudaSuccess || cudaStreamWaitEvent(chain, ev[0], 0) != cudaSuccess)
      return KFAC_ERR_CUDA;
  }
  cudaStream_t cs = split ? chain : stream;
  for (int k = 0; k < Tmax; ++k) {
    inv_diag_kernel<double><<<sms, 256, dsm, cs>>>(ctx, k);
    count_launch();
    if (Tmax > 1) {
      inv_panel_kernel<double><<<sms, kDfThreads, 0, cs>>>(ctx, k);
      count_launch();
      if (k + 1 < Tmax) {
        if (!split) {
          inv_update_kernel<double><<<sms, kDfThreads, 0, stream>>>(ctx, k, 0);
          count_launch();
          continue;
        }
        // the far update of step k - 1 has written block row and column k + 1
        if (k > 0 && cudaStreamWaitEvent(chain, ev[2], 0) != cudaSuccess) return KFAC_ERR_CUDA;
        inv_update_kernel<double><<<Tmax, kDfThreads, 0, chain>>>(ctx, k, 1);
        count_launch();
        if (cudaEventRecord(ev[1], chain) != cudaSuccess || cudaStreamWaitEvent(stream, ev[1], 0) != cudaSuccess)
          return KFAC_ERR_CUDA;
        const long long far = tri(Tmax) - tri(k + 1);
        inv_update_kernel<double><<<(unsigned)(far > 0 ? far : 1), kDfThreads, 0, stream>>>(ctx, k, 2);
        count_launch();
        if (cudaEventRecord(ev[2], stream) != cudaSuccess) return KFAC_ERR_CUDA;
      }
    }
  }
  if (split) {
    if (cudaEventRecord(ev[3], chain) != cudaSuccess || cudaStreamWaitEvent(stream, ev[3], 0) != cudaSuccess)
      return KFAC_ERR_CUDA;
  }
  inv_lauum_kernel<double><<<sms, kDfThreads, 0, stream>>>(ctx);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA;
}

// ------------------------------------------------------------------ AUTO's later passes, skipped when idle
// The Newton step and the fp64 pass are persistent grids over the flagged
// list, about 150 launches for the largest factors, each ending at once when
// nothing is flagged.  A call of AUTO instead launches them as one cached
// CUDA graph: a one-thread kernel sets a conditional handle from the flagged
// count, the Newton step runs inside an IF node, a second such kernel reads
// the count the Newton step left, and the fp64 pass (without its look-ahead
// stream) runs inside a second IF node.  With nothing flagged the call costs
// two tiny launches.  The graph is kept per (device, batch, work buffers), so
// a caller that repeats a call on the same buffers builds it once.
__global__ void inv_gate_kernel(cudaGraphConditionalHandle h, const int* nflagged) {
  if (threadIdx.x == 0 && blockIdx.x == 0) cudaGraphSetConditional(h, *nflagged > 0 ? 1u : 0u);
}

namespace {
constexpr int kGateKey = 16;
constexpr size_t kMaxGateGraphs = 64;  // built graphs kept for the process; more calls run the plain launches
struct GateGraph {
  unsigned long long key[kGateKey];
  cudaGraphExec_t exec;
};
std::mutex g_gate_mu;
std::vector<GateGraph> g_gate;
cudaStream_t g_capture[64];  // a private stream per device to record the bodies on

void gate_key(const InvCtx& c, int n, int Tmax, int dev, unsigned long long (&k)[kGateKey]) {
  unsigned int gbits = 0;
  memcpy(&gbits, &c.gamma_extra, sizeof(gbits));
  const unsigned long long v[kGateKey] = {
      (unsigned long long)dev, (unsigned long long)n, (unsigned long long)Tmax, (unsigned long long)gbits,
      (unsigned long long)(uintptr_t)c.ws, (unsigned long long)(uintptr_t)c.mats,
      (unsigned long long)(uintptr_t)c.st, (unsigned long long)(uintptr_t)c.rowsum,
      (unsigned long long)(uintptr_t)c.gpart, (unsigned long long)(uintptr_t)c.wpart,
      (unsigned long long)(uintptr_t)c.probe, (unsigned long long)(uintptr_t)c.flagged,
      (unsigned long long)(uintptr_t)c.nflagged, (unsigned long long)(uintptr_t)c.region,
      (unsigned long long)c.want_rowsum, 0ull};
  memcpy(k, v, sizeof(k));
}

bool add_gate(cudaGraph_t g, const cudaGraphNode_t* dep, int ndep, cudaGraphConditionalHandle h, const int* nflagged,
              cudaGraphNode_t* node) {
  void* argv[2] = {&h, const_cast<int**>(&nflagged)};
  cudaKernelNodeParams kp = {};
  kp.func = (void*)inv_gate_kernel;
  kp.gridDim = dim3(1);
  kp.blockDim = dim3(32);
  kp.kernelParams = argv;
  return cudaGraphAddKernelNode(node, g, dep, (size_t)ndep, &kp) == cudaSuccess;
}

bool add_if(cudaGraph_t g, cudaGraphNode_t dep, cudaGraphConditionalHandle h, cudaGraphNode_t* node,
            cudaGraph_t* body) {
  cudaGraphNodeParams np = {};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = h;
  np.conditional.type = cudaGraphCondTypeIf;
  np.conditional.size = 1;
  if (cudaGraphAddNode(node, g, &dep, nullptr, 1, &np) != cudaSuccess) return false;
  *body = np.conditional.phGraph_out[0];
  return true;
}
}  // namespace

// The executable graph for (ctx, n, Tmax) on the current device, built on
// first use; nullptr when it cannot be built (the caller then launches the
// passes directly).
static cudaGraphExec_t gated_passes(const InvCtx& ctx, int n, int Tmax) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned long long key[kGateKey];
  gate_key(ctx, n, Tmax, dev, key);
  std::lock_guard<std::mutex> lk(g_gate_mu);
  for (const GateGraph& e : g_gate)
    if (memcmp(e.key, key, sizeof(key)) == 0) return e.exec;
  if (g_gate.size() >= kMaxGateGraphs) return nullptr;
  if (!g_capture[dev] && cudaStreamCreateWithFlags(&g_capture[dev], cudaStreamNonBlocking) != cudaSuccess) {
    g_capture[dev] = nullptr;
    return nullptr;
  }
  const cudaStream_t cs = g_capture[dev];
  cudaGraph_t g = nullptr;
  cudaGraphExec_t exec = nullptr;
  bool ok = cudaGraphCreate(&g, 0) == cudaSuccess;
  cudaGraphConditionalHandle h1 = 0, h2 = 0;
  ok = ok && cudaGraphConditionalHandleCreate(&h1, g, 0, cudaGraphCondAssignDefault) == cudaSuccess &&
       cudaGraphConditionalHandleCreate(&h2, g, 0, cudaGraphCondAssignDefault) == cudaSuccess;
  cudaGraphNode_t g1 = nullptr, c1 = nullptr, g2 = nullptr, c2 = nullptr;
  cudaGraph_t b1 = nullptr, b2 = nullptr;
  ok = ok && add_gate(g, nullptr, 0, h1, ctx.nflagged, &g1) && add_if(g, g1, h1, &c1, &b1);
  if (ok) {  // body 1: the Newton step
    ok = cudaStreamBeginCaptureToGraph(cs, b1, nullptr, nullptr, 0, cudaStreamCaptureModeRelaxed) == cudaSuccess;
    if (ok) {
      const int rc = run_refine_pass(ctx, n, Tmax, cs);
      cudaGraph_t got = nullptr;
      ok = cudaStreamEndCapture(cs, &got) == cudaSuccess && rc == KFAC_OK;
    }
  }
  ok = ok && add_gate(g, &c1, 1, h2, ctx.nflagged, &g2) && add_if(g, g2, h2, &c2, &b2);
  if (ok) {  // body 2: the fp64 pass
    InvCtx c64 = ctx;
    c64.pass64 = 1;
    c64.want_rowsum = 0;
    ok = cudaStreamBeginCaptureToGraph(cs, b2, nullptr, nullptr, 0, cudaStreamCaptureModeRelaxed) == cudaSuccess;
    if (ok) {
      const int rc = run_fp64_pass(c64, Tmax, cs, false);
      cudaGraph_t got = nullptr;
      ok = cudaStreamEndCapture(cs, &got) == cudaSuccess && rc == KFAC_OK;
    }
  }
  ok = ok && cudaGraphInstantiate(&exec, g, 0) == cudaSuccess;
  if (g) cudaGraphDestroy(g);
  if (!ok) {
    if (exec) cudaGraphExecDestroy(exec);
    cudaGetLastError();  // a failed build leaves no error behind: the plain launches follow
    return nullptr;
  }
  GateGraph e;
  memcpy(e.key, key, sizeof(key));
  e.exec = exec;
  g_gate.push_back(e);
  return exec;
}

int launch_damped_inverse(int n, const kfac_inverse_args* args, float gamma_extra, int refine, int* info, int* route,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (workspace_bytes < inverse_workspace(n, args, refine) || workspace == nullptr) return KFAC_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  InvSetup prm;  // 18 KB of kernel parameters, staged on the host stack
  int Ts[kInvMaxGroup];
  for (int base = 0; base < n; base += kInvMaxGroup) {
    const int cnt = n - base < kInvMaxGroup ? n - base : kInvMaxGroup;
    memset(&prm, 0, sizeof(prm));
    long long rs_total = 0, probe_total = 0;
    const InvLayout L = inv_layout(cnt, args + base, refine, &rs_total, &probe_total, prm.mats);
    int Tmax = 0;
    for (int i = 0; i < cnt; ++i) {
      const kfac_inverse_args& a = args[base + i];
      InvMat& m = prm.mats[i];
      m.D = a.damped;
      m.X = a.inv;
      m.ld_in = a.ld_in;
      m.ld_out = a.ld_out;
      m.d = (int)a.d;
      m.T = (int)((a.d + 127) / 128);
      Ts[i] = m.T;
      if (m.T > Tmax) Tmax = m.T;
    }
    prm.n = cnt;
    prm.mode = refine;
    prm.rowsum_total = rs_total;
    prm.probe_total = refine == KFAC_REFINE_AUTO ? probe_total : 0;
    InvCtx ctx;
    ctx.ws = ws;
    ctx.mats = reinterpret_cast<const InvMat*>(ws + L.mats_off);
    ctx.st = reinterpret_cast<InvState*>(ws + L.st_off);
    ctx.flagged = reinterpret_cast<int*>(ws + L.flag_off);
    ctx.nflagged = ctx.flagged + cnt;
    ctx.rowsum = reinterpret_cast<float*>(ws + L.rowsum_off);
    ctx.probe = reinterpret_cast<float2*>(ws + L.probe_off);
    ctx.gpart = refine == KFAC_REFINE_AUTO ? reinterpret_cast<float*>(ws + L.gpart_off) : nullptr;
    ctx.wpart = refine == KFAC_REFINE_AUTO ? reinterpret_cast<float2*>(ws + L.wpart_off) : nullptr;
    ctx.region = ws + L.region_off;
    ctx.gamma_extra = gamma_extra;
    ctx.want_rowsum = refine == KFAC_REFINE_AUTO;
    {
      const long long work = probe_total > cnt ? probe_total : cnt;
      long long blocks = (work + 255) / 256;
      if (blocks > 1024) blocks = 1024;
      inv_setup_kernel<<<(unsigned)blocks, 256, 0, stream>>>(prm, ctx);
      count_launch();
    }
    int rc;
    if (refine != KFAC_REFINE_ALWAYS) {
      ctx.pass64 = 0;
      rc = run_tc_pass(ctx, prm.mats, cnt, Tmax, Ts, L.tc, stream);
      if (rc != KFAC_OK) return rc;
    }
    if (refine == KFAC_REFINE_AUTO) {
      ProfMark pm;
      prof_begin(stream, pm);
      inv_flag_kernel<<<cnt, 128, 0, stream>>>(ctx);
      prof_end(KFAC_K_INV_AUX, stream, pm, 0.0);
      count_launch();
      // the flagged matrices first get one Newton step on tensor cores; those
      // it settles leave the fp64 pass's list.  Both passes run from the
      // gated graph unless the launch profile records (its events would not
      // be captured) or the caller's stream is itself being captured.
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      const bool gated = !prof_recording() && cudaStreamIsCapturing(stream, &cap) == cudaSuccess &&
                         cap == cudaStreamCaptureStatusNone;
      cudaGraphExec_t exec = gated ? gated_passes(ctx, cnt, Tmax) : nullptr;
      if (exec) {
        if (cudaGraphLaunch(exec, stream) != cudaSuccess) return KFAC_ERR_CUDA;
        count_launch();
        count_launch();
      } else {
        rc = run_refine_pass(ctx, cnt, Tmax, stream);
        if (rc != KFAC_OK) return rc;
        ctx.pass64 = 1;
        ctx.want_rowsum = 0;
        rc = run_fp64_pass(ctx, Tmax, stream);
        if (rc != KFAC_OK) return rc;
      }
    } else if (refine == KFAC_REFINE_ALWAYS) {
      ctx.pass64 = 1;
      ctx.want_rowsum = 0;
      rc = run_fp64_pass(ctx, Tmax, stream);
      if (rc != KFAC_OK) return rc;
    }
    inv_finish_kernel<<<(cnt + 255) / 256, 256, 0, stream>>>(ctx, cnt, info + base, route ? route + base : nullptr);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

}  // namespace kfac
