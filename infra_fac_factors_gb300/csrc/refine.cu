// Refinement, on tensor cores, of the inverses that AUTO does not accept from
// the fp32 pass (SPD-KFAC §IV: the inverse of each damped factor; its accuracy
// is this library's own concern).  One Newton step
//
//     X1 = X0 + X0 (I - D X0),      D symmetric, X0 the fp32 pass's inverse,
//
// halves the number of correct digits lost to D's conditioning, provided the
// residual I - D X0 is formed well beyond fp32 accuracy: its entries are
// differences of products that are up to kappa(D) times larger than they are.
// The products are therefore taken exactly, in the error-free split of Ozaki,
// Ogita, Oishi and Rump (fixed-point slices that share one exponent per row,
// so that every bf16 x bf16 tensor-core product of two slices is an integer
// multiple of one power of two and a short sum of them is exact in fp32):
//
//   split   x_rc = 2^e_r (sum_{s=1..6} q_s(r, c) 2^(-8 s)),  q_s integers, |q_s| <= 256,
//           e_r the exponent of the largest |x_r.| (each slice a bf16 value
//           q_s 2^(-8 s), exact);
//   product (A B^T)_ij = 2^(e_i + f_j) sum_{s,t} sum_k a_s(i, k) b_t(j, k),
//           the pairs grouped by level L = s + t: every product of one level
//           is an integer multiple of 2^(-8 L), so the sum of the level's
//           pairs over one 32-wide k-block (at most four pairs below level 5,
//           |q q'| <= 2^16) stays below 2^24 and is exact in a tensor-core
//           fp32 accumulator.  Levels 2, 3 and 4 get an accumulator each;
//           levels 5 to 7 share one (their rounding error is below 2^-48 of the
//           products).  Each k-block's accumulators are drained into
//           double-float sums (fp32 pairs) by the epilogue warps.
//
// Host emulation on the ResNet-50 C = 512 conv factor (d = 4609,
// kappa = 7.4e5): six slices with the pairs up to level 7 (21 MMAs per 16-wide
// k-step) form the residual to 1.4e-9 (RMS) and the step lands on the fp32
// storage floor of the inverse, ||X1 D - I||_F / sqrt(d) = 2.3e-4 (1.0e-3
// before), relative error 8.5e-8; pairs up to level 6 leave 4.5e-7 in the
// residual and 2.0e-3 after the step.  The correction X0 (I - D X0) needs
// only three slices and the pairs up to level 4 (six MMAs).
//
// Steps, all on the device and only for the matrices AUTO flagged whose fp32
// factorisation succeeded (the others exit at once):
//   rf_split_kernel   D (upper triangle, + gamma_extra) and X0 into slices
//   rf_gemm_kernel    S = I - X0 D = (I - D X0)^T   (levels up to 7)
//   rf_split_kernel   S into slices
//   rf_gemm_kernel    T = X0 S^T = X0 (I - D X0)    (levels up to 4)
//   rf_sym_kernel     X1 = X0 + (T + T^T) / 2, written over X0 (exactly symmetric)
// then sixteen independent probes of its own (rf_w16_kernel, once;
// rf_y16_kernel) estimate the residual of X1, and a matrix whose estimate
// meets the refined bar keeps X1; the others take a second step from X1 (the
// D slices are taken again: their buffer held S), and those it does not
// settle go on to the fp64 pass.
#include "common.cuh"
#include "inverse_common.cuh"
#include "launch.h"

namespace kfac {

constexpr int kRfSlices = 6;
constexpr int kRfBK = 32;                              // k of one stage
constexpr int kRfDrain = 4;                            // stages per accumulator drain (128 k)
constexpr int kRfM = 128, kRfN = 128;                  // output tile
constexpr int kRfA = kRfM * kRfBK * 2;                 // one A slice of a stage: 8 KB (a whole slice tile)
constexpr int kRfB = kRfN * kRfBK * 2;                 // one B slice: 8 KB
constexpr int kRfStage = kRfSlices * (kRfA + kRfB);    // 96 KB
constexpr int kRfStages = 2;
constexpr int kRfEpiWarps = 16;                        // epilogue warps: four per TMEM lane quarter
constexpr int kRfThreads = 64 + 32 * kRfEpiWarps;      // producer warp, MMA warp, epilogue warps
constexpr int kRfSmem = kRfStages * kRfStage + 1024 + 256;
constexpr int kRfAcc = 4;                              // accumulators: levels 2, 3, 4, 5-7
// sets of the four accumulators in the 512 TMEM columns: with 128-wide tiles
// one set, drained in place (the MMAs of the next 128 k wait for the drain)
constexpr int kRfBufs = 512 / (kRfAcc * kRfN);
constexpr int kRfHalves = kRfM / kRfN;                 // B tiles per slice tile
static_assert(kRfBufs >= 1 && kRfHalves >= 1, "tile shape");

// Slices are stored tile by tile, each tile the byte image of the K-major,
// 64-byte-swizzled shared-memory layout the tensor cores read: tile (rb, kb)
// of a slice is 128 rows x 32 k of bf16, 8 KB contiguous, row r at 64 r
// bytes, its 16-byte chunk c (k = 8c .. 8c + 7) at chunk position
// c ^ ((r / 2) % 4); one bulk copy moves a stage's tile of a slice (the first
// or second 64 rows of a tile are its first or second 4 KB).
__host__ __device__ inline long long rf_tile_off(long long T, int s, long long rb, long long kb) {
  return (((long long)s * T + rb) * (4 * T) + kb) * (kRfM * kRfBK);
}

// Probes of the decision after a step: kRfProbes independent Rademacher
// vectors (probe16 in probes.cuh).  A Newton step leaves I - X1 D =
// (I - X0 D)^2 up to rounding, a residual close to rank one: the mean of
// sixteen squared projections then gives an estimate below half the true
// residual with a probability near 1e-3 (chi-square with sixteen degrees of
// freedom below four), against near 0.09 with four.
constexpr int kRfProbes = kProbes16;

// Per-matrix refinement buffers, at m.off_ref in the work region (np = 128 T):
//   xs  bf16 [6][T][4T] tiles   slices of X0
//   bs  bf16 [6][T][4T] tiles   slices of D, then of S
//   st  fp32 [np][np]           S, then T
//   ex, eb  int [np]            row exponents of xs and bs
//   w16, y16  double-float [kRfProbes][np]   D v and X1 D v for the decision's probes
struct RfBufs {
  uint16_t* xs;
  uint16_t* bs;
  float* st;
  int* ex;
  int* eb;
  float2* w16;
  float2* y16;
};
__host__ __device__ inline size_t rf_bytes(long long np) {
  return (size_t)np * np * (2 * kRfSlices * 2 + 4) + (size_t)np * 8 + (size_t)np * kRfProbes * 2 * sizeof(float2);
}
__device__ __forceinline__ RfBufs rf_bufs(const InvCtx& c, const InvMat& m) {
  const long long np = (long long)m.T * 128;
  uint8_t* base = c.region + m.off_ref;
  RfBufs b;
  b.xs = reinterpret_cast<uint16_t*>(base);
  b.bs = b.xs + (size_t)kRfSlices * np * np;
  b.st = reinterpret_cast<float*>(b.bs + (size_t)kRfSlices * np * np);
  b.ex = reinterpret_cast<int*>(b.st + (size_t)np * np);
  b.eb = b.ex + np;
  b.w16 = reinterpret_cast<float2*>(b.eb + np);  // np is a multiple of 128: 512-byte aligned
  b.y16 = b.w16 + (size_t)kRfProbes * np;
  return b;
}

// the f-th matrix of the flagged list, when it is a refinement candidate
__device__ __forceinline__ int rf_matrix(const InvCtx& c, int f) {
  if (f >= *c.nflagged) return -1;
  const int mi = c.flagged[f];
  return c.st[mi].refine ? mi : -1;
}

// ------------------------------------------------------------------ candidates
// Matrices AUTO sends away from the fp32 pass whose fp32 factorisation succeeded.
__global__ void rf_mark_kernel(InvCtx c, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  InvState& s = c.st[i];
  s.refine = (s.use64 && s.info32 == 0) ? 1 : 0;
  s.refined = 0;
}

// ------------------------------------------------------------------ split
// One CTA per 128-row block: the rows' largest |x| over all column tiles
// (through shared memory: a tile of D left of the diagonal is read from its
// mirror in the upper triangle and transposed), then the six slices of each
// tile, written tile by tile in the tensor cores' layout.
//   op 0: D (upper triangle read; the lower part by symmetry; gamma_extra on the diagonal)
//   op 1: X0 (the fp32 pass's full symmetric inverse in m.X)
//   op 2: S (fp32, in the refinement buffers)
constexpr int kRfPitch = 129;
__device__ void rf_load_tile(const InvCtx& c, const InvMat& m, const RfBufs& rb, int op, int rbk, int cb, float* t) {
  const long long np = (long long)m.T * 128;
  const bool mirror = op == 0 && cb < rbk;  // a tile of D left of the diagonal: its mirror, transposed
  const long long r0 = (long long)(mirror ? cb : rbk) * 128, c0 = (long long)(mirror ? rbk : cb) * 128;
  const float* src = op == 0 ? m.D : op == 1 ? m.X : rb.st;
  const long long ld = op == 0 ? m.ld_in : op == 1 ? m.ld_out : np;
  __syncthreads();
  // 16 float4 per thread, all loads issued before the stores (rows are
  // 16-byte multiples long, so a float4 starting inside a row stays in it)
  float4 v[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int e = threadIdx.x + 256 * k, a = e / 32, b4 = (e % 32) * 4;
    const long long gr = r0 + a, gc = c0 + b4;
    v[k] = (gr < m.d && gc < m.d) ? *reinterpret_cast<const float4*>(src + gr * ld + gc) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int e = threadIdx.x + 256 * k, a = e / 32, b4 = (e % 32) * 4;
    const long long gc = c0 + b4;
    const float x[4] = {v[k].x, gc + 1 < m.d ? v[k].y : 0.f, gc + 2 < m.d ? v[k].z : 0.f, gc + 3 < m.d ? v[k].w : 0.f};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (mirror)
        t[(b4 + u) * kRfPitch + a] = x[u];
      else
        t[a * kRfPitch + b4 + u] = x[u];
    }
  }
  __syncthreads();
  if (op == 0 && cb == rbk) {
    // the diagonal tile of D: its lower part by symmetry (whatever the caller
    // keeps below the diagonal is not read), gamma_extra on the diagonal
    for (int e = threadIdx.x; e < 128 * 128; e += 256) {
      const int a = e / 128, b = e % 128;
      if (b < a) t[a * kRfPitch + b] = t[b * kRfPitch + a];
    }
    __syncthreads();
    if (threadIdx.x < 128 && r0 + threadIdx.x < m.d) t[threadIdx.x * kRfPitch + threadIdx.x] += c.gamma_extra;
    __syncthreads();
  }
}

__device__ void rf_split_block(const InvCtx& c, int mi, int rbk, int op, float* t, int* rowexp) {
  const InvMat m = c.mats[mi];
  const RfBufs rb = rf_bufs(c, m);
  uint16_t* dst = op == 1 ? rb.xs : rb.bs;
  int* ex = op == 1 ? rb.ex : rb.eb;
  // pass 1: row maxima (two threads per row, 64 columns of each tile each)
  const int row = threadIdx.x % 128, half = threadIdx.x / 128;
  float mx = 0.f;
  for (int cb = 0; cb < m.T; ++cb) {
    rf_load_tile(c, m, rb, op, rbk, cb, t);
    for (int b = 64 * half; b < 64 * half + 64; ++b) mx = fmaxf(mx, fabsf(t[row * kRfPitch + b]));
  }
  __syncthreads();
  if (half == 1) rowexp[row] = __float_as_int(mx);
  __syncthreads();
  if (half == 0) {
    mx = fmaxf(mx, __int_as_float(rowexp[row]));
    int e = 0;
    if (mx > 0.f && isfinite(mx)) frexpf(mx, &e);  // mx = f 2^e, f in [0.5, 1): |x / 2^e| < 1
    rowexp[row] = e;
    ex[(long long)rbk * 128 + row] = e;
  }
  // pass 2: slices; each thread takes 16-byte chunks (8 values of one row),
  // consecutive threads along a row's four chunks, then the next rows: a warp
  // writes 512 contiguous bytes of a tile per slice
  for (int cb = 0; cb < m.T; ++cb) {
    rf_load_tile(c, m, rb, op, rbk, cb, t);  // (its first barrier also publishes rowexp)
    for (int qq = threadIdx.x; qq < 2048; qq += 256) {
      const int kbl = qq / 512, rr = (qq / 4) % 128, ck = qq % 4;
      const int k0 = kbl * 32 + ck * 8;
      const int e = rowexp[rr];
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = ldexpf(t[rr * kRfPitch + k0 + u], -e);
      const long long within = (long long)rr * 32 + ((ck ^ ((rr >> 1) & 3)) * 8);
#pragma unroll
      for (int sl = 0; sl < kRfSlices; ++sl) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 8; u += 2) {
          const float q0 = rintf(x[u] * 256.f), q1 = rintf(x[u + 1] * 256.f);  // |q| <= 256: exact in bf16
          x[u] = x[u] * 256.f - q0;                                           // exact
          x[u + 1] = x[u + 1] * 256.f - q1;
          const uint32_t b0 = __float_as_uint(ldexpf(q0, -8 * (sl + 1))) >> 16;
          const uint32_t b1 = __float_as_uint(ldexpf(q1, -8 * (sl + 1))) >> 16;
          w[u / 2] = b0 | (b1 << 16);
        }
        uint16_t* tile = dst + rf_tile_off(m.T, sl, rbk, (long long)cb * 4 + kbl);
        *reinterpret_cast<uint4*>(tile + within) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

__global__ void __launch_bounds__(256) rf_split_kernel(InvCtx c, int op_base) {
  extern __shared__ __align__(16) uint8_t rf_split_smem[];
  float* t = reinterpret_cast<float*>(rf_split_smem);  // 128 x kRfPitch
  int* rowexp = reinterpret_cast<int*>(t + 128 * kRfPitch);
  const int nf = *c.nflagged;
  for (int f = 0; f < nf; ++f) {
    const int mi = rf_matrix(c, f);
    if (mi < 0) continue;
    for (int rbk = blockIdx.x; rbk < c.mats[mi].T; rbk += gridDim.x)
      rf_split_block(c, mi, rbk, op_base + (int)blockIdx.y, t, rowexp);
  }
}
constexpr int kRfSplitSmem = (128 * kRfPitch + 128) * 4;

// ------------------------------------------------------------------ exact product
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
               "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// K-major shared-memory descriptor, 64-byte swizzle (rows of 64 B, 8-row
// groups 512 B apart, layout type 4)
__device__ __forceinline__ uint64_t rf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;
  return d;
}

// Job u of a matrix with T row blocks -> (A row block ib, B column tile jn):
// bands of kRfBand row blocks, column-major inside a band, so that the grid's
// concurrent jobs share few operand panels (about kRfBand A panels and
// gridDim / kRfBand B panels, which L2 holds).
constexpr int kRfBand = 8;
__device__ __forceinline__ void rf_job(long long u, long long T, long long& ib, long long& jn) {
  const long long tn = kRfHalves * T, per_band = (long long)kRfBand * tn;
  const long long band = u / per_band, w = u % per_band;
  const long long rows = (band + 1) * kRfBand <= T ? kRfBand : T - band * kRfBand;
  ib = band * kRfBand + w % rows;
  jn = w / rows;
}

// x 2^k for |k| <= 252: two exact power-of-two factors built from their
// IEEE-754 exponent fields (each in [-126, 127])
__device__ __forceinline__ float scale_pow2(float x, int k) {
  const int k1 = k / 2, k2 = k - k1;
  return x * __int_as_float((127 + k1) << 23) * __int_as_float((127 + k2) << 23);
}

// accumulator of the slice pair (s, t) (0-based): levels 2, 3, 4, then 5-7 together
__host__ __device__ constexpr int rf_slot(int s, int t) { return s + t < 3 ? s + t : 3; }

// The MMAs of one stage (two 16-wide k-steps): every slice pair up to level
// LMAX, each into its level's accumulator.  All indices are static; the first
// pair of each accumulator, (0, slot), overwrites it at the start of a drain
// period (`first`).
template <int LMAX>
__device__ __forceinline__ void rf_issue(uint32_t tmem_acc, uint32_t a0, uint32_t b0, uint32_t idesc, bool first) {
  const uint64_t da0 = rf_desc(a0), db0 = rf_desc(b0);  // the address field is linear in the address
#pragma unroll
  for (int kk = 0; kk < kRfBK / 16; ++kk) {
#pragma unroll
    for (int s = 0; s < kRfSlices; ++s) {
#pragma unroll
      for (int t = 0; t < kRfSlices; ++t) {
        if (s + t + 2 > LMAX) continue;
        const int a = rf_slot(s, t);
        const uint64_t da = da0 + (uint64_t)((s * kRfA + kk * 32) >> 4);
        const uint64_t db = db0 + (uint64_t)((t * kRfB + kk * 32) >> 4);
        const bool opens = kk == 0 && s == 0 && t == a;
        tc_mma_bf16(tmem_acc + a * kRfN, da, db, idesc, (opens && first) ? 0u : 1u);
      }
    }
  }
}

// C = A B^T over the flagged candidates, A = xs (rows of X0), B = bs (rows of
// D, or of S); tiles of 128 x 128, jobs dealt round-robin over a persistent
// grid.  LMAX: highest level taken (7 for the residual, 4 for the correction).
// mode 0: st = I - 2^(e_i + f_j) C  (the residual S);  mode 1: st = 2^(e_i + f_j) C  (T).
// The accumulators are drained every kRfDrain stages (128 k: every level up to
// 4 stays below 2^24 of its unit, |q_1| <= 256 and |q_s| <= 128 after it).
template <int LMAX>
__global__ void __launch_bounds__(kRfThreads, 1) rf_gemm_kernel(InvCtx c, int n, int mode, int* status) {
  constexpr int lmax = LMAX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRfStages * kRfStage);
  uint64_t* empty = full + kRfStages;
  uint64_t* acc_full = empty + kRfStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int nf = *c.nflagged;
  bool any = false;
  for (int f = 0; f < nf && !any; ++f) any = rf_matrix(c, f) >= 0;
  if (!any) return;  // uniform over the grid: nothing to refine
  (void)n;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRfStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kRfEpiWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- producer: one bulk copy per slice tile of a stage (the
    // slices the level cap reaches: s <= lmax - 2)
    if (lane == 0) {
      const int nsl = lmax - 1 < kRfSlices ? lmax - 1 : kRfSlices;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int f = 0; f < nf && ok; ++f) {
        const int mi = rf_matrix(c, f);
        if (mi < 0) continue;
        const InvMat m = c.mats[mi];
        const RfBufs rb = rf_bufs(c, m);
        const long long T = m.T, tn = kRfHalves * T, jobs = T * tn;
        for (long long u = blockIdx.x; u < jobs && ok; u += gridDim.x) {
          long long ib, jn;  // A row block; B rows: tile jn / kRfHalves, part jn % kRfHalves
          rf_job(u, T, ib, jn);
          for (long long kb = 0; kb < 4 * T; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
            uint8_t* s0 = smem + stage * kRfStage;
            mbar_arrive_expect_tx(&full[stage], nsl * (kRfA + kRfB));
#pragma unroll
            for (int sl = 0; sl < kRfSlices; ++sl) {
              if (sl >= nsl) break;
              bulk_load(smem_u32(s0 + sl * kRfA), rb.xs + rf_tile_off(T, sl, ib, kb), kRfA, &full[stage]);
              bulk_load(smem_u32(s0 + kRfSlices * kRfA + sl * kRfB),
                        rb.bs + rf_tile_off(T, sl, jn / kRfHalves, kb) + (jn % kRfHalves) * (kRfN * kRfBK), kRfB,
                        &full[stage]);
            }
            if (++stage == kRfStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kRfN, false, false);
      uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
      bool ok = true;
      for (int f = 0; f < nf && ok; ++f) {
        const int mi = rf_matrix(c, f);
        if (mi < 0) continue;
        const long long T = c.mats[mi].T, jobs = T * kRfHalves * T;
        for (long long u = blockIdx.x; u < jobs && ok; u += gridDim.x) {
          for (long long kb = 0; kb < 4 * T && ok; ++kb) {
            const bool first = kb % kRfDrain == 0, last = kb % kRfDrain == kRfDrain - 1;
            if (!mbar_wait(&full[stage], phase, abort_flag, status) ||
                (first && !mbar_wait(&acc_empty[abuf], aphase ^ 1, abort_flag, status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + stage * kRfStage);
            rf_issue<LMAX>(tmem_base + abuf * (kRfAcc * kRfN), a0, a0 + kRfSlices * kRfA, idesc, first);
            tc_commit(&empty[stage]);
            if (last) {
              tc_commit(&acc_full[abuf]);
              if (++abuf == kRfBufs) {
                abuf = 0;
                aphase ^= 1;
              }
            }
            if (++stage == kRfStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, status);
    }
  } else {
    // ---------------- epilogue: warp e holds TMEM lanes 32 q.. and the kCols columns of group h
    const int e = warp - 2;
    const int q = warp & 3;
    const int h = e / 4;
    const int nacc = lmax - 1 < kRfAcc ? lmax - 1 : kRfAcc;
    uint32_t abuf = 0, aphase = 0;
    bool ok = true;
    for (int f = 0; f < nf && ok; ++f) {
      const int mi = rf_matrix(c, f);
      if (mi < 0) continue;
      const int T = c.mats[mi].T;
      const int np = T * 128, jobs = T * (np / kRfN);  // 32-bit: few registers beside the sums
      for (int u = blockIdx.x; u < jobs && ok; u += gridDim.x) {
        long long ib64, jn64;
        rf_job(u, T, ib64, jn64);
        const int i0 = (int)ib64 * kRfM, j0 = (int)jn64 * kRfN;
        constexpr int kCols = kRfN / (kRfEpiWarps / 4);  // this warp's columns
        float hi[kCols], lo[kCols];
#pragma unroll
        for (int t = 0; t < kCols; ++t) hi[t] = lo[t] = 0.f;
        for (int kd = 0; kd < 4 * T / kRfDrain; ++kd) {
          if (!mbar_wait(&acc_full[abuf], aphase, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int a = 0; a < kRfAcc; ++a) {
            if (a >= nacc) break;
#pragma unroll
            for (int g = 0; g < kCols / 8; ++g) {  // eight columns at a time: few registers beside the sums
              uint32_t v[8];
              tc_ld_32x32b_x8(tmem_base + ((uint32_t)(q * 32) << 16) + abuf * (kRfAcc * kRfN) + a * kRfN + h * kCols +
                                  g * 8,
                              v);
              tc_wait_ld();
#pragma unroll
              for (int t = 0; t < 8; ++t) df_add(hi[g * 8 + t], lo[g * 8 + t], __uint_as_float(v[t]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[abuf]);
          if (++abuf == kRfBufs) {
            abuf = 0;
            aphase ^= 1;
          }
        }
        if (!ok) break;
        const RfBufs rb = rf_bufs(c, c.mats[mi]);
        const int row = i0 + q * 32 + lane;
        const int er = rb.ex[row];
        float* out = rb.st + (long long)row * np + j0 + h * kCols;
        const int* ebc = rb.eb + j0 + h * kCols;
#pragma unroll
        for (int t4 = 0; t4 < kCols; t4 += 4) {  // four columns at a time (16-byte loads and stores)
          const int4 e4 = *reinterpret_cast<const int4*>(ebc + t4);
          const int ecs[4] = {e4.x, e4.y, e4.z, e4.w};
          float o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int col = j0 + h * kCols + t4 + u;
            const int sc = er + ecs[u];
            const float vh = scale_pow2(hi[t4 + u], sc), vl = scale_pow2(lo[t4 + u], sc);
            o[u] = mode == 0 ? ((row == col ? 1.f : 0.f) - vh) - vl : vh + vl;
          }
          *reinterpret_cast<float4*>(out + t4) = make_float4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ X1 = X0 + (T + T^T) / 2
// One CTA per upper tile (I, J) of a candidate: reads X0(I, J), T(I, J) and
// T(J, I) (through shared memory, transposed), writes X1(I, J) and its mirror.
__device__ void rf_sym_tile(const InvCtx& c, int mi, long long q) {
  const InvMat m = c.mats[mi];
  const int J = tri_root(q), I = (int)(q - tri(J));  // I <= J
  const RfBufs rb = rf_bufs(c, m);
  const long long np = (long long)m.T * 128;
  __shared__ float tt[32][33];  // a 32 x 32 block of T(J, I), transposed
  __shared__ float xx[32][33];  // the 32 x 32 block of X1(I, J) for the mirror
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  for (int bi = 0; bi < 4; ++bi)
    for (int bj = 0; bj < 4; ++bj) {
      const long long r0 = (long long)I * 128 + bi * 32, c0 = (long long)J * 128 + bj * 32;
      __syncthreads();
      for (int yy = ty; yy < 32; yy += 8) tt[tx][yy] = rb.st[(c0 + yy) * np + r0 + tx];  // T(c0+yy, r0+tx)
      __syncthreads();
      for (int yy = ty; yy < 32; yy += 8) {
        const long long r = r0 + yy, col = c0 + tx;
        float v = 0.f;
        if (r < m.d && col < m.d) {
          const float x0 = m.X[r * m.ld_out + col];
          v = x0 + 0.5f * (rb.st[r * np + col] + tt[yy][tx]);
          m.X[r * m.ld_out + col] = v;
        }
        xx[yy][tx] = v;
      }
      __syncthreads();
      // the mirror (a diagonal tile is written whole above: its formula is
      // symmetric in (r, col), bit for bit)
      if (I != J)
        for (int yy = ty; yy < 32; yy += 8) {
          const long long r = c0 + yy, col = r0 + tx;  // X1(c0+yy, r0+tx) = X1(r0+tx, c0+yy)
          if (r < m.d && col < m.d) m.X[r * m.ld_out + col] = xx[tx][yy];
        }
    }
  __syncthreads();  // tt and xx are free for the next tile
}

__global__ void __launch_bounds__(256) rf_sym_kernel(InvCtx c) {
  const int nf = *c.nflagged;
  for (int f = 0; f < nf; ++f) {
    const int mi = rf_matrix(c, f);
    if (mi < 0) continue;
    for (long long q = blockIdx.x; q < tri(c.mats[mi].T); q += gridDim.x) rf_sym_tile(c, mi, q);
  }
}

// ------------------------------------------------------------------ probes of the decision
// w = D v for the kRfProbes probes of each candidate, once (D does not change
// over the steps).  A warp per row r, D read by symmetry from its upper
// triangle (the row segment from r on, the column segment above r), with
// gamma_extra on the diagonal; each lane keeps the double-float sums of all
// probes over its columns, and the warp adds them up.
__global__ void __launch_bounds__(256) rf_w16_kernel(InvCtx c) {
  const int nf = *c.nflagged;
  const int lane = threadIdx.x % 32;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long nw = (long long)gridDim.x * blockDim.x / 32;
  for (int f = 0; f < nf; ++f) {
    const int mi = rf_matrix(c, f);
    if (mi < 0) continue;
    const InvMat m = c.mats[mi];
    const RfBufs rb = rf_bufs(c, m);
    const long long np = (long long)m.T * 128;
    for (long long r = gw; r < m.d; r += nw) {
      float hi[kRfProbes], lo[kRfProbes];
#pragma unroll
      for (int p = 0; p < kRfProbes; ++p) hi[p] = lo[p] = 0.f;
      for (long long col = lane; col < m.d; col += 32) {
        float x = col >= r ? m.D[r * m.ld_in + col] : m.D[col * m.ld_in + r];
        if (col == r) x += c.gamma_extra;
        const uint32_t sb = probe16_bits(col);  // bit p: sign of probe p at col
#pragma unroll
        for (int p = 0; p < kRfProbes; ++p) df_add(hi[p], lo[p], ((sb >> p) & 1u) ? x : -x);  // exact
      }
#pragma unroll
      for (int p = 0; p < kRfProbes; ++p) {
        float h = hi[p], l = lo[p];
        for (int o = 16; o > 0; o >>= 1) {
          const float oh = __shfl_xor_sync(0xffffffffu, h, o), ol = __shfl_xor_sync(0xffffffffu, l, o);
          df_add(h, l, oh);
          l += ol;
        }
        if (lane == 0) rb.w16[p * np + r] = df_pack(h, l);
      }
    }
  }
}

// y = X1 w for the kRfProbes probes of each candidate: a CTA per 8 rows (a
// warp per row), columns in chunks of 128 with the chunk's w staged in shared
// memory; double-float products and sums.
__global__ void __launch_bounds__(256) rf_y16_kernel(InvCtx c) {
  __shared__ __align__(16) float2 ws[kRfProbes * 128];
  const int nf = *c.nflagged;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int f = 0; f < nf; ++f) {
    const int mi = rf_matrix(c, f);
    if (mi < 0) continue;  // uniform over the grid
    const InvMat m = c.mats[mi];
    const RfBufs rb = rf_bufs(c, m);
    const long long np = (long long)m.T * 128;
    for (long long r0 = (long long)blockIdx.x * 8; r0 < m.d; r0 += (long long)gridDim.x * 8) {  // uniform over the block
      const long long r = r0 + warp;
      float hi[kRfProbes], lo[kRfProbes];
#pragma unroll
      for (int p = 0; p < kRfProbes; ++p) hi[p] = lo[p] = 0.f;
      for (long long c0 = 0; c0 < m.d; c0 += 128) {
        __syncthreads();  // the previous chunk's w has been read
        for (int e = threadIdx.x; e < kRfProbes * 128; e += 256) {
          const long long col = c0 + e % 128;
          ws[e] = col < m.d ? rb.w16[(e / 128) * np + col] : make_float2(0.f, 0.f);
        }
        __syncthreads();
        const long long col = c0 + 4 * lane;  // float4 reads stay inside the row (ld_out % 4 == 0)
        if (r < m.d && col < m.d) {
          const float4 x4 = *reinterpret_cast<const float4*>(m.X + r * m.ld_out + col);
          const float xs[4] = {x4.x, col + 1 < m.d ? x4.y : 0.f, col + 2 < m.d ? x4.z : 0.f,
                               col + 3 < m.d ? x4.w : 0.f};
#pragma unroll
          for (int p = 0; p < kRfProbes; ++p) {
            const float4 w01 = *reinterpret_cast<const float4*>(ws + p * 128 + 4 * lane);
            const float4 w23 = *reinterpret_cast<const float4*>(ws + p * 128 + 4 * lane + 2);
            df_add_prod(hi[p], lo[p], xs[0], w01.x, w01.y);
            df_add_prod(hi[p], lo[p], xs[1], w01.z, w01.w);
            df_add_prod(hi[p], lo[p], xs[2], w23.x, w23.y);
            df_add_prod(hi[p], lo[p], xs[3], w23.z, w23.w);
          }
        }
      }
#pragma unroll
      for (int p = 0; p < kRfProbes; ++p) {
        float h = hi[p], l = lo[p];
        for (int o = 16; o > 0; o >>= 1) {
          const float oh = __shfl_xor_sync(0xffffffffu, h, o), ol = __shfl_xor_sync(0xffffffffu, l, o);
          df_add(h, l, oh);
          l += ol;
        }
        if (lane == 0 && r < m.d) rb.y16[p * np + r] = df_pack(h, l);
      }
    }
  }
}

// ------------------------------------------------------------------ decision after the step
// The refined estimate from the kRfProbes probes (y = X1 w formed by
// rf_y16_kernel): accepted at most kRefinedResidual (twice the 2.5e-4 of the
// fp32 pass: a matrix refined to its fp32 storage floor sits near 2.5e-4, and
// the fp64 pass, whose result is stored in fp32 as well, cannot do better
// there).
constexpr double kRefinedResidual = 5.0e-4;
// Newton steps at most: the fp32 pass leaves the 4609-wide ResNet-50 conv
// factor at a residual near 6e-3, which one step takes to about 7e-4 (inside
// the 1e-3 bar, not inside the 5e-4 acceptance) and a second one to the fp32
// storage floor.
constexpr int kRfSteps = 2;

__global__ void __launch_bounds__(128) rf_decide_kernel(InvCtx c) {
  const int mi = rf_matrix(c, blockIdx.x);
  if (mi < 0) return;
  const InvMat m = c.mats[mi];
  const long long np = (long long)m.T * 128;
  const float2* y = rf_bufs(c, m).y16;
  __shared__ double red[128];
  // (y - v) in fp32: y_hi - v is exact while y is within a factor two of v
  // (a residual far below one), and larger differences need no precision;
  // per-thread sums in fp32 (a few hundred terms), the block's in fp64
  float e2 = 0.f;
  for (long long r = threadIdx.x; r < m.d; r += 128) {
    const uint32_t sb = probe16_bits(r);
#pragma unroll
    for (int p = 0; p < kRfProbes; ++p) {
      const float2 yv = y[p * np + r];
      const float dv = (yv.x - (((sb >> p) & 1u) ? 1.f : -1.f)) + yv.y;
      e2 = fmaf(dv, dv, e2);
    }
  }
  red[threadIdx.x] = (double)e2;
  __syncthreads();
  for (int s = 64; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double est = sqrt(red[0] / kRfProbes / (double)m.d);
    InvState& s = c.st[mi];
    s.est_res = (float)est;
    if (est <= kRefinedResidual) {  // false for NaN
      s.use64 = 0;
      s.refined = 1;
      s.refine = 0;  // settled: later steps skip it
    }
  }
}

// the fp64 pass's list: the flagged matrices the step did not settle
__global__ void rf_relist_kernel(InvCtx c) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const int nf = *c.nflagged;
  int k = 0;
  for (int f = 0; f < nf; ++f) {
    const int mi = c.flagged[f];
    if (c.st[mi].use64) c.flagged[k++] = mi;
  }
  *c.nflagged = k;
}

size_t refine_bytes(long long np) { return rf_bytes(np); }

int run_refine_pass(const InvCtx& ctx, int n, int Tmax, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  if (!ensure_smem_attr(dev, (const void*)rf_gemm_kernel<7>, kRfSmem) ||
      !ensure_smem_attr(dev, (const void*)rf_gemm_kernel<4>, kRfSmem) ||
      !ensure_smem_attr(dev, (const void*)rf_split_kernel, kRfSplitSmem))
    return KFAC_ERR_CUDA;
  int* status = device_status_ptr();
  if (!status) return KFAC_ERR_CUDA;
  // persistent grids over the flagged list: with nothing flagged every launch ends at once
  auto timed = [&](auto&& launch) {
    ProfMark pm;
    prof_begin(stream, pm);
    launch();
    prof_end(KFAC_K_INV_NEWTON, stream, pm, 0.0);
    count_launch();
  };
  rf_mark_kernel<<<(n + 127) / 128, 128, 0, stream>>>(ctx, n);
  count_launch();
  (void)Tmax;
  timed([&] { rf_w16_kernel<<<4 * sms, 256, 0, stream>>>(ctx); });
  // up to kRfSteps steps; a matrix whose estimate meets the bar after a step
  // leaves the candidates (the ones that follow skip it)
  for (int step = 0; step < kRfSteps; ++step) {
    timed([&] { rf_split_kernel<<<dim3((unsigned)(2 * sms), 2), 256, kRfSplitSmem, stream>>>(ctx, 0); });  // D, X
    timed([&] { rf_gemm_kernel<7><<<sms, kRfThreads, kRfSmem, stream>>>(ctx, n, 0, status); });
    timed([&] { rf_split_kernel<<<dim3((unsigned)(2 * sms), 1), 256, kRfSplitSmem, stream>>>(ctx, 2); });  // S
    timed([&] { rf_gemm_kernel<4><<<sms, kRfThreads, kRfSmem, stream>>>(ctx, n, 1, status); });
    timed([&] { rf_sym_kernel<<<4 * sms, 256, 0, stream>>>(ctx); });
    timed([&] { rf_y16_kernel<<<4 * sms, 256, 0, stream>>>(ctx); });
    rf_decide_kernel<<<n, 128, 0, stream>>>(ctx);
    count_launch();
  }
  rf_relist_kernel<<<1, 32, 0, stream>>>(ctx);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA;
}

}  // namespace kfac
