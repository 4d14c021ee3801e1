// fp32 pass of the batched damped inverse on tcgen05 tensor cores (the
// algorithm is described in inverse.cu).  Every tile product is a split-bf16
// NT GEMM (three slices per fp32 value, six MMAs per 16-wide k-step, each
// 32-wide k-block drained into round-to-nearest fp32 sums, as in gemm_tc.cu),
// so the arithmetic has close to fp32 accuracy.
//
// To make every product NT with K-major operands, the blocked inverse
// W = L^-1 is kept transposed, U = W^T (block upper triangular), and so are
// the forward-substitution accumulators C:
//   panel(k)   L_rk = A_rk Winv_k^T                 (r > k)
//              U_rk = C'_rk Winv_k^T                 (r < k)     [C'_rk = C_kr^T]
//   update(k)  A_rc  -= L_rk L_ck^T                  (r >= c > k)
//              C'_cr -= U_ck L_rk^T, first time =    (c <= k < r)
//   X_ij = sum_{t >= j} U_it U_jt^T                  (i <= j), mirrored.
// Work buffers, stacked over the matrices of a group (matrix m owns rows
// [row_off, row_off + n_pad) of each, with one leading dimension LD = max n_pad):
//   Acc   fp32 [R][LD]  lower blocks: A (Schur complements), upper blocks: C'
//   U     bf16 [3][R][LD]   slices of U
//   P     bf16 [3][R][128]  slices of block column k of Acc (the panel inputs)
//   Lp    bf16 [3][2R][kOuter * 128]  slices of L_rj for the block columns j
//                                      of an outer panel (see kOuter); two
//                                      buffers, alternating between panels
//   Winv  bf16 [3][n*128][128]
// so that one tensor map per buffer serves every matrix.  Updates land in Acc
// through TMA add-reductions (no read-modify-write in the kernel).
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "inverse_common.cuh"
#include "launch.h"
#include "split.cuh"

namespace kfac {

constexpr int kItBK = 32;
constexpr int kItA = 128 * kItBK * 2;  // one slice of the A tile (8 KB)
constexpr int kItThreads = 320;
// 16-wide k-steps accumulated in one TMEM accumulator between two drains into
// the epilogue's round-to-nearest fp32 sums
constexpr int kItDrain = 2;
// the same with 16-bit operands (two slices, three MMAs per k-step): their
// slicing error (2^-16 of a product) dominates the accumulator's, so the
// accumulator is drained every eight k-steps, as in the 16-bit GEMM of the
// preconditioning
constexpr int kItDrain16 = 8;
// the tile; the probe signs s() of its two blocks, their indices in class
// order and the four class starts of each
constexpr int kLoadSmem = (128 * 129 + 2 * 128) * 4 + (2 * 128 + 2 * 8) * 4;

enum { kItPanel = 0, kItUpdate = 1, kItLauum = 2 };

// Shared-memory ring of each kind: a stage holds one 32-wide k-block of all
// three slices of A (128 rows) and B.  The panel's B is the 128-row diagonal
// inverse; its eight epilogue warps pass their 32 x 64 blocks through
// shared memory (64 KB): three 48 KB stages.  X = U U^T (B of 256 rows) also stores straight from registers
// (row stores of X and of its mirror): three 72 KB stages.  The updates add
// into the work buffer through 32 x 32 TMA reductions staged in shared memory
// (64 KB): two 72 KB stages.  (Vector reductions straight from registers,
// which would free room for a third stage, left the MMA issuer waiting for a
// drained accumulator 35 % of the time instead of 4 %: the lanes' rows are
// 128 B apart, so each reduction instruction touches 32 lines.)
constexpr int kItOutBlock = 4096;  // one 32 x 32 fp32 block
// The panel's epilogue warps pass their 32 rows through shared memory in
// 64-column halves (32 x 64 fp32 each) on the way to the bf16 slice stores.
constexpr int kItPanelStage = 32 * 64 * 4;
template <int KIND>
struct ItCfg {
  static constexpr int b_rows = KIND == kItPanel ? 128 : 256;
  static constexpr int stages = KIND == kItUpdate ? 2 : 3;
  static constexpr int b_slice = b_rows * kItBK * 2;
  static constexpr int stage = kSlices * (kItA + b_slice);
  static constexpr int out = KIND == kItUpdate ? 8 * 2 * kItOutBlock : KIND == kItPanel ? 8 * kItPanelStage : 0;
  static constexpr int smem = stages * stage + out + 1024 + 256;
};

// Two-level blocking of the update: block columns are grouped in outer panels
// of kOuter.  Inside an outer panel each step updates only the panel's own
// columns (and the substitution accumulators of the panel's block rows); the
// last step of the panel applies the whole panel (K = kOuter * 128) to
// everything right of it, so the fp32 trailing matrix is read and written once
// per outer panel instead of once per block column.  Lp keeps the L_rk of the
// panel's kOuter block columns side by side.
constexpr int kOuter = 4;
constexpr int kLpW = kOuter * 128;

struct TcBufs {
  float* acc;
  uint16_t* u;
  uint16_t* p;
  uint16_t* lp;
  uint16_t* winv;
  long long R, LD;
  int n;
};

struct ItParams {
  CUtensorMap mUA, mUB, mP, mLA, mLB, mW, mAcc;
  long long ro[kInvMaxGroup];
  int T[kInvMaxGroup];
  int job_begin[kInvMaxGroup + 1];
  TcBufs b;
  const InvMat* mats;
  InvState* st;
  int* status;
  long long total_jobs;
  int n, k;
  int upd_mode;  // update launches: kUpdInner / kUpdFull / kUpdNear / kUpdFar
  int use_route; // 1 once the operand widths of AUTO are decided (before: three slices for all)
  int lp_off;    // first row of the current outer panel's Lp buffer (0 or R)
};

struct ItJob {
  int m, valid;
  const CUtensorMap* ma;
  const CUtensorMap* mb;
  int a_y, a_x0, b_y, b_x0, b_box, K, n_mma;
  int o_y, o_x, mode;  // output rows/cols; panel: 0 -> Lp, 1 -> U; update: 0 add, 1 store
  int i, j;            // X tile (i, j) of the pair j, j+1 (lauum)
  int ns;              // bf16 slices per operand for this matrix: 3 (24-bit) or 2 (16-bit)
};

// k-steps of one accumulator drain for operands of `ns` slices
__device__ __forceinline__ int it_drain(int ns) { return ns == 2 ? kItDrain16 : kItDrain; }

// jobs of the update at step k for a matrix of T block rows: rows r > k pair
// their columns c in (k, r]; columns c <= k pair their rows r > k
__host__ __device__ inline long long it_pairs(long long R) { return ((R + 1) / 2) * ((R + 2) / 2); }

// The update jobs of step k for a matrix of T block rows.
//   outer step (k the last block column of its outer panel [p0, k]):
//     Schur  A_rc -= sum_{j=p0..k} L_rj L_cj^T          rows r >= c_lo, column pairs c in [c_lo, min(r, c_hi)]
//     subst  C'_cr -= sum_{j=max(c,p0)..k} U_cj L_rj^T   c <= k, row pairs r in [c_lo, c_hi]
//     with the column range [k+1, T) whole (kUpdFull), or cut into the next
//     outer panel's columns (kUpdNear: [k+1, k+kOuter]) and the rest (kUpdFar)
//   inner step (the panel continues after k; cl its last block column):
//     Schur  A_rc -= L_rk L_ck^T                       rows r > k, column pairs c in (k, min(r, cl)]
//     subst  C'_cr -= U_ck L_rk^T                      c <= k, row pairs r in (k, cl]
enum { kUpdInner = 0, kUpdFull = 1, kUpdNear = 2, kUpdFar = 3 };
struct UpdShape {
  int outer, p0, c_lo, c_hi;
  long long nschur, nsub;
};
__host__ __device__ inline UpdShape upd_shape(int T, int k, int mode) {
  UpdShape sh;
  sh.p0 = k - k % kOuter;
  sh.outer = mode != kUpdInner;
  if (mode == kUpdInner) {
    sh.c_lo = k + 1;
    sh.c_hi = (sh.p0 + kOuter < T ? sh.p0 + kOuter : T) - 1;
  } else if (mode == kUpdFull) {
    sh.c_lo = k + 1;
    sh.c_hi = T - 1;
  } else if (mode == kUpdNear) {
    sh.c_lo = k + 1;
    sh.c_hi = k + kOuter < T - 1 ? k + kOuter : T - 1;
  } else {
    sh.c_lo = k + kOuter + 1;
    sh.c_hi = T - 1;
  }
  sh.nschur = sh.nsub = 0;
  if (sh.c_lo > T - 1 || sh.c_hi < sh.c_lo) return sh;
  // rows [c_lo, c_hi) pair the columns [c_lo, r]; rows from c_hi on all pair [c_lo, c_hi]
  const int r1 = (sh.c_hi < T ? sh.c_hi : T) - sh.c_lo;
  const int cmax = (sh.c_hi - sh.c_lo + 2) / 2;
  sh.nschur = it_pairs(r1) + (long long)(T > sh.c_hi ? T - sh.c_hi : 0) * cmax;
  const int rl = sh.c_hi < T - 1 ? sh.c_hi : T - 1;
  sh.nsub = (long long)(k + 1) * ((rl - sh.c_lo + 2) / 2);
  return sh;
}

template <int KIND>
__device__ ItJob it_decode(const ItParams& prm, long long u) {
  int lo = 0, hi = prm.n;  // find m with job_begin[m] <= u < job_begin[m+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (prm.job_begin[mid] <= u)
      lo = mid;
    else
      hi = mid;
  }
  ItJob J;
  const int m = lo;
  const long long q = u - prm.job_begin[m];
  const long long ro = prm.ro[m];
  const int T = prm.T[m];
  const int k = prm.k;
  J.m = m;
  J.valid = !prm.st[m].failed;
  J.ns = (prm.use_route && prm.st[m].slices == 2) ? 2 : kSlices;
  J.i = J.j = 0;
  J.mode = 0;
  if (KIND == kItPanel) {
    const int r = q < k ? (int)q : (int)q + 1;
    J.ma = &prm.mP;
    J.a_y = (int)(ro + r * 128);
    J.a_x0 = 0;
    J.mb = &prm.mW;
    J.b_y = m * 128;
    J.b_x0 = 0;
    J.b_box = 128;
    J.K = 128;
    J.n_mma = 128;
    J.o_y = (int)(ro + r * 128);
    J.o_x = k * 128;
    J.mode = r > k ? 0 : 1;
  } else if (KIND == kItUpdate) {
    const UpdShape sh = upd_shape(T, k, prm.upd_mode);
    const int lp_off = prm.lp_off;  // this outer panel's half of the double-buffered Lp
    J.mb = &prm.mLB;
    J.b_box = 256;
    if (q < sh.nschur) {
      const int r1 = (sh.c_hi < T ? sh.c_hi : T) - sh.c_lo;
      int r, cp;
      if (q < it_pairs(r1)) {
        int lo = 0, hi = r1;  // it_pairs(lo) <= q < it_pairs(hi)
        while (hi - lo > 1) {
          const int mid = (lo + hi) / 2;
          if (it_pairs(mid) <= q)
            lo = mid;
          else
            hi = mid;
        }
        r = sh.c_lo + lo;
        cp = (int)(q - it_pairs(lo));
      } else {
        const int cmax = (sh.c_hi - sh.c_lo + 2) / 2;
        const long long qq = q - it_pairs(r1);
        r = sh.c_hi + (int)(qq / cmax);
        cp = (int)(qq % cmax);
      }
      const int c = sh.c_lo + 2 * cp;
      const int w = min(2, min(r, sh.c_hi) - c + 1);
      J.ma = &prm.mLA;
      J.a_y = (int)(lp_off + ro + r * 128);
      J.b_y = (int)(lp_off + ro + c * 128);
      J.a_x0 = J.b_x0 = sh.outer ? 0 : (k - sh.p0) * 128;
      J.K = sh.outer ? (k + 1 - sh.p0) * 128 : 128;
      J.n_mma = 128 * w;
      J.o_y = (int)(ro + r * 128);
      J.o_x = c * 128;
      J.mode = 0;
    } else {
      const long long q2 = q - sh.nschur;
      const int rl = sh.c_hi < T - 1 ? sh.c_hi : T - 1;  // rows r in [c_lo, rl]
      const int hp = (rl - sh.c_lo + 2) / 2;
      const int c = (int)(q2 / hp), rp = (int)(q2 % hp);
      const int r = sh.c_lo + 2 * rp;
      const int w = min(2, rl - r + 1);
      J.ma = &prm.mUA;
      J.a_y = (int)(ro + c * 128);
      J.b_y = (int)(lp_off + ro + r * 128);
      if (sh.outer) {
        const int j0 = max(c, sh.p0);  // U_cj = 0 for j < c
        J.a_x0 = j0 * 128;
        J.b_x0 = (j0 - sh.p0) * 128;
        J.K = (k + 1 - j0) * 128;
        J.mode = c >= sh.p0 ? 1 : 0;  // first contribution to C'_cr (r beyond the panel)
      } else {
        J.a_x0 = k * 128;
        J.b_x0 = (k - sh.p0) * 128;
        J.K = 128;
        J.mode = c == k ? 1 : 0;
      }
      J.n_mma = 128 * w;
      J.o_y = (int)(ro + c * 128);
      J.o_x = r * 128;
    }
  } else {
    // Row i pairs the columns (j, j + 1) for j = i, i + 2, ...; the jobs are
    // numbered so that consecutive ones share B = U rows (j, j + 1): even rows
    // first, then odd ones; within a parity class by the pair j = par + 2a,
    // then by the rows i = par + 2b, b <= a (a + 1 jobs per pair, all with
    // K = (T - j) * 128).
    const long long n_even = tri((T + 1) / 2);
    const int par = q < n_even ? 0 : 1;
    const long long qp = par ? q - n_even : q;
    const int a = tri_root(qp);
    const int i = par + 2 * (int)(qp - tri(a));
    const int j = par + 2 * a;
    const int w = min(2, T - j);
    J.i = i;
    J.j = j;
    J.ma = &prm.mUA;
    J.a_y = (int)(ro + i * 128);
    J.a_x0 = j * 128;
    J.mb = &prm.mUB;
    J.b_y = (int)(ro + j * 128);
    J.b_x0 = j * 128;
    J.b_box = 256;
    J.K = (T - j) * 128;
    J.n_mma = 128 * w;
  }
  return J;
}

// K-major shared-memory descriptor, 64-byte swizzle (as in gemm_tc.cu)
__device__ __forceinline__ uint64_t it_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;
  return d;
}

template <int KIND>
__global__ void __launch_bounds__(kItThreads, 1) inv_tc_kernel(const __grid_constant__ ItParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Cfg = ItCfg<KIND>;
  uint8_t* out_stage = smem + Cfg::stages * Cfg::stage;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + Cfg::out);
  uint64_t* empty = full + Cfg::stages;
  uint64_t* acc_full = empty + Cfg::stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);
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
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (long long u = blockIdx.x; u < prm.total_jobs && !*abort_flag; u += gridDim.x) {
        const ItJob J = it_decode<KIND>(prm, u);
        if (!J.valid) continue;
        const uint32_t bytes = J.ns * (kItA + J.b_box * kItBK * 2);
        for (int kb = 0; kb < J.K / kItBK; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, prm.status)) break;
          uint8_t* s0 = smem + stage * Cfg::stage;
          mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
          for (int s = 0; s < kSlices; ++s) {
            if (s >= J.ns) break;
            tma_load_3d(s0 + s * kItA, J.ma, J.a_x0 + kb * kItBK, J.a_y, s, &full[stage]);
            tma_load_3d(s0 + kSlices * kItA + s * Cfg::b_slice, J.mb, J.b_x0 + kb * kItBK, J.b_y, s, &full[stage]);
          }
          if (++stage == Cfg::stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (long long u = blockIdx.x; u < prm.total_jobs && ok; u += gridDim.x) {
        const ItJob J = it_decode<KIND>(prm, u);
        if (!J.valid) continue;
        const uint32_t idesc = idesc_bf16_f32(J.n_mma, false, false);
        const int n16 = J.K / 16;  // 16-wide k-steps of the job
        const int dr = it_drain(J.ns);
        int st16 = 0;
        for (int kb = 0; kb < J.K / kItBK && ok; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, prm.status)) {
            ok = false;
            break;
          }
          const uint32_t a0 = smem_u32(smem + stage * Cfg::stage);
          const uint32_t b0 = a0 + kSlices * kItA;
#pragma unroll
          for (int kk = 0; kk < kItBK / 16; ++kk, ++st16) {
            const bool gfirst = st16 % dr == 0;
            const bool glast = st16 % dr == dr - 1 || st16 == n16 - 1;
            if (gfirst) {
              if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, prm.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d_tmem = tmem_base + acc * 256;
            const uint32_t off = kk * 32;
            uint64_t da[kSlices], db[kSlices];
#pragma unroll
            for (int s = 0; s < kSlices; ++s) {
              da[s] = it_desc(a0 + s * kItA + off);
              db[s] = it_desc(b0 + s * Cfg::b_slice + off);
            }
            // hi*hi, hi*mid, mid*hi (16-bit operands); and hi*lo, lo*hi, mid*mid (24-bit)
            tc_mma_bf16(d_tmem, da[0], db[0], idesc, gfirst ? 0u : 1u);
            tc_mma_bf16(d_tmem, da[0], db[1], idesc, 1u);
            tc_mma_bf16(d_tmem, da[1], db[0], idesc, 1u);
            if (J.ns == kSlices) {
              tc_mma_bf16(d_tmem, da[0], db[2], idesc, 1u);
              tc_mma_bf16(d_tmem, da[2], db[0], idesc, 1u);
              tc_mma_bf16(d_tmem, da[1], db[1], idesc, 1u);
            }
            if (glast) {
              tc_commit(&acc_full[acc]);
              acc ^= 1;
              if (acc == 0) acc_phase ^= 1;
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == Cfg::stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, prm.status);
    }
  } else {
    const int e = warp - 2;
    const int q = warp & 3;  // TMEM lane quarter
    const int h = e / 4;     // column half of the 256-wide tile (of the panel's 128-wide one)
    // first column of this warp's share: 128 wide, or 64 wide on the panel's tile
    const int col0w = KIND == kItPanel ? h * 64 : h * 128;
    constexpr int kDrainGroups = KIND == kItPanel ? 2 : 4;  // 32-column TMEM loads per drain
    uint32_t acc = 0, acc_phase = 0;
    int obuf = 0;
    bool ok = true;
    for (long long u = blockIdx.x; u < prm.total_jobs && ok; u += gridDim.x) {
      const ItJob J = it_decode<KIND>(prm, u);
      if (!J.valid) continue;
      const bool mine = col0w < J.n_mma;  // this warp's columns exist
      float run[128];
#pragma unroll
      for (int t = 0; t < 128; ++t) run[t] = 0.f;
      const int nsteps = (J.K / 16 + it_drain(J.ns) - 1) / it_drain(J.ns);
      for (int st = 0; st < nsteps; ++st) {
        if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, prm.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (mine) {
          const uint32_t base = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256 + col0w;
#pragma unroll
          for (int g = 0; g < kDrainGroups; ++g) {
            uint32_t v[32];
            tc_ld_32x32b_x32(base + g * 32, v);
            tc_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) run[g * 32 + t] += __uint_as_float(v[t]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok || !mine) continue;
      const int mrow = q * 32 + lane;  // row of the 128-row output tile
      if (KIND == kItPanel) {
        // L_rk (r > k) into Lp, or U_rk (r < k) into U, as three bf16 slices.
        // The two warps of a lane quarter take 64 columns each; a warp's 32
        // rows go through shared memory (16-byte chunks XOR-swizzled by row:
        // conflict-free both ways), so that each store instruction writes four
        // whole 128-byte row segments instead of 32 pieces of 32 different rows.
        uint16_t* dst0;
        long long sstride, ld;
        if (J.mode == 0) {
          dst0 = prm.b.lp + (long long)(prm.lp_off + J.o_y + q * 32) * kLpW + (long long)((J.o_x / 128) % kOuter) * 128;
          sstride = 2 * prm.b.R * kLpW;
          ld = kLpW;
        } else {
          dst0 = prm.b.u + (long long)(J.o_y + q * 32) * prm.b.LD + J.o_x;
          sstride = prm.b.R * prm.b.LD;
          ld = prm.b.LD;
        }
        float* stg = reinterpret_cast<float*>(out_stage + e * kItPanelStage);
        __syncwarp();  // the previous job's rows have been read
#pragma unroll
        for (int j = 0; j < 16; ++j)
          *reinterpret_cast<float4*>(stg + lane * 64 + ((j ^ (lane & 7)) << 2)) =
              make_float4(run[4 * j], run[4 * j + 1], run[4 * j + 2], run[4 * j + 3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int r = it * 4 + lane / 8, k2 = 2 * (lane % 8);
          const float4 v0 = *reinterpret_cast<const float4*>(stg + r * 64 + ((k2 ^ (r & 7)) << 2));
          const float4 v1 = *reinterpret_cast<const float4*>(stg + r * 64 + (((k2 + 1) ^ (r & 7)) << 2));
          const float x8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          split8_store(x8, dst0 + (long long)r * ld + col0w + k2 * 4, sstride);
        }
      } else if (KIND == kItUpdate) {
        // -acc into Acc through 32 x 32 TMA add-reductions (or stores, first time)
        for (int g = 0; g < 4; ++g) {
          uint8_t* buf = out_stage + (e * 2 + obuf) * kItOutBlock;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float4 o = make_float4(-run[g * 32 + 4 * jj], -run[g * 32 + 4 * jj + 1], -run[g * 32 + 4 * jj + 2],
                                         -run[g * 32 + 4 * jj + 3]);
            *reinterpret_cast<float4*>(buf + lane * 128 + ((jj ^ (lane & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int cx = J.o_x + h * 128 + g * 32, cy = J.o_y + q * 32;
            if (J.mode == 1)
              tma_store_2d(&prm.mAcc, buf, cx, cy);
            else
              tma_reduce_add_2d(&prm.mAcc, buf, cx, cy);
            bulk_commit();
          }
          obuf ^= 1;
        }
      } else {
        // X tile (i, j + h) of the pair and its mirror, in 32 x 32 blocks: the
        // mirror straight from the registers (lanes hold consecutive rows, so
        // the stores run along the mirror's rows), the tile as row stores of
        // this thread's 32 columns
        const InvMat mt = prm.mats[J.m];
        const int jt = J.j + h;
        const long long row = (long long)J.i * 128 + q * 32 + lane;
        // rows 32-byte aligned: each lane writes whole sectors of its row
        const bool v8 = (mt.ld_out % 8) == 0 && (reinterpret_cast<uintptr_t>(mt.X) & 31) == 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const long long col0 = (long long)jt * 128 + g * 32;
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const long long col = col0 + t;
            if (row < mt.d && col < mt.d && (J.i != jt || mrow <= g * 32 + t))
              mt.X[col * mt.ld_out + row] = run[g * 32 + t];
          }
          if (row < mt.d) {
            float* xr = mt.X + row * mt.ld_out + col0;
            if (col0 + 32 <= mt.d && (J.i != jt || mrow <= g * 32)) {
              if (v8) {
#pragma unroll
                for (int t = 0; t < 32; t += 8)
                  st_global_v8(xr + t, run[g * 32 + t], run[g * 32 + t + 1], run[g * 32 + t + 2], run[g * 32 + t + 3],
                               run[g * 32 + t + 4], run[g * 32 + t + 5], run[g * 32 + t + 6], run[g * 32 + t + 7]);
              } else {
#pragma unroll
                for (int t = 0; t < 32; t += 4)
                  *reinterpret_cast<float4*>(xr + t) =
                      make_float4(run[g * 32 + t], run[g * 32 + t + 1], run[g * 32 + t + 2], run[g * 32 + t + 3]);
              }
            } else {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (col0 + t < mt.d && (J.i != jt || mrow <= g * 32 + t)) xr[t] = run[g * 32 + t];
            }
          }
        }
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ D -> Acc (lower blocks)
// Lower tiles counted column by column: block column C starts at tile
// C T - C (C - 1) / 2 (T - C tiles each).
__host__ __device__ inline long long load_col_start(long long C, long long T) { return C * T - C * (C - 1) / 2; }

// The lower tiles of block columns [c_begin, c_end) of every matrix.
// mode: kLoadCopy (the tiles into the work buffer), kLoadSums (AUTO's partial
// sums only), or both
constexpr int kLoadCopy = 1, kLoadSums = 2;
__global__ void __launch_bounds__(256) tc_load_kernel(InvCtx c, TcBufs b, int c_begin, int c_end, int mode) {
  const int mi = blockIdx.y;
  if (!inv_active(c, mi, false)) return;
  const InvMat m = c.mats[mi];
  const int ce = c_end < m.T ? c_end : m.T;
  if (c_begin >= ce) return;
  const long long q = load_col_start(c_begin, m.T) + blockIdx.x;
  if (q >= load_col_start(ce, m.T)) return;
  int C = c_begin;
  while (load_col_start(C + 1, m.T) <= q) ++C;
  const int R = C + (int)(q - load_col_start(C, m.T));  // lower tile (R, C), R >= C
  float* A = b.acc + m.row_off * b.LD;
  extern __shared__ __align__(16) uint8_t load_smem[];
  float* sub = reinterpret_cast<float*>(load_smem);  // 128 x 129: sub[i][j] = D[C*128 + i][R*128 + j]
  const int t = threadIdx.x;
  // read the upper tile (C, R) of D along its rows, 16 float4 per thread, all
  // issued before the first shared-memory store (ld_in % 4 == 0 keeps a
  // float4 that starts inside the row inside it)
  {
    float4 v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int e = t + 256 * u, i = e / 32, j4 = (e % 32) * 4;
      const long long gc = (long long)C * 128 + i, gr = (long long)R * 128 + j4;
      v[u] = (gc < m.d && gr < m.d) ? *reinterpret_cast<const float4*>(m.D + gc * m.ld_in + gr)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int e = t + 256 * u, i = e / 32, j4 = (e % 32) * 4;
      float* d = sub + i * 129 + j4;
      d[0] = v[u].x;
      d[1] = v[u].y;
      d[2] = v[u].z;
      d[3] = v[u].w;
    }
  }
  __syncthreads();
  if (c.gpart && (mode & kLoadSums)) {
    // AUTO: per tile, for the rows of block C along the tile's rows and for
    // the rows of block R down its columns (the mirror), the partial sums of
    //   |D_rc| (c != r)      -> gpart: Gershgorin radii (tc_route_kernel) and ||D||_1
    //   D_rc v_p(c)          -> wpart: w = D v for the residual probes
    // With v_p(c) = s(c) H4[p][class(c)] (probes.cuh), the four sums come
    // from one double-float sum of s(c) D_rc per class of c (the sign flips
    // are exact), combined by a 4-point Hadamard transform at the end; each
    // thread walks its columns (or rows) class by class, in index order within
    // a class (so that the sums do not depend on scheduling).  On a diagonal
    // tile only its upper triangle counts, and the diagonal itself (with
    // gamma_extra) goes into w only.  Columns of the tile at or past d hold
    // whatever the float4 loads brought from the padding: they are left out;
    // rows past d were loaded as zero.
    float* sr = sub + 128 * 129;  // s() of block R's indices
    float* sc = sr + 128;         // and of block C's
    int* lr = reinterpret_cast<int*>(sc + 128);  // block R's indices 0..127 in class order
    int* lc = lr + 128;                           // block C's
    int* orr = lc + 128;                          // class starts in lr (4, then the warps' counts)
    int* occ = orr + 8;                           // and in lc
    {
      // threads 0-127 sort block R's indices by class, 128-255 block C's:
      // each warp counts its indices of each class with a ballot, then every
      // index lands at (class start) + (the class's count in earlier warps) +
      // (its rank among the warp's indices of the class)
      const int half = t / 128, e = t % 128, wq = e / 32, ln = e % 32;
      const long long gi = (long long)(half ? C : R) * 128 + e;
      (half ? sc : sr)[e] = probe_base_sign(gi);
      const int cls = probe_class(gi);
      __shared__ int wcnt[2][4][4];  // [half][warp][class]
      unsigned masks[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        masks[b] = __ballot_sync(0xffffffffu, cls == b);
        if (ln == 0) wcnt[half][wq][b] = __popc(masks[b]);
      }
      __syncthreads();
      int start = 0;
      for (int b = 0; b < cls; ++b)
        for (int w = 0; w < 4; ++w) start += wcnt[half][w][b];
      for (int w = 0; w < wq; ++w) start += wcnt[half][w][cls];
      const unsigned mk = cls == 0 ? masks[0] : cls == 1 ? masks[1] : cls == 2 ? masks[2] : masks[3];
      start += __popc(mk & ((1u << ln) - 1u));
      (half ? lc : lr)[start] = e;
      if (e < 5) {  // class starts 0..4
        int o = 0;
        for (int b = 0; b < e; ++b)
          for (int w = 0; w < 4; ++w) o += wcnt[half][w][b];
        (half ? occ : orr)[e] = o;
      }
    }
    __syncthreads();
    float* gp = c.gpart + m.off_gpart;
    float2* wp = c.wpart + m.off_gpart * kProbes;
    const long long cleft = m.d - (long long)R * 128;
    const int jmax = cleft < 128 ? (int)cleft : 128;
    float s = 0.f, yhi[4] = {0.f, 0.f, 0.f, 0.f}, ylo[4] = {0.f, 0.f, 0.f, 0.f};  // class sums
    long long slot = -1;  // (row block, column block) of this thread's sums
    int row = 0;
    if (R == C) {
      if (t < 128) {
        row = t;
        slot = (long long)C * m.T + C;
        if (t < jmax) {
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            for (int q = orr[b]; q < orr[b + 1]; ++q) {
              const int j = lr[q];
              if (j <= t || j >= jmax) continue;
              const float x = sub[t * 129 + j];
              s += fabsf(x);
              df_add(yhi[b], ylo[b], x * sr[j]);
            }
            for (int q = occ[b]; q < occ[b + 1]; ++q) {
              const int i2 = lc[q];
              if (i2 >= t) continue;
              const float x = sub[i2 * 129 + t];
              s += fabsf(x);
              df_add(yhi[b], ylo[b], x * sc[i2]);
            }
          }
          const float dg = sub[t * 129 + t] + c.gamma_extra;
          const int bt = probe_class((long long)C * 128 + t);
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (b == bt) df_add(yhi[b], ylo[b], dg * sc[t]);
        }
      }
    } else if (t < 128) {
      row = t;
      slot = (long long)C * m.T + R;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        for (int q = orr[b]; q < orr[b + 1]; ++q) {
          const int j = lr[q];
          if (j >= jmax) continue;
          const float x = sub[t * 129 + j];
          s += fabsf(x);
          df_add(yhi[b], ylo[b], x * sr[j]);
        }
    } else {
      row = t - 128;
      slot = (long long)R * m.T + C;
      if (row < jmax) {
#pragma unroll
        for (int b = 0; b < 4; ++b)
          for (int q = occ[b]; q < occ[b + 1]; ++q) {
            const int i2 = lc[q];
            const float x = sub[i2 * 129 + row];
            s += fabsf(x);
            df_add(yhi[b], ylo[b], x * sc[i2]);
          }
      }
    }
    if (slot >= 0) {
      gp[slot * 128 + row] = s;
      // w_p = sum_b H4[p][b] Y_b (double-float butterflies)
      float ah = yhi[0], al = ylo[0], bh = yhi[0], bl = ylo[0], ch = yhi[2], cl = ylo[2], dh = yhi[2], dl = ylo[2];
      df_add(ah, al, yhi[1]);
      al += ylo[1];
      df_add(bh, bl, -yhi[1]);
      bl -= ylo[1];
      df_add(ch, cl, yhi[3]);
      cl += ylo[3];
      df_add(dh, dl, -yhi[3]);
      dl -= ylo[3];
      float w0h = ah, w0l = al, w2h = ah, w2l = al, w1h = bh, w1l = bl, w3h = bh, w3l = bl;
      df_add(w0h, w0l, ch);  // Y0 + Y1 + Y2 + Y3
      w0l += cl;
      df_add(w2h, w2l, -ch);  // Y0 + Y1 - Y2 - Y3
      w2l -= cl;
      df_add(w1h, w1l, dh);  // Y0 - Y1 + Y2 - Y3
      w1l += dl;
      df_add(w3h, w3l, -dh);  // Y0 - Y1 - Y2 + Y3
      w3l -= dl;
      wp[(slot * kProbes + 0) * 128 + row] = make_float2(w0h, w0l);
      wp[(slot * kProbes + 1) * 128 + row] = make_float2(w1h, w1l);
      wp[(slot * kProbes + 2) * 128 + row] = make_float2(w2h, w2l);
      wp[(slot * kProbes + 3) * 128 + row] = make_float2(w3h, w3l);
    }
  }
  // write the lower tile (R, C) of the work buffer along its rows: element
  // (R*128 + j, C*128 + i) = D(C*128 + i, R*128 + j); identity past d, zero
  // above the diagonal, gamma_extra on it
  if (!(mode & kLoadCopy)) return;
#pragma unroll 4
  for (int e = t; e < 128 * 32; e += 256) {
    const int j = e / 32, i4 = (e % 32) * 4;
    const long long gr = (long long)R * 128 + j;
    float o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i4 + u;
      const long long gc = (long long)C * 128 + i;
      if (gr >= m.d || gc >= m.d)
        o[u] = (gr == gc) ? 1.f : 0.f;
      else if (gr < gc)
        o[u] = 0.f;
      else
        o[u] = sub[i * 129 + j] + ((gr == gc) ? c.gamma_extra : 0.f);
    }
    *reinterpret_cast<float4*>(A + gr * b.LD + (long long)C * 128 + i4) = make_float4(o[0], o[1], o[2], o[3]);
  }
  // zero the sub-diagonal U block (R, R-1): the X = U U^T products read it when they pair block rows
  if (R == C + 1) {
    const long long ss = b.R * b.LD;
    for (int e = threadIdx.x; e < 128 * 16; e += 256) {
      const int rr = e / 16, cc = (e % 16) * 8;
      uint16_t* dst = b.u + (m.row_off + (long long)R * 128 + rr) * b.LD + (long long)C * 128 + cc;
#pragma unroll
      for (int s = 0; s < kSlices; ++s) *reinterpret_cast<uint4*>(dst + s * ss) = make_uint4(0, 0, 0, 0);
    }
  }
}

// ------------------------------------------------------------------ operand width (AUTO)
// The Gershgorin discs of D + gamma_extra I hold every eigenvalue in
// [min_r (D_rr - s_r), max_r (D_rr + s_r)], s_r = sum_{c != r} |D_rc| (the
// partial sums of tc_load_kernel).  When the lower end is positive and the
// ratio is at most kSlices16Kappa, the matrix is that well conditioned and its
// fp32 pass runs with 16-bit operands (two slices); else with 24-bit ones.
// The residual probe checks the result either way.
__device__ __forceinline__ unsigned ordered_bits(float x) {  // monotone float -> unsigned map
  const unsigned b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(unsigned u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// One CTA per (128-row block, matrix): its rows' disc ends, reduced over the
// CTA, then into the matrix's running min / max (exact, so the order of the
// CTAs does not matter); the matrix's last CTA to finish takes the decision.
__global__ void __launch_bounds__(128) tc_route_kernel(InvCtx c) {
  const int mi = blockIdx.y;
  if (!inv_active(c, mi, false)) return;
  const InvMat m = c.mats[mi];
  const int b = blockIdx.x;
  if (b >= m.T) return;
  const float* gp = c.gpart + m.off_gpart + (long long)b * m.T * 128;
  __shared__ float slo[128], shi[128];
  __shared__ int sbad, slast;
  if (threadIdx.x == 0) sbad = 0;
  __syncthreads();
  const long long r = (long long)b * 128 + threadIdx.x;
  float lo = 3.0e38f, hi = 0.f;
  if (r < m.d) {
    float off = 0.f;
#pragma unroll 8
    for (int cb = 0; cb < m.T; ++cb) off += gp[(long long)cb * 128 + threadIdx.x];
    const float dg = m.D[r * m.ld_in + r] + c.gamma_extra;
    lo = dg - off;
    hi = dg + off;
    if (!isfinite(lo) || !isfinite(hi)) sbad = 1;
    // ||D||_1 row sum, and w = D v for the residual probes, from the load's partial sums
    c.rowsum[m.off_rowsum + r] = off + fabsf(dg);
    const float2* wp = c.wpart + (m.off_gpart + (long long)b * m.T * 128) * kProbes;
    const long long np = (long long)m.T * 128;
#pragma unroll
    for (int p = 0; p < kProbes; ++p) {
      float whi = 0.f, wlo = 0.f;
      for (int cb = 0; cb < m.T; ++cb) {
        const float2 v = wp[((long long)cb * kProbes + p) * 128 + threadIdx.x];
        df_add(whi, wlo, v.x);
        wlo += v.y;
      }
      c.probe[m.off_probe + p * np + r] = df_pack(whi, wlo);
    }
  }
  slo[threadIdx.x] = lo;
  shi[threadIdx.x] = hi;
  __syncthreads();
  for (int s = 64; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      slo[threadIdx.x] = fminf(slo[threadIdx.x], slo[threadIdx.x + s]);
      shi[threadIdx.x] = fmaxf(shi[threadIdx.x], shi[threadIdx.x + s]);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    InvState& st = c.st[mi];
    if (sbad) atomicOr(&st.gbad, 1);
    atomicMin(&st.glo, ordered_bits(slo[0]));
    atomicMax(&st.ghi, ordered_bits(shi[0]));
    __threadfence();
    slast = atomicAdd(&st.gdone, 1) == m.T - 1;
  }
  __syncthreads();
  if (slast && threadIdx.x == 0) {
    InvState& st = c.st[mi];
    __threadfence();
    const float glo = from_ordered_bits(atomicOr(&st.glo, 0u));
    const float ghi = from_ordered_bits(atomicOr(&st.ghi, 0u));
    const int bad = atomicOr(&st.gbad, 0);
    st.slices = (!bad && glo > 0.f && ghi <= kSlices16Kappa * glo) ? 2 : kSlices;
  }
}

// ------------------------------------------------------------------ step k: diagonal block
// Cholesky and inverse of the diagonal block k: Winv_k rows (the panel's B
// operand) and U_kk = Winv_k^T, as bf16 slices.
__global__ void __launch_bounds__(256, 2) tc_diag_kernel(InvCtx c, TcBufs b, int k) {
  const int mi = blockIdx.x;
  if (!inv_active(c, mi, true)) return;
  const InvMat m = c.mats[mi];
  if (k >= m.T) return;
  const int t = threadIdx.x;
  extern __shared__ __align__(16) uint8_t diag_smem[];
  float* a = reinterpret_cast<float*>(diag_smem);
  const float* src = b.acc + (m.row_off + (long long)k * 128) * b.LD + (long long)k * 128;
  {
    // 16 float4 per thread (LD is a multiple of 128), all loads issued before the stores
    float4 v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = t + 256 * q;  // row e / 32, columns 4 (e % 32) ..
      v[q] = *reinterpret_cast<const float4*>(src + (long long)(e / 32) * b.LD + (e % 32) * 4);
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = t + 256 * q, r = e / 32, c4 = (e % 32) * 4;
      float* d = a + r * kDiagPitch + c4;
      d[0] = c4 <= r ? v[q].x : 0.f;
      d[1] = c4 + 1 <= r ? v[q].y : 0.f;
      d[2] = c4 + 2 <= r ? v[q].z : 0.f;
      d[3] = c4 + 3 <= r ? v[q].w : 0.f;
    }
  }
  __syncthreads();
  float min_piv;
  const int fail = block_chol_inv<float>(a, m.d - k * 128, min_piv);
  if (fail >= 0) {
    if (t == 0) {
      c.st[mi].failed = 1;
      c.st[mi].info32 = k * 128 + fail + 1;
    }
    return;
  }
  if (t == 0) atomicMin(reinterpret_cast<int*>(&c.st[mi].min_piv), __float_as_int(min_piv));
  // the 128 rows of Winv, then the 128 rows of U_kk = Winv^T: a half-warp per
  // row, each lane 8 consecutive columns, so that every store is coalesced
  const int half = t / 16, c8 = (t % 16) * 8;
  for (int rr = half; rr < 256; rr += 16) {
    const bool upper = rr >= 128;
    const int row = rr % 128;
    uint16_t* dst = upper ? b.u + (m.row_off + (long long)k * 128 + row) * b.LD + (long long)k * 128
                          : b.winv + ((long long)mi * 128 + row) * 128;
    const long long slice = upper ? b.R * b.LD : (long long)b.n * 128 * 128;
    float v8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)  // Winv[row][c] (zero above the diagonal), or Winv[c][row]
      v8[e] = upper ? a[(c8 + e) * kDiagPitch + row] : a[row * kDiagPitch + c8 + e];
    split8_store(v8, dst + c8, slice);
  }
}

// ------------------------------------------------------------------ step k: slices of block column k
// tile row r (the x-th row other than k) of block column k of Acc -> P slices;
// a warp per row, coalesced
__global__ void __launch_bounds__(256) tc_prep_kernel(InvCtx c, TcBufs b, int k) {
  const int mi = blockIdx.y;
  if (!inv_active(c, mi, true)) return;
  const InvMat m = c.mats[mi];
  if (k >= m.T) return;
  const int x = blockIdx.x;
  const int r = x < k ? x : x + 1;
  if (r >= m.T) return;
  const int lane = threadIdx.x % 32, wq = threadIdx.x / 32;
  for (int rr = wq; rr < 128; rr += 8) {
    const float* src = b.acc + (m.row_off + (long long)r * 128 + rr) * b.LD + (long long)k * 128 + lane * 4;
    const float4 v = *reinterpret_cast<const float4*>(src);
    uint16_t* dst = b.p + (m.row_off + (long long)r * 128 + rr) * 128 + lane * 4;
    __nv_bfloat16 s0[kSlices], s1[kSlices], s2[kSlices], s3[kSlices];
    split_value(v.x, s0);
    split_value(v.y, s1);
    split_value(v.z, s2);
    split_value(v.w, s3);
#pragma unroll
    for (int s = 0; s < kSlices; ++s) {
      __nv_bfloat162 p0, p1;
      p0.x = s0[s];
      p0.y = s1[s];
      p1.x = s2[s];
      p1.y = s3[s];
      *reinterpret_cast<uint2*>(dst + s * b.R * 128) =
          make_uint2(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1));
    }
  }
}

// ------------------------------------------------------------------ residual probe y = X w, ||X||_F^2 (AUTO)
// A CTA per strip of kPrRows rows of X (full symmetric, as written by the
// X = U U^T step), columns in chunks of 128: the CTA stages the chunk's w (all
// probes) in shared memory, lane l of each warp takes columns 4l..4l+3 of the
// chunk for the kPrWarpRows rows of its warp, and the next chunk's X and w are
// fetched while the current one is summed.  Double-float products and sums.
constexpr int kPrWarpRows = 4;
constexpr int kPrRows = 8 * kPrWarpRows;
// y = X w over one strip of kPrRows rows of matrix mi (each warp its own
// kPrWarpRows rows); ||X||_F^2 of the strip is added to the matrix's state
// when count_norm is set.  Called by all threads of the block alike.
__device__ void probe_strip(const InvCtx& c, int mi, long long strip, bool count_norm) {
  __shared__ __align__(16) float2 ws[2][kProbes * 128];  // w of a chunk, [probe][column], double-buffered
  const InvMat m = c.mats[mi];
  if (strip * kPrRows >= m.d) return;
  const int t = threadIdx.x, lane = t % 32;
  const long long rw = strip * kPrRows + (t / 32) * kPrWarpRows;  // the warp's first row
  const long long np = (long long)m.T * 128;
  const float2* w = c.probe + m.off_probe;
  float2* y = c.probe + m.off_probe + (long long)kProbes * np;
  const int nrow = rw >= m.d ? 0 : (int)(m.d - rw < kPrWarpRows ? m.d - rw : kPrWarpRows);
  const int nchunk = (int)((m.d + 127) / 128);
  float2 wn[2];                // this thread's share of the next chunk's w
  float4 xn[kPrWarpRows];      // and of its X (columns past d are masked when summed)
  auto fetch = [&](int ch) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = t + 256 * h;
      const long long col = (long long)ch * 128 + e % 128;
      wn[h] = col < m.d ? w[(e / 128) * np + col] : make_float2(0.f, 0.f);
    }
    const long long col = (long long)ch * 128 + 4 * lane;  // float4 reads of columns col..col+3 stay inside the row (ld_out % 4 == 0)
#pragma unroll
    for (int q = 0; q < kPrWarpRows; ++q)
      xn[q] = (q < nrow && col < m.d) ? *reinterpret_cast<const float4*>(m.X + (rw + q) * m.ld_out + col)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  float hi[kPrWarpRows][kProbes], lo[kPrWarpRows][kProbes];
#pragma unroll
  for (int q = 0; q < kPrWarpRows; ++q)
#pragma unroll
    for (int p = 0; p < kProbes; ++p) hi[q][p] = lo[q][p] = 0.f;
  float sq = 0.f;
  fetch(0);
  for (int ch = 0; ch < nchunk; ++ch) {
    float2* wb = ws[ch & 1];
    wb[t] = wn[0];
    wb[t + 256] = wn[1];
    __syncthreads();  // (the other buffer was last read before the previous barrier)
    const long long col = (long long)ch * 128 + 4 * lane;
    float xs[kPrWarpRows][4];
#pragma unroll
    for (int q = 0; q < kPrWarpRows; ++q) {
      xs[q][0] = col < m.d ? xn[q].x : 0.f;
      xs[q][1] = col + 1 < m.d ? xn[q].y : 0.f;
      xs[q][2] = col + 2 < m.d ? xn[q].z : 0.f;
      xs[q][3] = col + 3 < m.d ? xn[q].w : 0.f;
    }
    if (ch + 1 < nchunk) fetch(ch + 1);
#pragma unroll
    for (int q = 0; q < kPrWarpRows; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) sq += xs[q][e] * xs[q][e];
#pragma unroll
    for (int p = 0; p < kProbes; ++p) {
      const float4 w01 = *reinterpret_cast<const float4*>(wb + p * 128 + 4 * lane);
      const float4 w23 = *reinterpret_cast<const float4*>(wb + p * 128 + 4 * lane + 2);
      const float wh[4] = {w01.x, w01.z, w23.x, w23.z}, wl[4] = {w01.y, w01.w, w23.y, w23.w};
#pragma unroll
      for (int q = 0; q < kPrWarpRows; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) df_add_prod(hi[q][p], lo[q][p], xs[q][e], wh[e], wl[e]);
    }
  }
#pragma unroll
  for (int q = 0; q < kPrWarpRows; ++q) {
#pragma unroll
    for (int p = 0; p < kProbes; ++p) {
      // combine the 32 lanes' double-float partial sums
      float h = hi[q][p], l = lo[q][p];
      for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, h, o), ol = __shfl_xor_sync(0xffffffffu, l, o);
        df_add(h, l, oh);
        l += ol;
      }
      if (lane == 0 && q < nrow) y[p * np + rw + q] = df_pack(h, l);
    }
  }
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (lane == 0 && nrow > 0 && count_norm) atomicAdd(&c.st[mi].xnorm2, sq);
  __syncthreads();  // the next strip of this block (persistent callers) rewrites ws
}

__global__ void __launch_bounds__(256, 2) tc_probe_kernel(InvCtx c, int t_only) {
  const int mi = blockIdx.y;
  if (!inv_active(c, mi, true)) return;
  if (t_only && c.mats[mi].T != t_only) return;  // only the matrices of T block rows
  probe_strip(c, mi, blockIdx.x, true);
}

// ------------------------------------------------------------------ host side
static size_t al256(size_t v) { return (v + 255) & ~size_t(255); }



TcLayout tc_layout(int n, const int* T) {
  TcLayout L;
  long long R = 0, LD = 128;
  for (int i = 0; i < n; ++i) {
    R += (long long)T[i] * 128;
    if ((long long)T[i] * 128 > LD) LD = (long long)T[i] * 128;
  }
  L.R_tot = R;
  L.LD = LD;
  size_t off = 0;
  L.acc = off;
  off += al256((size_t)R * LD * 4);
  L.u = off;
  off += al256((size_t)kSlices * R * LD * 2);
  L.p = off;
  off += al256((size_t)kSlices * R * 128 * 2);
  L.lp = off;
  off += al256((size_t)kSlices * 2 * R * kLpW * 2);  // two outer panels' worth (see run_tc_pass)
  L.winv = off;
  off += al256((size_t)kSlices * n * 128 * 128 * 2);
  L.bytes = off;
  return L;
}

// slices [3][rows][cols] bf16, K-major boxes {32, box_rows}
static bool enc_slices(EncodeTiledFn enc, CUtensorMap* map, uint16_t* base, long long rows, long long cols,
                       int box_rows) {
  cuuint64_t gdim[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)kSlices};
  cuuint64_t gstride[2] = {(cuuint64_t)cols * 2, (cuuint64_t)(rows * cols * 2)};
  cuuint32_t box[3] = {(cuuint32_t)kItBK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 128 x 128 x 128 tile products (units of 128^3 multiply-adds) of one
// launch's jobs for a matrix of T block rows
template <int KIND>
static double tile_macs(int T, int k, int upd_mode, int t_only) {
  double u = 0.0;
  if (KIND == kItPanel) {
    u = T > k ? T - 1 : 0;  // one 128 x 128 tile, K = 128, per job
  } else if (KIND == kItUpdate) {
    const UpdShape sh = upd_shape(T, k, upd_mode);
    if (sh.nschur + sh.nsub == 0) return 0.0;
    const int kunits = sh.outer ? k + 1 - sh.p0 : 1;
    for (int r = sh.c_lo; r < T; ++r) u += (double)((r < sh.c_hi ? r : sh.c_hi) - sh.c_lo + 1) * kunits;
    const int rl = sh.c_hi < T - 1 ? sh.c_hi : T - 1;
    for (int c = 0; c <= k; ++c)
      u += (double)(rl - sh.c_lo + 1) * (sh.outer ? k + 1 - (c > sh.p0 ? c : sh.p0) : 1);
  } else if (t_only == 0 || T == t_only) {
    for (int j = 0; j < T; ++j) {  // pair (j, j + 1): rows i = j % 2, j % 2 + 2, .., j
      const int w = T - j < 2 ? T - j : 2;
      u += (double)(j / 2 + 1) * w * (T - j);
    }
  }
  return u;
}

// Job counts of one launch (filling prm->job_begin); *work gets the launch's
// flops (2 per multiply-add of its tile products).
template <int KIND>
static long long count_jobs(ItParams* prm, const int* Ts, int n, int k, int upd_mode, double* work,
                            int t_only = 0) {
  long long jobs = 0;
  double w = 0.0;
  for (int i = 0; i < n; ++i) {
    prm->job_begin[i] = (int)jobs;
    long long cnt = 0;
    const int T = Ts[i];
    if (KIND == kItPanel) {
      cnt = T > k ? T - 1 : 0;
    } else if (KIND == kItUpdate) {
      const UpdShape sh = upd_shape(T, k, upd_mode);
      cnt = sh.nschur + sh.nsub;
    } else {
      cnt = (t_only == 0 || T == t_only) ? it_pairs(T) : 0;
    }
    if (work && cnt > 0) w += tile_macs<KIND>(T, k, upd_mode, t_only);
    jobs += cnt;
  }
  prm->job_begin[n] = (int)jobs;
  if (work) *work = w * 2.0 * 128.0 * 128.0 * 128.0;
  return jobs;
}

template <int KIND>
static int launch_it(ItParams* prm, const int* Ts, int n, int k, int grid_cap, cudaStream_t stream,
                     int upd_mode = kUpdInner, int t_only = 0) {
  double work = 0.0;
  const long long jobs = count_jobs<KIND>(prm, Ts, n, k, upd_mode, &work, t_only);
  prm->total_jobs = jobs;
  prm->k = k;
  prm->upd_mode = upd_mode;
  if (jobs == 0) return KFAC_OK;
  const int grid = (int)(jobs < grid_cap ? jobs : grid_cap);
  ProfMark pm;
  prof_begin(stream, pm);
  inv_tc_kernel<KIND><<<grid, kItThreads, ItCfg<KIND>::smem, stream>>>(*prm);
  prof_end(KIND == kItPanel ? KFAC_K_INV_PANEL : KIND == kItUpdate ? KFAC_K_INV_UPDATE : KFAC_K_INV_LAUUM, stream,
           pm, work);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA;
}

// Five streams of this library per device, three of highest and two of lowest
// priority, and the events that fork work from the caller's stream onto them
// and join it back (created once, kept until exit).
struct AuxStream {
  cudaStream_t hi = nullptr, hi2 = nullptr, hi3 = nullptr, lo = nullptr, lo2 = nullptr;
  cudaEvent_t start = nullptr, fork = nullptr, join = nullptr, end = nullptr, norms = nullptr, early = nullptr,
              lodone = nullptr, prep0 = nullptr, prep1 = nullptr, early2 = nullptr, lodone2 = nullptr,
              loaded = nullptr;
};
// One set per (device, caller's stream), up to kAuxSets per device, so that
// inverses issued on different streams run concurrently.  A further caller
// stream gets no set (false): its calls run on that stream alone, without the
// look-ahead, since sharing a set's events between two callers would let one
// call wait on the other's event records.
constexpr int kAuxSets = 4;
static bool aux_stream(int dev, cudaStream_t caller, AuxStream* out) {
  static std::mutex mu;
  static AuxStream table[64][kAuxSets];
  static cudaStream_t owner[64][kAuxSets];
  if (dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  int slot = -1;
  for (int i = 0; i < kAuxSets && slot < 0; ++i)
    if (table[dev][i].hi && owner[dev][i] == caller) slot = i;
  for (int i = 0; i < kAuxSets && slot < 0; ++i)
    if (!table[dev][i].hi) {
      slot = i;
      owner[dev][i] = caller;
    }
  if (slot < 0) return false;
  AuxStream& t = table[dev][slot];
  if (!t.hi) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return false;
    cudaEvent_t ev[12];
    for (int i = 0; i < 12; ++i)
      if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) return false;
    cudaStream_t st, st2, st3, sl, sl2;
    if (cudaStreamCreateWithPriority(&st3, cudaStreamNonBlocking, greatest) != cudaSuccess) return false;
    if (cudaStreamCreateWithPriority(&sl, cudaStreamNonBlocking, least) != cudaSuccess) return false;
    if (cudaStreamCreateWithPriority(&sl2, cudaStreamNonBlocking, least) != cudaSuccess) return false;
    if (cudaStreamCreateWithPriority(&st2, cudaStreamNonBlocking, greatest) != cudaSuccess) return false;
    if (cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, greatest) != cudaSuccess) return false;
    t.lo = sl;
    t.lo2 = sl2;
    t.hi3 = st3;
    t.early2 = ev[9];
    t.lodone2 = ev[10];
    t.loaded = ev[11];
    t.hi2 = st2;
    t.start = ev[0];
    t.fork = ev[1];
    t.join = ev[2];
    t.end = ev[3];
    t.norms = ev[4];
    t.early = ev[5];
    t.lodone = ev[6];
    t.prep0 = ev[7];
    t.prep1 = ev[8];
    t.hi = st;
  }
  *out = t;
  return true;
}

bool fp64_chain_stream(int dev, cudaStream_t caller, cudaStream_t* chain, cudaEvent_t (&ev)[4]) {
  AuxStream aux;
  if (!aux_stream(dev, caller, &aux)) return false;
  *chain = aux.hi;
  ev[0] = aux.start;
  ev[1] = aux.fork;
  ev[2] = aux.join;
  ev[3] = aux.end;
  return true;
}

// A CUDA-core launch of the inverse, timed as `kind` while the launch profile
// records (kfac_profile).
template <typename F>
static void timed_launch(int kind, cudaStream_t stream, F&& launch) {
  ProfMark pm;
  prof_begin(stream, pm);
  launch();
  prof_end(kind, stream, pm, 0.0);
  count_launch();
}


// Jobs per CTA of a far update: its CTAs retire every few jobs, so that the
// higher-priority chain on the other stream finds SMs within tens of us.
constexpr int kFarJobsPerCta = 4;

int run_tc_pass(const InvCtx& ctx, const InvMat* host_mats, int n, int Tmax, const int* Ts, const TcLayout& L,
                cudaStream_t stream) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return KFAC_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  if (!ensure_smem_attr(dev, (const void*)inv_tc_kernel<kItPanel>, ItCfg<kItPanel>::smem) ||
      !ensure_smem_attr(dev, (const void*)inv_tc_kernel<kItUpdate>, ItCfg<kItUpdate>::smem) ||
      !ensure_smem_attr(dev, (const void*)inv_tc_kernel<kItLauum>, ItCfg<kItLauum>::smem) ||
      !ensure_smem_attr(dev, (const void*)tc_diag_kernel, diag_smem_bytes<float>()) ||
      !ensure_smem_attr(dev, (const void*)tc_load_kernel, kLoadSmem))
    return KFAC_ERR_CUDA;
  int* status = device_status_ptr();
  if (!status) return KFAC_ERR_CUDA;

  TcBufs b;
  b.acc = reinterpret_cast<float*>(ctx.region + L.acc);
  b.u = reinterpret_cast<uint16_t*>(ctx.region + L.u);
  b.p = reinterpret_cast<uint16_t*>(ctx.region + L.p);
  b.lp = reinterpret_cast<uint16_t*>(ctx.region + L.lp);
  b.winv = reinterpret_cast<uint16_t*>(ctx.region + L.winv);
  b.R = L.R_tot;
  b.LD = L.LD;
  b.n = n;

  ItParams* prm = new ItParams;
  memset(prm, 0, sizeof(ItParams));
  bool ok = enc_slices(enc, &prm->mUA, b.u, b.R, b.LD, 128) && enc_slices(enc, &prm->mUB, b.u, b.R, b.LD, 256) &&
            enc_slices(enc, &prm->mP, b.p, b.R, 128, 128) && enc_slices(enc, &prm->mLA, b.lp, 2 * b.R, kLpW, 128) &&
            enc_slices(enc, &prm->mLB, b.lp, 2 * b.R, kLpW, 256) &&
            enc_slices(enc, &prm->mW, b.winv, (long long)n * 128, 128, 128);
  {
    cuuint64_t gdim[2] = {(cuuint64_t)b.LD, (cuuint64_t)b.R};
    cuuint64_t gstride[1] = {(cuuint64_t)b.LD * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    ok = ok && enc(&prm->mAcc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, b.acc, gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  if (!ok) {
    delete prm;
    return KFAC_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) {
    prm->ro[i] = host_mats[i].row_off;
    prm->T[i] = Ts[i];
  }
  prm->b = b;
  prm->mats = ctx.mats;
  prm->st = ctx.st;
  prm->status = status;
  prm->n = n;

  int rc = KFAC_OK;
  // Look-ahead: at the last step of each outer panel the trailing update is
  // cut into the next outer panel's block columns (near) and the rest (far).
  // The sweep itself (diagonal blocks, slicing, panels, inner and near
  // updates) runs on the library's highest-priority stream; each far update
  // runs on the caller's stream, in CTAs of a few jobs, and is joined before
  // the next outer step.  Whenever SMs come free the hardware gives them to
  // the sweep first, and the far update fills the rest.  The next panel's
  // steps only touch their own block columns, and the far update's inputs stay
  // intact meanwhile: Lp is double-buffered between outer panels, and the next
  // panel writes U only in its own block columns.
  AuxStream aux;
  const bool fork_ok = aux_stream(dev, stream, &aux);
  cudaStream_t main = stream;  // the sweep's stream
  if (fork_ok) {
    if (cudaEventRecord(aux.start, stream) != cudaSuccess || cudaStreamWaitEvent(aux.hi, aux.start, 0) != cudaSuccess)
      rc = KFAC_ERR_CUDA;
    main = aux.hi;
  }
  // D into the work buffer: the first outer panel's block columns on the
  // sweep's stream, the rest (and AUTO's operand-width decision, which needs
  // every row sum) on a third highest-priority stream beside the first steps
  // of the sweep, which only touch the first outer panel; the sweep waits for
  // them before its first outer update.  Until then every matrix runs with
  // three slices.
  bool split_load = false;
  prm->use_route = ctx.gpart ? 0 : 1;
  if (rc == KFAC_OK) {
    const int c_split = fork_ok && Tmax > kOuter ? kOuter : Tmax;
    split_load = c_split < Tmax;
    long long cnt_a = 0, cnt_b = 0;
    for (int i = 0; i < n; ++i) {
      const int ci = c_split < Ts[i] ? c_split : Ts[i];
      const long long a = load_col_start(ci, Ts[i]);
      cnt_a = a > cnt_a ? a : cnt_a;
      const long long bb = tri(Ts[i]) - a;
      cnt_b = bb > cnt_b ? bb : cnt_b;
    }
    // with the load split, the first outer panel is only copied on the
    // sweep's stream (the first diagonal block waits for it); its partial
    // sums are formed beside the sweep with the rest of D
    const int mode_a = split_load && ctx.gpart ? kLoadCopy : kLoadCopy | kLoadSums;
    timed_launch(KFAC_K_INV_AUX, main, [&] {
      tc_load_kernel<<<dim3((unsigned)cnt_a, n), 256, kLoadSmem, main>>>(ctx, b, 0, c_split, mode_a);
    });
    cudaStream_t rs = main;  // where the rest of D and the decision go
    if (split_load) {
      // the rest of D at lowest priority (its CTAs take the SMs the first
      // steps leave free), the decision at highest once both parts are in
      rs = aux.hi3;
      if (cudaStreamWaitEvent(aux.lo, aux.start, 0) != cudaSuccess) rc = KFAC_ERR_CUDA;
      if (ctx.gpart)
        timed_launch(KFAC_K_INV_AUX, aux.lo, [&] {
          tc_load_kernel<<<dim3((unsigned)cnt_a, n), 256, kLoadSmem, aux.lo>>>(ctx, b, 0, c_split, kLoadSums);
        });
      timed_launch(KFAC_K_INV_AUX, aux.lo, [&] {
        tc_load_kernel<<<dim3((unsigned)cnt_b, n), 256, kLoadSmem, aux.lo>>>(ctx, b, c_split, Tmax,
                                                                             kLoadCopy | kLoadSums);
      });
      if (cudaEventRecord(aux.norms, aux.lo) != cudaSuccess || cudaStreamWaitEvent(rs, aux.norms, 0) != cudaSuccess ||
          cudaEventRecord(aux.fork, main) != cudaSuccess || cudaStreamWaitEvent(rs, aux.fork, 0) != cudaSuccess)
        rc = KFAC_ERR_CUDA;
    }
    if (ctx.gpart) timed_launch(KFAC_K_INV_AUX, rs, [&] { tc_route_kernel<<<dim3((unsigned)Tmax, n), 128, 0, rs>>>(ctx); });
    // the residual probes read the decision kernel's w = D v: the early ones
    // (on lo2) may be issued before the sweep has waited for it
    if (split_load && (cudaEventRecord(aux.loaded, rs) != cudaSuccess ||
                       cudaStreamWaitEvent(aux.lo2, aux.loaded, 0) != cudaSuccess))
      rc = KFAC_ERR_CUDA;
    if (!split_load) prm->use_route = 1;
  }
  bool pending = false;  // a far update in flight on `stream`
  bool early_any = false;
  for (int k = 0; k < Tmax && rc == KFAC_OK; ++k) {
    if (split_load && k == kOuter - 1) {
      // the rest of D is in the work buffer and the operand widths are known
      if (cudaStreamWaitEvent(main, aux.loaded, 0) != cudaSuccess) {
        rc = KFAC_ERR_CUDA;
        break;
      }
      prm->use_route = 1;
    }
    // matrices of k block rows finished their sweep at step k - 1: their
    // X = U U^T and residual probe run now, at lowest priority, in CTAs of
    // two jobs, beside the larger matrices' sweep; the probes on a stream of
    // their own, so that the next group's X = U U^T need not wait for them
    bool ends_here = false;
    for (int i = 0; i < n; ++i) ends_here = ends_here || Ts[i] == k;
    if (fork_ok && k > 0 && ends_here) {
      if (cudaEventRecord(aux.early, main) != cudaSuccess || cudaStreamWaitEvent(aux.lo, aux.early, 0) != cudaSuccess) {
        rc = KFAC_ERR_CUDA;
        break;
      }
      const long long lj = count_jobs<kItLauum>(prm, Ts, n, 0, kUpdInner, nullptr, k);
      rc = launch_it<kItLauum>(prm, Ts, n, 0, (int)((lj + 1) / 2), aux.lo, kUpdInner, k);
      if (rc != KFAC_OK) break;
      if (ctx.want_rowsum) {
        if (cudaEventRecord(aux.early2, aux.lo) != cudaSuccess ||
            cudaStreamWaitEvent(aux.lo2, aux.early2, 0) != cudaSuccess) {
          rc = KFAC_ERR_CUDA;
          break;
        }
        timed_launch(KFAC_K_INV_AUX, aux.lo2,
                     [&] { tc_probe_kernel<<<dim3((unsigned)(k * 128 / kPrRows), n), 256, 0, aux.lo2>>>(ctx, k); });
      }
      early_any = true;
    }
    prm->lp_off = (int)(((k / kOuter) & 1) * b.R);
    // the diagonal block and the slicing of the rest of block column k are
    // independent: the slicing runs on the second sweep stream
    const bool fork_prep = fork_ok && Tmax > 1;
    if (fork_prep && (cudaEventRecord(aux.prep0, main) != cudaSuccess ||
                      cudaStreamWaitEvent(aux.hi2, aux.prep0, 0) != cudaSuccess)) {
      rc = KFAC_ERR_CUDA;
      break;
    }
    timed_launch(KFAC_K_INV_DIAG, main, [&] { tc_diag_kernel<<<n, 256, diag_smem_bytes<float>(), main>>>(ctx, b, k); });
    if (Tmax > 1) {
      cudaStream_t ps = fork_prep ? aux.hi2 : main;
      timed_launch(KFAC_K_INV_PREP, ps, [&] { tc_prep_kernel<<<dim3((unsigned)(Tmax - 1), n), 256, 0, ps>>>(ctx, b, k); });
    }
    if (fork_prep && (cudaEventRecord(aux.prep1, aux.hi2) != cudaSuccess ||
                      cudaStreamWaitEvent(main, aux.prep1, 0) != cudaSuccess)) {
      rc = KFAC_ERR_CUDA;
      break;
    }
    rc = launch_it<kItPanel>(prm, Ts, n, k, sms, main);
    if (rc != KFAC_OK) break;
    if (k % kOuter != kOuter - 1) {
      rc = launch_it<kItUpdate>(prm, Ts, n, k, sms, main, kUpdInner);
      continue;
    }
    if (pending) {
      if (cudaStreamWaitEvent(main, aux.join, 0) != cudaSuccess) {
        rc = KFAC_ERR_CUDA;
        break;
      }
      pending = false;
    }
    const long long far_jobs = fork_ok ? count_jobs<kItUpdate>(prm, Ts, n, k, kUpdFar, nullptr) : 0;
    if (far_jobs < 2 * sms) {
      rc = launch_it<kItUpdate>(prm, Ts, n, k, sms, main, kUpdFull);
      continue;
    }
    if (cudaEventRecord(aux.fork, main) != cudaSuccess || cudaStreamWaitEvent(stream, aux.fork, 0) != cudaSuccess) {
      rc = KFAC_ERR_CUDA;
      break;
    }
    const int far_grid = (int)((far_jobs + kFarJobsPerCta - 1) / kFarJobsPerCta);
    rc = launch_it<kItUpdate>(prm, Ts, n, k, far_grid, stream, kUpdFar);
    if (rc != KFAC_OK) break;
    if (cudaEventRecord(aux.join, stream) != cudaSuccess) {
      rc = KFAC_ERR_CUDA;
      break;
    }
    pending = true;
    rc = launch_it<kItUpdate>(prm, Ts, n, k, sms, main, kUpdNear);
  }
  if (pending && cudaStreamWaitEvent(main, aux.join, 0) != cudaSuccess) rc = KFAC_ERR_CUDA;
  // the matrices that finished last (all of them when nothing was started early)
  const int t_last = early_any ? Tmax : 0;
  if (rc == KFAC_OK) rc = launch_it<kItLauum>(prm, Ts, n, 0, sms, main, kUpdInner, t_last);
  if (rc == KFAC_OK && ctx.want_rowsum) {
    // y = X w (w = D v from the decision kernel, ordered before on this stream)
    timed_launch(KFAC_K_INV_AUX, main,
                 [&] { tc_probe_kernel<<<dim3((unsigned)(Tmax * 128 / kPrRows), n), 256, 0, main>>>(ctx, t_last); });
  }
  // the early X = U U^T and probes on the lowest-priority stream
  if (early_any && (cudaEventRecord(aux.lodone, aux.lo) != cudaSuccess ||
                    cudaStreamWaitEvent(main, aux.lodone, 0) != cudaSuccess ||
                    cudaEventRecord(aux.lodone2, aux.lo2) != cudaSuccess ||
                    cudaStreamWaitEvent(main, aux.lodone2, 0) != cudaSuccess))
    rc = KFAC_ERR_CUDA;
  // everything is ordered on the caller's stream again, also after an error
  if (fork_ok && (cudaEventRecord(aux.end, main) != cudaSuccess || cudaStreamWaitEvent(stream, aux.end, 0) != cudaSuccess))
    rc = KFAC_ERR_CUDA;
  delete prm;
  if (rc == KFAC_OK && cudaGetLastError() != cudaSuccess) rc = KFAC_ERR_CUDA;
  return rc;
}

}  // namespace kfac
