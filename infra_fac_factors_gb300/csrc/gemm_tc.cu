// Split-bf16 NT GEMM on tcgen05 tensor cores, grouped over many problems:
//
//     C[m, n] = alpha * sum_k A[m, k] B[n, k]        (A: M x K, B: N x K)
//
// Every fp32 operand x is carried as three bf16 slices x = hi + mid + lo (all
// 24 bits of fp32).  With all three read (NS = 3), each 16-wide k-step issues
// six MMAs: hi*hi + hi*mid + mid*hi + hi*lo + lo*hi + mid*mid (the dropped
// terms are below 2^-24 of the product).  With two (NS = 2: x ~ hi + mid, 16
// bits), three MMAs: hi*hi + hi*mid + mid*hi (dropped terms below 2^-16).  The
// slices of an operand are the z-planes of one row-major buffer [3][rows][ld],
// read by TMA K-major (32 values of k per stage row, 64-byte swizzle; three
// stages of all six tiles in shared memory for NS = 3, four of four for NS = 2).
//
// Accumulation.  The products the K-FAC step multiplies cancel heavily (the
// preconditioner has gain up to 1/gamma on directions the gradient does not
// occupy: |grad| |inv_a| can be 6e3 times |grad inv_a|).  The tensor-core
// accumulator does not round to nearest, and its error grows with the number
// of accumulations, so every twelve MMAs (two 16-wide k-steps for NS = 3,
// four for NS = 2) go to a fresh TMEM accumulator (two, ping-pong) and the
// epilogue warps add them into fp32 registers with round-to-nearest: the
// result keeps close to the accuracy of an fp32 FMA loop.
//
// Kernel roles (320 threads, one CTA per SM, persistent over 128 x 256 tiles):
//   warp 0: TMA producer; warp 1: TMEM allocation + MMA issuer;
//   warps 2-9: epilogue; warp w reads TMEM lanes 32*(w%4).. and columns
//   128*((w-2)/4) .. +127 of the tile.  The epilogue writes fp32 C, or C split
//   again into three bf16 slices so one GEMM feeds the next directly.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_tc.h"
#include "launch.h"
#include "split.cuh"

namespace kfac {

constexpr int kGtBK = 32;
constexpr int kGtA = 128 * kGtBK * 2;  // one slice of the A tile (8 KB)
constexpr int kGtB = 256 * kGtBK * 2;  // one slice of the B tile (16 KB)
constexpr int kGtThreads = 320;
constexpr int kGtEpiWarps = 8;

template <int NS>
struct GtCfg {
  static constexpr int stage = NS * (kGtA + kGtB);
  static constexpr int stages = NS == 3 ? 3 : 4;
  static constexpr int smem = stages * stage + 1024 + 256;
  // 16-wide k-steps accumulated in one TMEM accumulator between two drains
  // into the epilogue's round-to-nearest fp32 sums (twelve MMAs either way)
  static constexpr int drain = NS == 3 ? 2 : 8;
};

struct GtParams {
  CUtensorMap mapA[kGtMaxProbs];
  CUtensorMap mapB[kGtMaxProbs];
  GtProb probs[kGtMaxProbs];
  const int* flags;
  long long total_tiles;
  int* status;
  int n_probs;
};

// a tile of a problem switched off by its flag is skipped by every role alike
__device__ __forceinline__ bool gt_skip(const GtParams& prm, int prob) {
  const int f = prm.probs[prob].flag_idx;
  return prm.flags != nullptr && f >= 0 && prm.flags[f] == 0;
}

struct GtTile {
  int prob, m0, n0, n_mma, K;
};

// w[r][c] = w[r][c] - lr * v, one rounding (the weight step of a row segment
// of n <= 32 values; every index below is static, so v stays in registers)
__device__ __forceinline__ void gt_weight_step(float* w, float lr, const float (&v)[32], int n) {
  if (n == 32) {
#pragma unroll
    for (int t = 0; t < 32; t += 4) {
      float4 x = *reinterpret_cast<const float4*>(w + t);
      x.x = __fmaf_rn(-lr, v[t], x.x);
      x.y = __fmaf_rn(-lr, v[t + 1], x.y);
      x.z = __fmaf_rn(-lr, v[t + 2], x.z);
      x.w = __fmaf_rn(-lr, v[t + 3], x.w);
      *reinterpret_cast<float4*>(w + t) = x;
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (t < n) w[t] = __fmaf_rn(-lr, v[t], w[t]);
  }
}

// tile u -> (problem, m0, n0): binary search over the problems, 32-bit
// arithmetic inside one (every role decodes every tile).  With CTA pairs (MC)
// a work item is two vertically adjacent tiles; CTA `rank` of the pair takes
// rows m0 + 128 * rank.
template <bool MC>
__device__ __forceinline__ GtTile gt_decode(const GtParams& prm, long long u, uint32_t rank) {
  int lo = 0, hi = prm.n_probs;  // largest pi with tile_begin <= u
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (prm.probs[mid].tile_begin <= u)
      lo = mid;
    else
      hi = mid;
  }
  const int pi = lo;
  const GtProb& p = prm.probs[pi];
  const int t = (int)(u - p.tile_begin);
  GtTile r;
  r.prob = pi;
  r.m0 = (t / p.tiles_n) * (MC ? 256 : 128) + (int)rank * 128;
  r.n0 = (t - (t / p.tiles_n) * p.tiles_n) * 256;
  r.n_mma = (min(256, p.N - r.n0) + 15) / 16 * 16;
  r.K = p.K;
  return r;
}

// K-major shared-memory descriptor, 64-byte swizzle: rows of 64 B, 8-row
// groups 512 B apart (layout type 4 at bits 61..63).
__device__ __forceinline__ uint64_t gt_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;
  return d;
}

// MC: CTA pairs (clusters of two) on vertically adjacent tiles share the B
// tile: each CTA loads one 128-row half of it with a TMA multicast into both
// CTAs' shared memory, so an SM reads 128 + 128 operand rows per k instead of
// 128 + 256.  A stage is refilled only when both CTAs' MMAs have released it
// (each commit arrives on the empty barriers of both CTAs).
template <int NS, bool MC>
__global__ void __launch_bounds__(kGtThreads, 1) gemm_tc_kernel(const __grid_constant__ GtParams prm) {
  using Cfg = GtCfg<NS>;
  constexpr int kGtStages = Cfg::stages;
  constexpr int kGtStage = Cfg::stage;
  constexpr int kGtDrain = Cfg::drain;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGtStages * kGtStage);
  uint64_t* empty = full + kGtStages;
  uint64_t* acc_full = empty + kGtStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (prm.flags != nullptr) {
    // a re-run over the flagged problems: nothing to do when none is flagged
    // (the same answer in every CTA, so whole clusters leave together)
    bool any = false;
    for (int i = 0; i < prm.n_probs && !any; ++i) {
      const int f = prm.probs[i].flag_idx;
      any = f < 0 || prm.flags[f] != 0;
    }
    if (!any) return;
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MC ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kGtEpiWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc_alloc(tmem_slot, 512);
  tc_fence_before();
  if (MC)
    cluster_sync();  // the partner's barriers exist before any multicast reaches them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t rank = MC ? cluster_ctarank() : 0u;
  const long long item0 = MC ? blockIdx.x / 2 : blockIdx.x;
  const long long items_step = MC ? gridDim.x / 2 : gridDim.x;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (long long u = item0; u < prm.total_tiles && !*abort_flag; u += items_step) {
        const GtTile tl = gt_decode<MC>(prm, u, rank);
        if (gt_skip(prm, tl.prob)) continue;
        const CUtensorMap* ma = &prm.mapA[tl.prob];
        const CUtensorMap* mb = &prm.mapB[tl.prob];
        const int nk = (tl.K + kGtBK - 1) / kGtBK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, prm.status)) break;
          uint8_t* s0 = smem + stage * kGtStage;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)kGtStage);
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            tma_load_3d(s0 + s * kGtA, ma, kb * kGtBK, tl.m0, s, &full[stage]);
            if (MC)  // this CTA's half of B (rows n0 + 128 rank ..), into both CTAs
              tma_load_3d_mc(s0 + NS * kGtA + s * kGtB + rank * (kGtB / 2), mb, kb * kGtBK,
                             tl.n0 + 128 * (int)rank, s, &full[stage], (uint16_t)0x3);
            else
              tma_load_3d(s0 + NS * kGtA + s * kGtB, mb, kb * kGtBK, tl.n0, s, &full[stage]);
          }
          if (++stage == kGtStages) {
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
      for (long long u = item0; u < prm.total_tiles && ok; u += items_step) {
        const GtTile tl = gt_decode<MC>(prm, u, rank);
        if (gt_skip(prm, tl.prob)) continue;
        const uint32_t idesc = idesc_bf16_f32(tl.n_mma, false, false);
        const int nk = (tl.K + kGtBK - 1) / kGtBK;
        const int n16 = nk * (kGtBK / 16);  // 16-wide k-steps of the tile
        int st16 = 0;
        for (int kb = 0; kb < nk && ok; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, prm.status)) {
            ok = false;
            break;
          }
          const uint32_t a0 = smem_u32(smem + stage * kGtStage);
          const uint32_t b0 = a0 + NS * kGtA;
#pragma unroll
          for (int kk = 0; kk < kGtBK / 16; ++kk, ++st16) {
            const bool gfirst = st16 % kGtDrain == 0;
            const bool glast = st16 % kGtDrain == kGtDrain - 1 || st16 == n16 - 1;
            if (gfirst) {
              if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, prm.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d_tmem = tmem_base + acc * 256;
            const uint32_t off = kk * 32;  // 16 values of k = 32 bytes along the swizzled row
            uint64_t da[NS], db[NS];
#pragma unroll
            for (int s = 0; s < NS; ++s) {
              da[s] = gt_desc(a0 + s * kGtA + off);
              db[s] = gt_desc(b0 + s * kGtB + off);
            }
            tc_mma_bf16(d_tmem, da[0], db[0], idesc, gfirst ? 0u : 1u);
            tc_mma_bf16(d_tmem, da[0], db[1], idesc, 1u);
            tc_mma_bf16(d_tmem, da[1], db[0], idesc, 1u);
            if (NS == 3) {
              tc_mma_bf16(d_tmem, da[0], db[NS - 1], idesc, 1u);
              tc_mma_bf16(d_tmem, da[NS - 1], db[0], idesc, 1u);
              tc_mma_bf16(d_tmem, da[1], db[1], idesc, 1u);
            }
            if (glast) {
              tc_commit(&acc_full[acc]);
              acc ^= 1;
              if (acc == 0) acc_phase ^= 1;
            }
          }
          if (MC)
            tc_commit_mc(&empty[stage], (uint16_t)0x3);
          else
            tc_commit(&empty[stage]);
          if (++stage == kGtStages) {
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
    const int q = warp & 3;           // TMEM lane quarter
    const int h = e / 4;              // column half of the 256-wide tile
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    for (long long u = item0; u < prm.total_tiles && ok; u += items_step) {
      const GtTile tl = gt_decode<MC>(prm, u, rank);
      if (gt_skip(prm, tl.prob)) continue;
      const GtProb& pr = prm.probs[tl.prob];
      const int nsteps = ((tl.K + kGtBK - 1) / kGtBK * (kGtBK / 16) + kGtDrain - 1) / kGtDrain;
      float run[128];
#pragma unroll
      for (int t = 0; t < 128; ++t) run[t] = 0.f;
      for (int st = 0; st < nsteps; ++st) {
        if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, prm.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256 + h * 128;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t v[32];
          tc_ld_32x32b_x32(base + g * 32, v);
          tc_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) run[g * 32 + t] += __uint_as_float(v[t]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) break;
      const int r = tl.m0 + q * 32 + lane;
      if (r < pr.M) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int col0 = tl.n0 + h * 128 + g * 32;
          if (col0 >= pr.N) continue;
          const bool fullc = col0 + 32 <= pr.N;
          if (!pr.out_split) {
            float* dst = static_cast<float*>(pr.out) + (long long)r * pr.ldc + col0;
            if (fullc) {
#pragma unroll
              for (int t = 0; t < 32; t += 4)
                *reinterpret_cast<float4*>(dst + t) =
                    make_float4(run[g * 32 + t] * pr.alpha, run[g * 32 + t + 1] * pr.alpha,
                                run[g * 32 + t + 2] * pr.alpha, run[g * 32 + t + 3] * pr.alpha);
            } else {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (col0 + t < pr.N) dst[t] = run[g * 32 + t] * pr.alpha;
            }
            if (pr.w != nullptr) {
              float v[32];
#pragma unroll
              for (int t = 0; t < 32; ++t) v[t] = run[g * 32 + t] * pr.alpha;
              gt_weight_step(pr.w + (long long)r * pr.ldw + col0, pr.lr, v, fullc ? 32 : pr.N - col0);
            }
          } else {
            uint16_t* dst = static_cast<uint16_t*>(pr.out) + (long long)r * pr.ldc + col0;
            if (fullc) {
#pragma unroll
              for (int t = 0; t < 32; t += 8) {
                float x8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) x8[k] = run[g * 32 + t + k] * pr.alpha;
                split8_store<NS>(x8, dst + t, pr.out_slice_stride);
              }
            } else {
#pragma unroll
              for (int t = 0; t < 32; ++t)
                if (col0 + t < pr.N) {
                  __nv_bfloat16 s[kSlices];
                  split_value(run[g * 32 + t] * pr.alpha, s);
#pragma unroll
                  for (int k = 0; k < NS; ++k)
                    dst[t + k * pr.out_slice_stride] = *reinterpret_cast<uint16_t*>(&s[k]);
                }
            }
          }
        }
      }
    }
  }
  if (MC)
    cluster_sync();  // no multicast or remote arrival is still headed for this CTA
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ fp32 -> bf16 slices
constexpr int kSplitSeg = 256;  // columns of one warp unit (32 lanes x 8)
// Two shapes of the split: eight warps per block over a grid of eight blocks
// per SM (the split running alone), or four warps per block with one block
// per chunk, small enough (128 threads, 8 K registers) to run beside a
// preconditioning GEMM block on the same SM.  A block iteration takes a chunk
// of kSplitUnits warp units per warp.
constexpr int kSplitUnits = 8;
__host__ __device__ constexpr int split_chunk(int nw) { return nw * kSplitUnits; }

// p[k] = sum_e z_k[c0 + e] x[e] for the eight probes z_k of gemm_tc.h
// (c0 a multiple of 8; bit offset `shift`)
__device__ __forceinline__ void probe8(const float (&x)[8], long long c0, int shift, float (&p)[8]) {
  const uint32_t hh = probe_hash((uint32_t)(c0 >> 3)), h = hh >> shift;
  const int t = probe_class_offset(hh, shift);
#pragma unroll
  for (int e = 0; e < 8; ++e) p[e] = ((h >> e) & 1u) ? -x[e] : x[e];
  // 8-point Walsh-Hadamard transform: p[k] = sum_e (-1)^popcount(k & e) p[e]
#pragma unroll
  for (int len = 1; len < 8; len <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if ((e & len) == 0) {
        const float a = p[e], b = p[e + len];
        p[e] = a + b;
        p[e + len] = a - b;
      }
#pragma unroll
  for (int k = 0; k < 8; ++k) p[k] *= hadamard8(k, t);  // the class offset t
}

template <int NP, int NW>
__global__ void __launch_bounds__(NW * 32, 32 / NW) split_kernel(const __grid_constant__ SplitParams prm) {
  // warp unit = 256 consecutive columns of one row (8 per lane); chunks of
  // split_chunk(NW) units never straddle two matrices, so the matrix lookup is
  // block-uniform.  Each warp fetches its next unit's row segment while it
  // slices the current one.
  if (prm.flags != nullptr) {  // a re-run over the flagged matrices: none flagged, nothing to do
    bool any = false;
    for (int i = 0; i < prm.n && !any; ++i) {
      const int f = prm.items[i].flag_idx;
      any = f < 0 || prm.flags[f] != 0;
    }
    if (!any) return;
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (long long ch = blockIdx.x; ch < prm.total_items; ch += gridDim.x) {
    int lo = 0, hi = prm.n;  // matrix with item_begin (in chunks) <= ch
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prm.items[mid].item_begin <= ch)
        lo = mid;
      else
        hi = mid;
    }
    const SplitItem& it = prm.items[lo];
    if (prm.flags != nullptr && it.flag_idx >= 0 && prm.flags[it.flag_idx] == 0) continue;
    const long long segs = (it.cols + kSplitSeg - 1) / kSplitSeg;
    const long long work = it.rows * segs;
    const long long w0 = (ch - it.item_begin) * split_chunk(NW);
    const long long w_end = w0 + split_chunk(NW) < work ? w0 + split_chunk(NW) : work;
    // the lane's 8 values of unit u (zero past the row's end)
    auto fetch = [&](long long u, float (&x)[8]) {
      const long long r = u / segs;
      const long long c0 = (u - r * segs) * kSplitSeg + lane * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
      if (c0 < it.cols) {
        const float* src = it.src + r * it.ld_src + c0;
        if (c0 + 8 <= it.cols) {
          const float4 a = *reinterpret_cast<const float4*>(src);
          const float4 b = *reinterpret_cast<const float4*>(src + 4);
          x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
          x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = (c0 + e < it.cols) ? src[e] : 0.f;
        }
      }
    };
    long long unit = w0 + warp;
    float xn[8];
    if (unit < w_end) fetch(unit, xn);
    for (; unit < w_end; unit += NW) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = xn[e];
      if (unit + NW < w_end) fetch(unit + NW, xn);
      const long long r = unit / segs;
      const long long c0 = (unit - r * segs) * kSplitSeg + lane * 8;
      if (c0 < it.cols) split8_store<NP>(x, it.dst + r * it.ld_dst + c0, it.slice_stride);
      if (it.probe != nullptr) {  // warp-uniform
        float p[8];
        probe8(x, c0, it.probe_shift, p);
        // reduce-scatter over the warp: offsets 16, 8, 4 halve the values
        // held, offsets 2 and 1 complete the sum; lane 4k + j then holds
        // probe k's sum over the unit
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool up = lane & 16;
          const float send = up ? p[i] : p[i + 4], keep = up ? p[i + 4] : p[i];
          p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const bool up = lane & 8;
          const float send = up ? p[i] : p[i + 2], keep = up ? p[i + 2] : p[i];
          p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        {
          const bool up = lane & 4;
          const float send = up ? p[0] : p[1], keep = up ? p[1] : p[0];
          p[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        p[0] += __shfl_xor_sync(0xffffffffu, p[0], 2);
        p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
        if ((lane & 3) == 0) atomicAdd(it.probe + r * kProbeN + (lane >> 2), p[0]);
      }
    }
  }
}

// ------------------------------------------------------------------ host side
// Slices of one operand: [3][rows][ld] bf16, K = inner extent.
static bool encode_slices(EncodeTiledFn enc, CUtensorMap* map, const uint16_t* base, long long rows, long long K,
                          long long ld, int box_rows) {
  cuuint64_t gdim[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)kSlices};
  cuuint64_t gstride[2] = {(cuuint64_t)ld * 2, (cuuint64_t)(rows * ld * 2)};
  cuuint32_t box[3] = {(cuuint32_t)kGtBK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), gdim, gstride, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_split(const SplitItem* items, int n, int planes, const int* flags, cudaStream_t stream, bool compact) {
  if (planes != 2 && planes != 3) return KFAC_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  const int nw = compact ? 4 : 8;
  for (int base = 0; base < n; base += kSplitMax) {
    const int cnt = n - base < kSplitMax ? n - base : kSplitMax;
    SplitParams prm;
    memset(&prm, 0, sizeof(prm));
    long long total = 0;
    for (int i = 0; i < cnt; ++i) {
      prm.items[i] = items[base + i];
      prm.items[i].item_begin = total;  // in chunks of split_chunk(nw) warp units
      const long long work = prm.items[i].rows * ((prm.items[i].cols + kSplitSeg - 1) / kSplitSeg);
      total += (work + split_chunk(nw) - 1) / split_chunk(nw);
    }
    prm.n = cnt;
    prm.flags = flags;
    prm.planes = planes;
    prm.total_items = total;
    if (total == 0) continue;
    if (compact) {  // one block per chunk: blocks come and go beside the GEMM's
      const unsigned grid = (unsigned)total;
      if (planes == 3)
        split_kernel<3, 4><<<grid, 128, 0, stream>>>(prm);
      else
        split_kernel<2, 4><<<grid, 128, 0, stream>>>(prm);
    } else {
      const long long cap = (long long)sms * 8;
      const unsigned grid = (unsigned)(total < cap ? total : cap);
      if (planes == 3)
        split_kernel<3, 8><<<grid, 256, 0, stream>>>(prm);
      else
        split_kernel<2, 8><<<grid, 256, 0, stream>>>(prm);
    }
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

int launch_gemm_tc(const GtOperand* ops_in, int n, int ns, const int* flags, cudaStream_t stream, bool pairs) {
  // longest K first: tiles are dealt round-robin to a persistent grid
  GtOperand* ops = new GtOperand[n > 0 ? n : 1];
  std::copy(ops_in, ops_in + n, ops);
  std::stable_sort(ops, ops + n, [](const GtOperand& x, const GtOperand& y) { return x.K > y.K; });
  const int rc = launch_gemm_tc_sorted(ops, n, ns, flags, stream, pairs);
  delete[] ops;
  return rc;
}

template <int NS, bool MC>
static int launch_gemm_kernel(const GtParams& prm, int grid, cudaStream_t stream, double work) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kGtThreads);
  cfg.dynamicSmemBytes = GtCfg<NS>::smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = MC ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfMark pm;
  prof_begin(stream, pm);
  if (cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NS, MC>, prm) != cudaSuccess) return KFAC_ERR_CUDA;
  prof_end(NS == 2 ? KFAC_K_GEMM16 : KFAC_K_GEMM24, stream, pm, work);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA;
}

int launch_gemm_tc_sorted(const GtOperand* ops, int n, int ns, const int* flags, cudaStream_t stream, bool pairs) {
  if (ns != 2 && ns != 3) return KFAC_ERR_INVALID_ARG;
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return KFAC_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms < 2) return KFAC_ERR_CUDA;
  const void* kern = ns == 3 ? (pairs ? (const void*)gemm_tc_kernel<3, true> : (const void*)gemm_tc_kernel<3, false>)
                             : (pairs ? (const void*)gemm_tc_kernel<2, true> : (const void*)gemm_tc_kernel<2, false>);
  const int smem = ns == 3 ? GtCfg<3>::smem : GtCfg<2>::smem;
  if (!ensure_smem_attr(dev, kern, smem)) return KFAC_ERR_CUDA;
  int* status = device_status_ptr();
  if (!status) return KFAC_ERR_CUDA;
  GtParams* prm = new GtParams;
  int rc = KFAC_OK;
  for (int base = 0; base < n && rc == KFAC_OK; base += kGtMaxProbs) {
    const int cnt = n - base < kGtMaxProbs ? n - base : kGtMaxProbs;
    memset(prm, 0, sizeof(GtParams));
    long long tiles = 0;
    for (int i = 0; i < cnt && rc == KFAC_OK; ++i) {
      const GtOperand& o = ops[base + i];
      if (!encode_slices(enc, &prm->mapA[i], o.a, o.M, o.K, o.lda, 128) ||
          !encode_slices(enc, &prm->mapB[i], o.b, o.N, o.K, o.ldb, pairs ? 128 : 256)) {
        rc = KFAC_ERR_INVALID_ARG;
        break;
      }
      GtProb& p = prm->probs[i];
      p.out = o.out;
      p.ldc = o.ldc;
      p.out_slice_stride = o.out_slice_stride;
      p.M = (int)o.M;
      p.N = (int)o.N;
      p.K = (int)o.K;
      p.tiles_n = (int)((o.N + 255) / 256);
      p.out_split = o.out_split;
      p.flag_idx = flags != nullptr ? o.flag_idx : -1;
      p.alpha = o.alpha;
      p.w = o.w;
      p.ldw = o.ldw;
      p.lr = o.lr;
      p.tile_begin = tiles;
      const long long tiles_m = (o.M + 127) / 128;
      tiles += (pairs ? (tiles_m + 1) / 2 : tiles_m) * p.tiles_n;  // work items (tile pairs with `pairs`)
    }
    if (rc != KFAC_OK) break;
    // work of the launch (2 M N K per problem); unknown when flags pick the problems
    double work = 0.0;
    if (flags == nullptr)
      for (int i = 0; i < cnt; ++i) work += 2.0 * (double)ops[base + i].M * ops[base + i].N * ops[base + i].K;
    prm->n_probs = cnt;
    prm->flags = flags;
    prm->total_tiles = tiles;
    prm->status = status;
    if (tiles > 0) {
      if (pairs) {
        const long long clusters = tiles < sms / 2 ? tiles : sms / 2;
        const int grid = (int)(2 * clusters);
        rc = ns == 3 ? launch_gemm_kernel<3, true>(*prm, grid, stream, work)
                     : launch_gemm_kernel<2, true>(*prm, grid, stream, work);
      } else {
        const int grid = (int)(tiles < sms ? tiles : sms);
        rc = ns == 3 ? launch_gemm_kernel<3, false>(*prm, grid, stream, work)
                     : launch_gemm_kernel<2, false>(*prm, grid, stream, work);
      }
    }
  }
  delete prm;
  return rc;
}

}  // namespace kfac
