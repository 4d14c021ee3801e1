// Split-bf16 NT GEMM on tcgen05 tensor cores, grouped over many problems:
//
//     C[m, n] = alpha * sum_k A[m, k] B[n, k]        (A: M x K, B: N x K)
//
// Every fp32 operand x is carried as NS bf16 slices whose sum is x:
//   NS = 2: x = hi + lo (16 significant bits); products hi*hi + hi*lo + lo*hi;
//   NS = 3: x = hi + mid + lo (24 bits, all of fp32); products hi*hi + hi*mid +
//           mid*hi + hi*lo + lo*hi + mid*mid (the dropped terms are below 2^-24
//           of the product).
// All products of a tile go into one fp32 TMEM accumulator.  The slices of an
// operand are the z-planes of one row-major buffer [NS][rows][ld], read by TMA
// K-major with a swizzle as wide as one stage row (NS = 2: 64 values of k,
// 128-byte swizzle; NS = 3: 32 values of k, 64-byte swizzle, so that three
// stages of all six tiles fit in shared memory).
//
// Kernel roles (192 threads, one CTA per SM, persistent over 128 x 256 tiles):
//   warp 0: TMA producer; warp 1: TMEM allocation + MMA issuer;
//   warps 2-5: epilogue (fp32 C, or C split again into NS bf16 slices so one
//   GEMM feeds the next directly).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_tc.h"
#include "launch.h"

namespace kfac {

template <int NS>
struct GtCfg;
template <>
struct GtCfg<2> {
  static constexpr int BK = 64, STAGES = 2, SWZ = 2 /*128 B*/, ROWB = 128, NPROD = 3;
};
template <>
struct GtCfg<3> {
  static constexpr int BK = 32, STAGES = 3, SWZ = 4 /*64 B*/, ROWB = 64, NPROD = 6;
};
template <int NS>
struct GtLayout {
  static constexpr int BK = GtCfg<NS>::BK;
  static constexpr int A = 128 * BK * 2;  // one slice of the A tile
  static constexpr int B = 256 * BK * 2;  // one slice of the B tile
  static constexpr int STAGE = NS * (A + B);
  static constexpr int SMEM = GtCfg<NS>::STAGES * STAGE + 1024 + 256;
};

struct GtParams {
  CUtensorMap mapA[kGtMaxProbs];
  CUtensorMap mapB[kGtMaxProbs];
  GtProb probs[kGtMaxProbs];
  long long total_tiles;
  int* status;
  int n_probs;
};

struct GtTile {
  int prob, m0, n0, n_mma, K;
};

__device__ __forceinline__ GtTile gt_decode(const GtParams& prm, long long u) {
  int pi = 0;
  while (pi + 1 < prm.n_probs && prm.probs[pi + 1].tile_begin <= u) ++pi;
  const GtProb& p = prm.probs[pi];
  const long long t = u - p.tile_begin;
  GtTile r;
  r.prob = pi;
  r.m0 = (int)(t / p.tiles_n) * 128;
  r.n0 = (int)(t % p.tiles_n) * 256;
  r.n_mma = (min(256, p.N - r.n0) + 15) / 16 * 16;
  r.K = p.K;
  return r;
}

// K-major shared-memory descriptor for the NS configuration (SBO = 8 rows).
template <int NS>
__device__ __forceinline__ uint64_t gt_desc(uint32_t saddr) {
  constexpr int ROWB = GtCfg<NS>::ROWB;
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)((8 * ROWB) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)GtCfg<NS>::SWZ << 61;
  return d;
}

// x -> NS bf16 slices (each slice carries the remainder of the previous ones)
template <int NS>
__device__ __forceinline__ void split_value(float x, __nv_bfloat16 (&s)[NS]) {
  float r = x;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    s[k] = __float2bfloat16_rn(r);
    r = r - __bfloat162float(s[k]);
  }
}

template <int NS>
__device__ __forceinline__ void split8_store(const float (&x)[8], uint16_t* dst, long long slice_stride) {
  uint32_t w[NS][4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat16 a[NS], b[NS];
    split_value<NS>(x[2 * e], a);
    split_value<NS>(x[2 * e + 1], b);
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      __nv_bfloat162 p;
      p.x = a[k];
      p.y = b[k];
      w[k][e] = *reinterpret_cast<const uint32_t*>(&p);
    }
  }
#pragma unroll
  for (int k = 0; k < NS; ++k)
    *reinterpret_cast<uint4*>(dst + k * slice_stride) = make_uint4(w[k][0], w[k][1], w[k][2], w[k][3]);
}

template <int NS>
__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ GtParams prm) {
  using Lay = GtLayout<NS>;
  constexpr int STAGES = GtCfg<NS>::STAGES;
  constexpr int BK = Lay::BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Lay::STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);
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
      for (long long u = blockIdx.x; u < prm.total_tiles && !*abort_flag; u += gridDim.x) {
        const GtTile tl = gt_decode(prm, u);
        const CUtensorMap* ma = &prm.mapA[tl.prob];
        const CUtensorMap* mb = &prm.mapB[tl.prob];
        const int nk = (tl.K + BK - 1) / BK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, prm.status)) break;
          uint8_t* s0 = smem + stage * Lay::STAGE;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)Lay::STAGE);
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            tma_load_3d(s0 + s * Lay::A, ma, kb * BK, tl.m0, s, &full[stage]);
            tma_load_3d(s0 + NS * Lay::A + s * Lay::B, mb, kb * BK, tl.n0, s, &full[stage]);
          }
          if (++stage == STAGES) {
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
      for (long long u = blockIdx.x; u < prm.total_tiles && ok; u += gridDim.x) {
        const GtTile tl = gt_decode(prm, u);
        const uint32_t idesc = idesc_bf16_f32(tl.n_mma, false, false);
        const int nk = (tl.K + BK - 1) / BK;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, prm.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 256;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, prm.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * Lay::STAGE);
          const uint32_t b0 = a0 + NS * Lay::A;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // 16 values of k = 32 bytes along the swizzled row
            const uint32_t off = kk * 32;
            uint64_t da[NS], db[NS];
#pragma unroll
            for (int s = 0; s < NS; ++s) {
              da[s] = gt_desc<NS>(a0 + s * Lay::A + off);
              db[s] = gt_desc<NS>(b0 + s * Lay::B + off);
            }
            tc_mma_bf16(d_tmem, da[0], db[0], idesc, (kb | kk) != 0);
            tc_mma_bf16(d_tmem, da[0], db[1], idesc, 1u);
            tc_mma_bf16(d_tmem, da[1], db[0], idesc, 1u);
            if constexpr (NS == 3) {
              tc_mma_bf16(d_tmem, da[0], db[2], idesc, 1u);
              tc_mma_bf16(d_tmem, da[2], db[0], idesc, 1u);
              tc_mma_bf16(d_tmem, da[1], db[1], idesc, 1u);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, prm.status);
    }
  } else {
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (long long u = blockIdx.x; u < prm.total_tiles; u += gridDim.x) {
      const GtTile tl = gt_decode(prm, u);
      const GtProb& pr = prm.probs[tl.prob];
      if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, prm.status)) break;
      tc_fence_after();
      const int r = tl.m0 + q * 32 + lane;
      const int nchunk = (tl.n_mma + 31) / 32;
      for (int c = 0; c < nchunk; ++c) {
        uint32_t v[32];
        tc_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256 + c * 32, v);
        tc_wait_ld();
        const int col0 = tl.n0 + c * 32;
        if (r >= pr.M || col0 >= pr.N) continue;
        const bool fullc = col0 + 32 <= pr.N;
        float o[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) o[t] = __uint_as_float(v[t]) * pr.alpha;
        if (!pr.out_split) {
          float* dst = static_cast<float*>(pr.out) + (long long)r * pr.ldc + col0;
          if (fullc) {
#pragma unroll
            for (int t = 0; t < 32; t += 4)
              *reinterpret_cast<float4*>(dst + t) = make_float4(o[t], o[t + 1], o[t + 2], o[t + 3]);
          } else {
            for (int t = 0; t < 32; ++t)
              if (col0 + t < pr.N) dst[t] = o[t];
          }
        } else {
          uint16_t* dst = static_cast<uint16_t*>(pr.out) + (long long)r * pr.ldc + col0;
          if (fullc) {
#pragma unroll
            for (int t = 0; t < 32; t += 8) {
              float x8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) x8[e] = o[t + e];
              split8_store<NS>(x8, dst + t, pr.out_slice_stride);
            }
          } else {
            for (int t = 0; t < 32; ++t)
              if (col0 + t < pr.N) {
                __nv_bfloat16 s[NS];
                split_value<NS>(o[t], s);
#pragma unroll
                for (int k = 0; k < NS; ++k) dst[t + k * pr.out_slice_stride] = *reinterpret_cast<uint16_t*>(&s[k]);
              }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ fp32 -> bf16 slices
template <int NS>
__global__ void __launch_bounds__(256) split_kernel(const __grid_constant__ SplitParams prm) {
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nth = (long long)gridDim.x * blockDim.x;
  // work item = 8 consecutive columns of one row
  for (long long g = tid; g < prm.total_items; g += nth) {
    int pi = 0;
    while (pi + 1 < prm.n && prm.items[pi + 1].item_begin <= g) ++pi;
    const SplitItem& it = prm.items[pi];
    const long long local = g - it.item_begin;
    const long long per_row = (it.cols + 7) / 8;
    const long long r = local / per_row;
    const long long c0 = (local % per_row) * 8;
    const float* src = it.src + r * it.ld_src + c0;
    float x[8];
    if (c0 + 8 <= it.cols) {
      const float4 a = *reinterpret_cast<const float4*>(src);
      const float4 b = *reinterpret_cast<const float4*>(src + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = (c0 + e < it.cols) ? src[e] : 0.f;
    }
    split8_store<NS>(x, it.dst + r * it.ld_dst + c0, it.slice_stride);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn gt_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Slices of one operand: [NS][rows][ld] bf16, K = inner extent.
static bool encode_slices(EncodeTiledFn enc, int NS, CUtensorMap* map, const uint16_t* base, long long rows,
                          long long K, long long ld, int box_rows) {
  const int bk = NS == 3 ? GtCfg<3>::BK : GtCfg<2>::BK;
  cuuint64_t gdim[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)NS};
  cuuint64_t gstride[2] = {(cuuint64_t)ld * 2, (cuuint64_t)(rows * ld * 2)};
  cuuint32_t box[3] = {(cuuint32_t)bk, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = NS == 3 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), gdim, gstride, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_split(const SplitItem* items, int n, int NS, cudaStream_t stream) {
  if (NS != 2 && NS != 3) return KFAC_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  for (int base = 0; base < n; base += kSplitMax) {
    const int cnt = n - base < kSplitMax ? n - base : kSplitMax;
    SplitParams prm;
    memset(&prm, 0, sizeof(prm));
    long long total = 0;
    for (int i = 0; i < cnt; ++i) {
      prm.items[i] = items[base + i];
      prm.items[i].item_begin = total;
      total += prm.items[i].rows * ((prm.items[i].cols + 7) / 8);
    }
    prm.n = cnt;
    prm.total_items = total;
    if (total == 0) continue;
    const long long want = (total + 255) / 256, cap = (long long)sms * 16;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    if (NS == 3)
      split_kernel<3><<<grid, 256, 0, stream>>>(prm);
    else
      split_kernel<2><<<grid, 256, 0, stream>>>(prm);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

int launch_gemm_tc(const GtOperand* ops_in, int n, int NS, cudaStream_t stream) {
  // longest K first: tiles are dealt round-robin to a persistent grid
  GtOperand* ops = new GtOperand[n > 0 ? n : 1];
  std::copy(ops_in, ops_in + n, ops);
  std::stable_sort(ops, ops + n, [](const GtOperand& x, const GtOperand& y) { return x.K > y.K; });
  const int rc = launch_gemm_tc_sorted(ops, n, NS, stream);
  delete[] ops;
  return rc;
}

int launch_gemm_tc_sorted(const GtOperand* ops, int n, int NS, cudaStream_t stream) {
  if (NS != 2 && NS != 3) return KFAC_ERR_INVALID_ARG;
  EncodeTiledFn enc = gt_encode_fn();
  if (!enc) return KFAC_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  const void* fn = NS == 3 ? (const void*)gemm_tc_kernel<3> : (const void*)gemm_tc_kernel<2>;
  const int smem = NS == 3 ? GtLayout<3>::SMEM : GtLayout<2>::SMEM;
  if (!ensure_smem_attr(dev, fn, smem)) return KFAC_ERR_CUDA;
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
      if (!encode_slices(enc, NS, &prm->mapA[i], o.a, o.M, o.K, o.lda, 128) ||
          !encode_slices(enc, NS, &prm->mapB[i], o.b, o.N, o.K, o.ldb, 256)) {
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
      p.alpha = o.alpha;
      p.tile_begin = tiles;
      tiles += (long long)((o.M + 127) / 128) * p.tiles_n;
    }
    if (rc != KFAC_OK) break;
    prm->n_probs = cnt;
    prm->total_tiles = tiles;
    prm->status = status;
    if (tiles > 0) {
      const int grid = (int)(tiles < sms ? tiles : sms);
      if (NS == 3)
        gemm_tc_kernel<3><<<grid, 192, smem, stream>>>(*prm);
      else
        gemm_tc_kernel<2><<<grid, 192, smem, stream>>>(*prm);
      count_launch();
      if (cudaGetLastError() != cudaSuccess) rc = KFAC_ERR_CUDA;
    }
  }
  delete prm;
  return rc;
}

}  // namespace kfac
