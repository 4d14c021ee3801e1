// Split-bf16 NT GEMM on tcgen05 tensor cores, grouped over many problems:
//
//     C[m, n] = alpha * sum_k A[m, k] B[n, k]        (A: M x K, B: N x K)
//
// Every fp32 operand x is carried as two bf16 slices x = hi + lo with
// hi = bf16(x), lo = bf16(x - hi) (16 significant bits), and the three
// products hi*hi + hi*lo + lo*hi are accumulated in one fp32 TMEM accumulator
// (the dropped lo*lo term is below 2^-16 of the product).  The two slices of
// an operand are the z = 0 / 1 planes of one row-major buffer [2][rows][ld],
// read by TMA with the 128-byte swizzle (K-major, 64 values of k per row).
//
// Kernel roles (192 threads, one CTA per SM, persistent over 128 x 256 tiles):
//   warp 0: TMA producer, 2 stages of {A_hi, A_lo, B_hi, B_lo} (96 KB each);
//   warp 1: TMEM allocation + MMA issuer; warps 2-5: epilogue.
// The epilogue writes either fp32 C or C split again into bf16 hi/lo slices
// (so one GEMM can feed the next one directly).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_tc.h"
#include "launch.h"

namespace kfac {

constexpr int kGtBK = 64;
constexpr int kGtStages = 2;
constexpr int kGtABytes = 128 * kGtBK * 2;  // one slice of the A tile: 16 KB
constexpr int kGtBBytes = 256 * kGtBK * 2;  // one slice of the B tile: 32 KB
constexpr int kGtStageBytes = 2 * kGtABytes + 2 * kGtBBytes;
constexpr int kGtSmem = kGtStages * kGtStageBytes + 1024 + 256;

struct GtParams {
  CUtensorMap mapA[kGtMaxProbs];
  CUtensorMap mapB[kGtMaxProbs];
  GtProb probs[kGtMaxProbs];
  long long total_tiles;
  int* status;
  int n_probs;
};

struct GtTile {
  int prob, m0, n0, n_valid, n_mma, K;
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
  r.n_valid = min(256, p.N - r.n0);
  r.n_mma = (r.n_valid + 15) / 16 * 16;
  r.K = p.K;
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(192, 1) gemm_tc_kernel(const __grid_constant__ GtParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGtStages * kGtStageBytes);
  uint64_t* empty = full + kGtStages;
  uint64_t* acc_full = empty + kGtStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGtStages; ++s) {
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
        const int nk = (tl.K + kGtBK - 1) / kGtBK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, prm.status)) break;
          uint8_t* s0 = smem + stage * kGtStageBytes;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)kGtStageBytes);
          tma_load_3d(s0, ma, kb * kGtBK, tl.m0, 0, &full[stage]);
          tma_load_3d(s0 + kGtABytes, ma, kb * kGtBK, tl.m0, 1, &full[stage]);
          tma_load_3d(s0 + 2 * kGtABytes, mb, kb * kGtBK, tl.n0, 0, &full[stage]);
          tma_load_3d(s0 + 2 * kGtABytes + kGtBBytes, mb, kb * kGtBK, tl.n0, 1, &full[stage]);
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
      for (long long u = blockIdx.x; u < prm.total_tiles && ok; u += gridDim.x) {
        const GtTile tl = gt_decode(prm, u);
        const uint32_t idesc = idesc_bf16_f32(tl.n_mma, false, false);
        const int nk = (tl.K + kGtBK - 1) / kGtBK;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, prm.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 256;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, prm.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_hi = smem_u32(smem + stage * kGtStageBytes);
          const uint32_t a_lo = a_hi + kGtABytes;
          const uint32_t b_hi = a_hi + 2 * kGtABytes;
          const uint32_t b_lo = b_hi + kGtBBytes;
#pragma unroll
          for (int kk = 0; kk < kGtBK / 16; ++kk) {
            // K-major, 128-byte swizzle: 16 values of k = 32 bytes along the row;
            // 8-row groups are 1024 bytes apart.
            const uint32_t off = kk * 32;
            const uint64_t dah = smem_desc_sw128(a_hi + off, 16, 1024);
            const uint64_t dal = smem_desc_sw128(a_lo + off, 16, 1024);
            const uint64_t dbh = smem_desc_sw128(b_hi + off, 16, 1024);
            const uint64_t dbl = smem_desc_sw128(b_lo + off, 16, 1024);
            tc_mma_bf16(d_tmem, dah, dbh, idesc, (kb | kk) != 0);
            tc_mma_bf16(d_tmem, dah, dbl, idesc, 1u);
            tc_mma_bf16(d_tmem, dal, dbh, idesc, 1u);
          }
          tc_commit(&empty[stage]);
          if (++stage == kGtStages) {
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
      const int nchunk = tl.n_mma / 32 + ((tl.n_mma % 32) ? 1 : 0);
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
          uint16_t* hi = static_cast<uint16_t*>(pr.out) + (long long)r * pr.ldc + col0;
          uint16_t* lo = hi + pr.out_slice_stride;
          if (fullc) {
#pragma unroll
            for (int t = 0; t < 32; t += 8) {
              uint32_t h[4], l[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x0 = o[t + 2 * e], x1 = o[t + 2 * e + 1];
                const __nv_bfloat162 hb = __floats2bfloat162_rn(x0, x1);
                const float2 hf = __bfloat1622float2(hb);
                h[e] = *reinterpret_cast<const uint32_t*>(&hb);
                l[e] = pack_bf16x2(x0 - hf.x, x1 - hf.y);
              }
              *reinterpret_cast<uint4*>(hi + t) = make_uint4(h[0], h[1], h[2], h[3]);
              *reinterpret_cast<uint4*>(lo + t) = make_uint4(l[0], l[1], l[2], l[3]);
            }
          } else {
            for (int t = 0; t < 32; ++t)
              if (col0 + t < pr.N) {
                const __nv_bfloat16 hb = __float2bfloat16_rn(o[t]);
                const __nv_bfloat16 lb = __float2bfloat16_rn(o[t] - __bfloat162float(hb));
                hi[t] = *reinterpret_cast<const uint16_t*>(&hb);
                lo[t] = *reinterpret_cast<const uint16_t*>(&lb);
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

// ------------------------------------------------------------------ fp32 -> (hi, lo) bf16 slices
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
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      const float2 hf = __bfloat1622float2(hb);
      h[e] = *reinterpret_cast<const uint32_t*>(&hb);
      l[e] = pack_bf16x2(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
    }
    uint16_t* dst = it.dst + r * it.ld_dst + c0;
    *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(dst + it.slice_stride) = make_uint4(l[0], l[1], l[2], l[3]);
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

// Slices of one operand: [2][rows][ld] bf16, K = inner extent, box rows = box_rows.
static bool encode_slices(EncodeTiledFn enc, CUtensorMap* map, const uint16_t* base, long long rows, long long K,
                          long long ld, int box_rows) {
  cuuint64_t gdim[3] = {(cuuint64_t)K, (cuuint64_t)rows, 2};
  cuuint64_t gstride[2] = {(cuuint64_t)ld * 2, (cuuint64_t)(rows * ld * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), gdim, gstride, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_split(const SplitItem* items, int n, cudaStream_t stream) {
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
    split_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, stream>>>(prm);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

int launch_gemm_tc(const GtOperand* ops_in, int n, cudaStream_t stream) {
  // longest K first: tiles are dealt round-robin to a persistent grid
  GtOperand* ops = new GtOperand[n > 0 ? n : 1];
  std::copy(ops_in, ops_in + n, ops);
  std::stable_sort(ops, ops + n, [](const GtOperand& x, const GtOperand& y) { return x.K > y.K; });
  const int rc = launch_gemm_tc_sorted(ops, n, stream);
  delete[] ops;
  return rc;
}

int launch_gemm_tc_sorted(const GtOperand* ops, int n, cudaStream_t stream) {
  EncodeTiledFn enc = gt_encode_fn();
  if (!enc) return KFAC_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  if (!ensure_smem_attr(dev, (const void*)gemm_tc_kernel, kGtSmem)) return KFAC_ERR_CUDA;
  int* status = device_status_ptr();
  if (!status) return KFAC_ERR_CUDA;
  for (int base = 0; base < n; base += kGtMaxProbs) {
    const int cnt = n - base < kGtMaxProbs ? n - base : kGtMaxProbs;
    GtParams* prm = new GtParams;
    memset(prm, 0, sizeof(GtParams));
    long long tiles = 0;
    for (int i = 0; i < cnt; ++i) {
      const GtOperand& o = ops[base + i];
      if (!encode_slices(enc, &prm->mapA[i], o.a, o.M, o.K, o.lda, 128) ||
          !encode_slices(enc, &prm->mapB[i], o.b, o.N, o.K, o.ldb, 256)) {
        delete prm;
        return KFAC_ERR_INVALID_ARG;
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
    prm->n_probs = cnt;
    prm->total_tiles = tiles;
    prm->status = status;
    if (tiles > 0) {
      const int grid = (int)(tiles < sms ? tiles : sms);
      gemm_tc_kernel<<<grid, 192, kGtSmem, stream>>>(*prm);
      count_launch();
    }
    delete prm;
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

}  // namespace kfac
