// Kronecker factor A of a 3 x 3 convolution (stride 1, zero padding 1, with
// bias) formed straight from the layer's NHWC input activations: implicit
// im2col.  SPD-KFAC §II-B, Eq. (7) defines A from a layer's inputs; for a
// convolution the input of one output position is its 3 x 3 x C patch and a
// ones column carries the bias (the pages do not spell conv factors out; this
// is the plainest reading).  Per worker p (§II-C: local factors):
//
//     out[p] = scale * X_p^T X_p,   X_p = patch rows of worker p's images,
//     X[(b, h, w), (dh*3 + dw)*C + c] = x[b, h+dh-1, w+dw-1, c] (0 outside),
//     X[(b, h, w), 9C] = 1.
//
// The patch matrix (9 times the activations' bytes) is never written.
// Producer warps gather each 64-row x 64-column operand box from x with
// cp.async (16-byte copies; zero fill for the padding, for rows past the
// shard and for columns past d) straight into the 128-byte-swizzled MN-major
// layout a TMA load would give (row t of a box at t * 128, its 16-byte chunk
// j at chunk j ^ (t & 7)), which the tensor-core SYRK reads.  With C % 64 == 0
// a box holds 64 channels of one tap, so one box row is one 128-byte run of x.
//
// Kernel roles (288 threads, one CTA per SM, persistent over work units):
//   warps 0-3 producers: thread t owns row t / 2 of every box of a stage and
//             four of its eight 16-byte chunks.  Per stage it decodes its
//             row's position once, issues its copies as one cp.async group and
//             then releases the stage before (wait until one group is left in
//             flight, proxy fence, mbarrier arrival): two stages in flight;
//   warp 4    TMEM allocation and the MMA issuer (one thread);
//   warps 5-8 epilogue (factor_epilogue.cuh).
// Work units (tilemap.cuh), the two 128 x 256 TMEM accumulators, the K-chunked
// accumulation and the output staging are those of the linear-layer SYRK
// (factors.cu).  The CTAs work alone (a cp.async gather has no multicast), so
// a unit's columns left of its own row block are trimmed instead of computed.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "factor_epilogue.cuh"
#include "launch.h"
#include "tilemap.cuh"

namespace kfac {

constexpr int kCvBK = 64;                      // patch rows (k) per stage
constexpr int kCvStages = 4;
constexpr int kCvBox = 64 * kCvBK * 2;         // one 64-column x 64-row bf16 box: 8 KB
constexpr int kCvABytes = 2 * kCvBox;          // 128 columns
constexpr int kCvBBytes = 4 * kCvBox;          // up to 256 columns
constexpr int kCvStageBytes = kCvABytes + kCvBBytes;
constexpr int kCvOutBytes = 4 * 2 * kFeStageOut;
constexpr int kCvSmem = kCvStages * kCvStageBytes + kCvOutBytes + 1024 + 256;
constexpr int kCvChunkKB = 16;  // accumulator restarted every 1024 rows (as in factors.cu)
constexpr int kCvProducers = 128;
constexpr int kCvThreads = 288;
constexpr int kCvMaxProbs = 64;

// bf16 1.0 followed by seven zeros: the bias column's 16-byte chunk.
__device__ __align__(16) uint16_t kCvOnesChunk[8] = {0x3F80, 0, 0, 0, 0, 0, 0, 0};

struct CvProb {
  const uint16_t* x;  // NHWC activations of all P workers' images
  float* out;
  long long ld_out, stride_out, unit_begin;
  int d, C, H, W, rows_p, units_per_shard;
  float scale;
};

struct CvParams {  // 128-byte aligned through CUtensorMap
  CUtensorMap omaps[kCvMaxProbs];  // outputs {d, d, P} fp32, box 32 x 32, swizzled
  CvProb probs[kCvMaxProbs];
  long long total_units;
  int* status;
  int n_probs, mirror;
};

struct CvUnit {
  int prob, p, i, w;
  int j0;
  bool live;  // false: a stand-in of the tile map (no row block)
};

// Unit u -> (problem, shard, row block, columns), walking the problem table
// with a cursor as units only increase.  Columns left of the row block's
// diagonal tile are not stored, so they are not computed either.
__device__ __forceinline__ CvUnit cv_decode(const CvParams& prm, long long u, int& lo) {
  while (lo + 1 < prm.n_probs && prm.probs[lo + 1].unit_begin <= u) ++lo;
  const CvProb& pr = prm.probs[lo];
  const int local = (int)(u - pr.unit_begin);
  CvUnit r;
  r.prob = lo;
  r.p = local / pr.units_per_shard;
  factor_unit_fast(pr.d, local - r.p * pr.units_per_shard, r.i, r.j0, r.w);
  r.live = r.i * 128 < pr.d;
  if (r.live && r.j0 < r.i * 128) {
    r.w -= r.i * 128 - r.j0;
    r.j0 = r.i * 128;
  }
  return r;
}

// Copies of one box row: column box q (columns 64q .. 64q+63 of the patch
// matrix), this thread's chunks hc .. hc+3 into the swizzled row `dst_row`.
// `pos` is the row's output position (b*H + h)*W + w; rmask / cmask hold which
// of the rows h-1, h, h+1 and columns w-1, w, w+1 lie inside the image (0 for a
// row past the shard).
__device__ __forceinline__ void cv_gather_box(uint8_t* dst_row, int sw, int hc, int q, const CvProb& pr, int c64,
                                              int pos, uint32_t rmask, uint32_t cmask) {
  if (q < 9 * c64) {
    const int tap = q / c64;
    const int dh = tap / 3, dw = tap - 3 * dh;
    const bool in = ((rmask >> dh) & (cmask >> dw) & 1u) != 0;
    const uint16_t* src = pr.x;
    if (in)
      src += (long long)(pos + (dh - 1) * pr.W + (dw - 1)) * pr.C + (q - tap * c64) * 64 + hc * 8;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      cp_async16(dst_row + (((hc + jj) ^ sw) << 4), in ? src + jj * 8 : pr.x, in ? 16u : 0u);
  } else {
    // the bias column (first column of box 9C/64) and the columns past d
    const bool ones = q == 9 * c64 && hc == 0 && rmask != 0;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      cp_async16(dst_row + (((hc + jj) ^ sw) << 4), kCvOnesChunk, (ones && jj == 0) ? 16u : 0u);
  }
}

__global__ void __launch_bounds__(kCvThreads, 1) conv_factor_tc_kernel(const __grid_constant__ CvParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + kCvStages * kCvStageBytes;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + kCvOutBytes);
  uint64_t* empty = full + kCvStages;
  uint64_t* acc_full = empty + kCvStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kCvStages; ++s) {
      mbar_init(&full[s], kCvProducers);
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
  if (warp == 4) tc_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 4) {
    const int t = threadIdx.x >> 1, hc = (threadIdx.x & 1) * 4, sw = t & 7;
    uint32_t stage = 0, phase = 0, prev = 0;
    bool have_prev = false, ok = true;
    int cur = 0;
    for (long long u = blockIdx.x; u < prm.total_units && ok && !*abort_flag; u += gridDim.x) {
      const CvUnit un = cv_decode(prm, u, cur);
      if (!un.live) continue;
      const CvProb& pr = prm.probs[un.prob];
      const int nb = (un.w + 63) / 64;
      const int nk = (pr.rows_p + kCvBK - 1) / kCvBK;
      const int c64 = pr.C / 64, hw = pr.H * pr.W;
      const int qa = un.i * 2, qb = un.j0 / 64;
      const long long row0 = (long long)un.p * pr.rows_p;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, prm.status)) {
          ok = false;
          break;
        }
        const int kr = kb * kCvBK + t;
        int pos = 0;
        uint32_t rmask = 0, cmask = 0;
        if (kr < pr.rows_p) {
          pos = (int)(row0 + kr);
          const int s = pos % hw;
          const int h = s / pr.W, w = s - h * pr.W;
          rmask = (h > 0 ? 1u : 0u) | 2u | (h + 1 < pr.H ? 4u : 0u);
          cmask = (w > 0 ? 1u : 0u) | 2u | (w + 1 < pr.W ? 4u : 0u);
        }
        uint8_t* row = smem + stage * kCvStageBytes + t * 128;
        cv_gather_box(row, sw, hc, qa, pr, c64, pos, rmask, cmask);
        cv_gather_box(row + kCvBox, sw, hc, qa + 1, pr, c64, pos, rmask, cmask);
        for (int b = 0; b < nb; ++b)
          cv_gather_box(row + kCvABytes + b * kCvBox, sw, hc, qb + b, pr, c64, pos, rmask, cmask);
        cp_async_commit();
        if (have_prev) {
          cp_async_wait<1>();
          fence_proxy_async_smem();
          mbar_arrive(&full[prev]);
        }
        prev = stage;
        have_prev = true;
        if (++stage == kCvStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    cp_async_wait<0>();  // no copy is still headed for this CTA's shared memory
    if (have_prev) {
      fence_proxy_async_smem();
      mbar_arrive(&full[prev]);
    }
  } else if (warp == 4) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      int cur = 0;
      for (long long u = blockIdx.x; u < prm.total_units && ok; u += gridDim.x) {
        const CvUnit un = cv_decode(prm, u, cur);
        if (!un.live) continue;
        const CvProb& pr = prm.probs[un.prob];
        const int nb = (un.w + 63) / 64;
        const uint32_t idesc = idesc_bf16_f32(nb * 64, true, true);
        const int nk = (pr.rows_p + kCvBK - 1) / kCvBK;
        for (int kc = 0; kc < nk && ok; kc += kCvChunkKB) {
          const int kend = kc + kCvChunkKB < nk ? kc + kCvChunkKB : nk;
          if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, prm.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * 256;
          for (int kb = kc; kb < kend; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, prm.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + stage * kCvStageBytes);
            const uint32_t b0 = a0 + kCvABytes;
#pragma unroll
            for (int kk = 0; kk < kCvBK / 16; ++kk) {
              // 16 rows of k = two 8-row groups of 1024 B; 64-column boxes are kCvBox apart.
              const uint64_t ad = smem_desc_sw128(a0 + kk * 2048, kCvBox, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, kCvBox, 1024);
              tc_mma_bf16(d_tmem, ad, bd, idesc, (kb != kc || kk != 0) ? 1u : 0u);
            }
            tc_commit(&empty[stage]);
            if (++stage == kCvStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc_commit(&acc_full[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
      }
      // Every MMA issued above has completed once done_bar flips.
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, prm.status);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t acc = 0, acc_phase = 0;
    int obuf = 0;
    bool ok = true;
    int cur = 0;
    for (long long u = blockIdx.x; u < prm.total_units && ok; u += gridDim.x) {
      const CvUnit un = cv_decode(prm, u, cur);
      if (!un.live) continue;
      const CvProb& pr = prm.probs[un.prob];
      const int nk = (pr.rows_p + kCvBK - 1) / kCvBK;
      const int nchunks = (nk + kCvChunkKB - 1) / kCvChunkKB;
      const FeUnit fu{pr.out + (long long)un.p * pr.stride_out, &prm.omaps[un.prob], pr.ld_out, un.j0, pr.d,
                      un.i, un.w, un.p, pr.scale};
      for (int ch = 0; ch < nchunks; ++ch) {
        if (!mbar_wait(&acc_full[acc], acc_phase, abort_flag, prm.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        factor_epilogue_chunk(tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256, q, lane, fu, ch == 0,
                              ch == nchunks - 1, prm.mirror != 0, out_stage + q * 2 * kFeStageOut, obuf);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait<0>();  // all TMA stores of this warp complete before exit
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tc_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ host side
int launch_conv_factors(int n, const kfac_conv_factor_args* args, int P, int mirror, cudaStream_t stream) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return KFAC_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  if (!ensure_smem_attr(dev, (const void*)conv_factor_tc_kernel, kCvSmem)) return KFAC_ERR_CUDA;
  for (int base = 0; base < n; base += kCvMaxProbs) {
    const int cnt = n - base < kCvMaxProbs ? n - base : kCvMaxProbs;
    CvParams prm;
    memset(&prm, 0, sizeof(prm));
    long long units = 0, live = 0;
    double work = 0.0;  // algorithmic flops of the launch: 2 rows d(d+1)/2 per factor
    for (int k = 0; k < cnt; ++k) {
      const kfac_conv_factor_args& a = args[base + k];
      const long long d = 9 * a.C + 1;
      const long long rows_p = a.B / P * a.H * a.W;
      const long long so = P > 1 ? a.stride_out : d * a.ld_out;
      cuuint64_t odim[3] = {(cuuint64_t)d, (cuuint64_t)d, (cuuint64_t)P};
      cuuint64_t ostride[2] = {(cuuint64_t)a.ld_out * 4, (cuuint64_t)so * 4};
      cuuint32_t obox[3] = {32, 32, 1};
      cuuint32_t estr[3] = {1, 1, 1};
      const CUresult cr = enc(&prm.omaps[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.out, odim, ostride, obox, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (cr != CUDA_SUCCESS) return KFAC_ERR_INVALID_ARG;
      CvProb& pr = prm.probs[k];
      pr.x = static_cast<const uint16_t*>(a.x);
      pr.out = a.out;
      pr.ld_out = a.ld_out;
      pr.stride_out = a.stride_out;
      pr.d = (int)d;
      pr.C = (int)a.C;
      pr.H = (int)a.H;
      pr.W = (int)a.W;
      pr.rows_p = (int)rows_p;
      pr.units_per_shard = (int)factor_units(d);
      pr.unit_begin = units;
      pr.scale = a.scale;
      units += (long long)pr.units_per_shard * P;
      // with an odd number of row blocks one unit per shard is a stand-in
      live += (long long)P * (pr.units_per_shard - ((d + 127) / 128 & 1));
      work += 2.0 * (double)rows_p * P * (double)d * ((double)d + 1.0) / 2.0;
    }
    prm.n_probs = cnt;
    prm.mirror = mirror;
    prm.total_units = units;
    prm.status = device_status_ptr();
    if (!prm.status) return KFAC_ERR_CUDA;
    if (live == 0) continue;
    const int grid = (int)(live < sms ? live : sms);
    ProfMark pm;
    prof_begin(stream, pm);
    conv_factor_tc_kernel<<<grid, kCvThreads, kCvSmem, stream>>>(prm);
    prof_end(KFAC_K_CONV_SYRK, stream, pm, work);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

}  // namespace kfac
