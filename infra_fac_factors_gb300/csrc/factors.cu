// Kronecker factors of P emulated workers (SPD-KFAC §II-B, Eq. (7)/(8);
// §II-C: each worker p forms its local factor from its own rows):
//
//     out[p] = scale * x_p^T x_p,   x_p = rows [p*rows_p, (p+1)*rows_p) of x
//
// bf16 inputs: tcgen05 tensor cores.  The operand tiles are x[k0:k0+64,
// i0:i0+128] and x[k0:k0+64, j0:j0+N]; both are MN-major in shared memory
// (x is row-major, so the factor's row index m is the contiguous one), loaded
// by TMA with the 128-byte swizzle from a 3-D tensor map {d, rows_p, P}, so the
// tail of each worker's rows and of the columns reads as zero.
//
// Kernel roles (192 threads, one CTA per SM, persistent over work units):
//   warp 0   TMA producer (one thread), 4-stage shared-memory ring;
//   warp 1   TMEM allocation and the MMA issuer (one thread);
//   warps 2-5 epilogue: TMEM -> registers -> scale -> global fp32 stores.
// Two 128 x 256 fp32 accumulators in TMEM (all 512 columns) let the epilogue
// of one unit overlap the main loop of the next.
// CTA pairs (clusters of two) take the two row blocks of one pair-chunk of the
// tile map (tilemap.cuh): they share the column operand x[k, j0:j0+w], each
// CTA loading half of its 64-column boxes with a TMA multicast into both, so
// an SM reads 128 + 128 operand columns per k instead of 128 + 256.  A stage
// is refilled once both CTAs' MMAs have released it.
//
// fp32 inputs: exact fp32 products on CUDA cores (simt.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "factor_epilogue.cuh"
#include "conv_geom.cuh"
#include "launch.h"
#include "simt.cuh"
#include "tilemap.cuh"

namespace kfac {

// Device status word (KFAC_OK or KFAC_ERR_TIMEOUT) of this library.
__device__ int g_device_status = 0;

int* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

// ------------------------------------------------------------------ tcgen05 SYRK
constexpr int kSyBK = 64;                      // rows (k) per stage
constexpr int kSyStages = 4;
constexpr int kSyBox = 64 * kSyBK * 2;         // one 64-column x 64-row bf16 box: 8 KB
constexpr int kSyABytes = 2 * kSyBox;          // 128 columns
constexpr int kSyBBytes = 4 * kSyBox;          // up to 256 columns
constexpr int kSyStageBytes = kSyABytes + kSyBBytes;
constexpr int kSyMaxProbs = 96;
// Epilogue staging: per epilogue warp two 32 x 32 fp32 blocks (4 KB each,
// 128-byte swizzled), written to global memory by TMA stores.
constexpr int kSyOutBytes = 4 * 2 * kFeStageOut;
constexpr int kSySmem = kSyStages * kSyStageBytes + kSyOutBytes + 1024 + 256;
// The TMEM accumulator is restarted every kSyChunkKB stages (1024 rows) and the
// partial products are summed in fp32 by the epilogue: long worker shards
// (12544 rows in the ResNet workload) then keep ~1e-6 relative accuracy.
constexpr int kSyChunkKB = 16;

struct SyProb {
  float* out;
  long long ld_out, stride_out;
  long long unit_begin;
  int d, rows_p, units_per_shard;
  float scale;
};

// Input side of a launch: the rows of bf16 matrices (linear layers) ...
struct SyLinear {};
// ... or the 3 x 3 patches of NHWC activations (conv layers, implicit im2col):
// one problem per worker, its tensor map an im2col map over the worker's
// images; the bias column and the columns past d come from `ones`.
struct SyConv {
  CUtensorMap ones;  // {64, 128} bf16: rows 0-63 = (1, 0, ..., 0), rows 64-127 = 0; box 64 x 64
  ConvGeom g[kSyMaxProbs];
};

template <class In>
struct SyParams {  // 128-byte aligned through CUtensorMap
  // inputs: linear {d, rows_p, P} bf16, box 64 x 64; conv: im2col {C, W, H, B/P}
  // of one worker, bounding box corners -1 (3 x 3, padding 1), 64 pixels x 64 channels
  CUtensorMap maps[kSyMaxProbs];
  CUtensorMap omaps[kSyMaxProbs];  // outputs {d, d, P} fp32, box 32 x 32, swizzled
  SyProb probs[kSyMaxProbs];
  In in;
  long long total_units;
  int* status;
  int n_probs, P, mirror;
};
static_assert(sizeof(SyParams<SyConv>) <= 32764, "kernel parameters exceed 32764 bytes");

struct SyUnit {
  int prob, p, i, w;
  int64_t j0;
};

// Work unit u -> (problem, shard, row block, columns), then the constant-time
// tile map (all three roles decode every unit).  Each role walks its units in
// increasing order, so the problem is found by advancing a cursor (`lo`, 0 at
// the start) over the problem table, which lives in the kernel's parameter
// space: a search with data-dependent indices there costs a constant-cache
// miss per probe.
template <class In>
__device__ __forceinline__ SyUnit sy_decode(const SyParams<In>& prm, long long u, int& lo) {
  while (lo + 1 < prm.n_probs && prm.probs[lo + 1].unit_begin <= u) ++lo;
  const SyProb& pr = prm.probs[lo];
  const int local = (int)(u - pr.unit_begin);
  SyUnit r;
  r.prob = lo;
  r.p = local / pr.units_per_shard;
  int j0;
  factor_unit_fast(pr.d, local - r.p * pr.units_per_shard, r.i, j0, r.w);
  r.j0 = j0;
  return r;
}

// One box of the 64 patch rows that start at output position (n, h, w) of the
// worker's images, `rem` of them inside the worker's rows.  A tap box is an
// im2col load from (w - 1, h - 1) (the map's bounding box starts one pixel
// before the image) with offsets (dw, dh); rows past the worker's last image
// fall outside the map and read zero.  The bias box reads rows 0-63 of
// `ones` (from row 64 - rem for a tail), a box past d rows 64-127.
template <bool MC>
__device__ __forceinline__ void sy_conv_load(const SyParams<SyConv>& prm, int e, const ConvBox& b, int n, int h,
                                             int w, int rem, void* dst, uint64_t* bar) {
  if (b.kind == 0) {
    if (MC)
      tma_load_im2col_4d_mc(dst, &prm.maps[e], b.c0, w - 1, h - 1, n, (uint16_t)b.dw, (uint16_t)b.dh, bar,
                            (uint16_t)0x3);
    else
      tma_load_im2col_4d(dst, &prm.maps[e], b.c0, w - 1, h - 1, n, (uint16_t)b.dw, (uint16_t)b.dh, bar);
  } else {
    const int y = b.kind == 1 ? (rem >= 64 ? 0 : 64 - rem) : 64;
    if (MC)
      tma_load_2d_mc(dst, &prm.in.ones, 0, y, bar, (uint16_t)0x3);
    else
      tma_load_2d(dst, &prm.in.ones, 0, y, bar);
  }
}

template <class In>
__global__ void __launch_bounds__(192, 1) syrk_tc_kernel(const __grid_constant__ SyParams<In> prm) {
  constexpr bool kConv = std::is_same<In, SyConv>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + kSyStages * kSyStageBytes;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + kSyOutBytes);
  uint64_t* empty = full + kSyStages;
  uint64_t* acc_full = empty + kSyStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSyStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);  // both CTAs' MMAs release a stage
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
  cluster_sync();  // the partner's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t rank = cluster_ctarank();
  // this CTA's units: 2 v + rank for the pair-chunks v of its cluster
  const long long pair0 = blockIdx.x / 2, pair_step = gridDim.x / 2, npairs = prm.total_units / 2;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int cur = 0;
      for (long long v = pair0; v < npairs && !*abort_flag; v += pair_step) {
        const SyUnit un = sy_decode(prm, 2 * v + rank, cur);
        const SyProb& pr = prm.probs[un.prob];
        const CUtensorMap* map = &prm.maps[un.prob];
        const int nb = (un.w + 63) / 64;
        const int nk = (pr.rows_p + kSyBK - 1) / kSyBK;
        // this CTA's share of the column boxes (multicast to both CTAs)
        const int half = (nb + 1) / 2, q0 = rank == 0 ? 0 : half, q1 = rank == 0 ? half : nb;
        // conv: the unit's box sources (at most two column boxes per CTA) and the
        // output position (n, h, w) of the k-block's first patch row, stepped by 64
        ConvBox bx[4];
        ConvGeom g{};
        int n = 0, h = 0, w = 0;
        if constexpr (kConv) {
          g = prm.in.g[un.prob];
          bx[0] = conv_box_source(g, un.i * 2);
          bx[1] = conv_box_source(g, un.i * 2 + 1);
          bx[2] = conv_box_source(g, (int)(un.j0 / 64) + q0);
          bx[3] = conv_box_source(g, (int)(un.j0 / 64) + q0 + 1);
        }
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, prm.status)) break;
          uint8_t* sa = smem + stage * kSyStageBytes;
          uint8_t* sb = sa + kSyABytes;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)((2 + nb) * kSyBox));
          if constexpr (kConv) {
            const int rem = pr.rows_p - kb * kSyBK;
            sy_conv_load<false>(prm, un.prob, bx[0], n, h, w, rem, sa, &full[stage]);
            sy_conv_load<false>(prm, un.prob, bx[1], n, h, w, rem, sa + kSyBox, &full[stage]);
            if (q1 > q0) sy_conv_load<true>(prm, un.prob, bx[2], n, h, w, rem, sb + q0 * kSyBox, &full[stage]);
            if (q1 > q0 + 1)
              sy_conv_load<true>(prm, un.prob, bx[3], n, h, w, rem, sb + (q0 + 1) * kSyBox, &full[stage]);
            conv_step(g, n, h, w);
          } else {
            tma_load_3d(sa, map, un.i * 128, kb * kSyBK, un.p, &full[stage]);
            tma_load_3d(sa + kSyBox, map, un.i * 128 + 64, kb * kSyBK, un.p, &full[stage]);
            for (int q = q0; q < q1; ++q)
              tma_load_3d_mc(sb + q * kSyBox, map, (int)un.j0 + 64 * q, kb * kSyBK, un.p, &full[stage],
                             (uint16_t)0x3);
          }
          if (++stage == kSyStages) {
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
      int cur = 0;
      for (long long v = pair0; v < npairs && ok; v += pair_step) {
        const SyUnit un = sy_decode(prm, 2 * v + rank, cur);
        const SyProb& pr = prm.probs[un.prob];
        const int nb = (un.w + 63) / 64;
        const uint32_t idesc = idesc_bf16_f32(nb * 64, true, true);
        const int nk = (pr.rows_p + kSyBK - 1) / kSyBK;
        for (int kc = 0; kc < nk && ok; kc += kSyChunkKB) {
          const int kend = kc + kSyChunkKB < nk ? kc + kSyChunkKB : nk;
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
            const uint32_t a0 = smem_u32(smem + stage * kSyStageBytes);
            const uint32_t b0 = a0 + kSyABytes;
#pragma unroll
            for (int kk = 0; kk < kSyBK / 16; ++kk) {
              // 16 rows of k = two 8-row groups of 1024 B; 64-column blocks are kSyBox apart.
              const uint64_t ad = smem_desc_sw128(a0 + kk * 2048, kSyBox, 1024);
              const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, kSyBox, 1024);
              tc_mma_bf16(d_tmem, ad, bd, idesc, (kb != kc || kk != 0) ? 1u : 0u);
            }
            tc_commit_mc(&empty[stage], (uint16_t)0x3);
            if (++stage == kSyStages) {
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
    int obuf = 0;  // staging buffer of this warp in use
    bool ok = true;
    int cur = 0;
    for (long long v = pair0; v < npairs && ok; v += pair_step) {
      const SyUnit un = sy_decode(prm, 2 * v + rank, cur);
      const SyProb& pr = prm.probs[un.prob];
      const int nk = (pr.rows_p + kSyBK - 1) / kSyBK;
      const int nchunks = (nk + kSyChunkKB - 1) / kSyChunkKB;
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
  cluster_sync();  // no multicast or remote arrival is still headed for this CTA
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ fp32 (CUDA-core) factors
constexpr int kSmMaxProbs = 128;
struct SmProb {
  const void* x;
  float* out;
  long long ld_x, ld_out, stride_out;
  long long tile_begin;
  int d, rows_p, tiles_per_shard;
  float scale;
};
struct SmParams {
  SmProb probs[kSmMaxProbs];
  long long total_tiles;
  int n_probs, P, mirror;
};

template <typename Tin>
__global__ void __launch_bounds__(256) syrk_simt_kernel(const __grid_constant__ SmParams prm) {
  __shared__ __align__(16) float smem[simt_smem_bytes<float>() / sizeof(float)];
  int pi = 0;  // tiles are visited in increasing order: the problem only advances
  for (long long u = blockIdx.x; u < prm.total_tiles; u += gridDim.x) {
    while (pi + 1 < prm.n_probs && prm.probs[pi + 1].tile_begin <= u) ++pi;
    const SmProb& pr = prm.probs[pi];
    const long long local = u - pr.tile_begin;
    const int p = (int)(local / pr.tiles_per_shard);
    int t = (int)(local % pr.tiles_per_shard);
    // upper tile (i, j) of the 128-grid, row-major over i
    const int T = (pr.d + 127) / 128;
    int i = 0;
    while (t >= T - i) {
      t -= T - i;
      ++i;
    }
    const int j = i + t;
    const Tin* xs = static_cast<const Tin*>(pr.x) + (long long)p * pr.rows_p * pr.ld_x;
    Opnd<Tin> A{xs + i * 128, 1, pr.ld_x, min(128, pr.d - i * 128)};
    Opnd<Tin> B{xs + j * 128, 1, pr.ld_x, min(128, pr.d - j * 128)};
    float acc[8][8];
    zero_acc(acc);
    simt_tile<float, Tin, Tin>(acc, A, B, pr.rows_p, smem);
    float* outp = pr.out + (long long)p * pr.stride_out;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const int r = i * 128 + ty * 8 + a;
      if (r >= pr.d) continue;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int c = j * 128 + tx * 8 + b;
        if (c >= pr.d) continue;
        const float v = acc[a][b] * pr.scale;
        outp[(long long)r * pr.ld_out + c] = v;
        if (prm.mirror && j > i) outp[(long long)c * pr.ld_out + r] = v;
      }
    }
  }
}

// ------------------------------------------------------------------ spatial sum (conv G helper)
template <typename Tin>
__global__ void __launch_bounds__(256) spatial_sum_kernel(const Tin* __restrict__ g, long long hw, long long C,
                                                          long long ld_g, float* __restrict__ gs, long long ld_gs) {
  // block: 64 channels x 4 position lanes; grid: (ceil(C/64), batch)
  __shared__ float red[4][64];
  const int cl = threadIdx.x % 64, sl = threadIdx.x / 64;
  const long long c = (long long)blockIdx.x * 64 + cl;
  const long long b = blockIdx.y;
  float acc = 0.f;
  if (c < C) {
    const Tin* base = g + (b * hw) * ld_g + c;
    for (long long s = sl; s < hw; s += 4) acc += load_as<float, Tin>(base + s * ld_g);
  }
  red[sl][cl] = acc;
  __syncthreads();
  if (sl == 0 && c < C) gs[b * ld_gs + c] = (red[0][cl] + red[1][cl]) + (red[2][cl] + red[3][cl]);
}

// ------------------------------------------------------------------ host side
// Output side of one problem: the fp32 factors {d, d, P} (TMA map and unit table).
static int sy_set_output(EncodeTiledFn enc, CUtensorMap* omap, SyProb& pr, float* out, long long d, long long ld_out,
                         long long stride_out, int P, long long rows_p, float scale, long long& units) {
  const long long so = P > 1 ? stride_out : d * ld_out;
  cuuint64_t odim[3] = {(cuuint64_t)d, (cuuint64_t)d, (cuuint64_t)P};
  cuuint64_t ostride[2] = {(cuuint64_t)ld_out * 4, (cuuint64_t)so * 4};
  cuuint32_t obox[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (enc(omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, odim, ostride, obox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return KFAC_ERR_INVALID_ARG;
  pr.out = out;
  pr.ld_out = ld_out;
  pr.stride_out = stride_out;
  pr.d = (int)d;
  pr.rows_p = (int)rows_p;
  pr.units_per_shard = (int)factor_units(d);
  pr.unit_begin = units;
  pr.scale = scale;
  units += (long long)pr.units_per_shard * P;
  return KFAC_OK;
}

// One launch: clusters of two CTAs, one per pair-chunk of the tile map.
template <class In>
static int sy_launch(const SyParams<In>& prm, int sms, double work, int kind, cudaStream_t stream) {
  if (prm.total_units == 0) return KFAC_OK;
  const long long pairs = prm.total_units / 2, clusters = pairs < sms / 2 ? pairs : sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = kSySmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfMark pm;
  prof_begin(stream, pm);
  if (cudaLaunchKernelEx(&cfg, syrk_tc_kernel<In>, prm) != cudaSuccess) return KFAC_ERR_CUDA;
  prof_end(kind, stream, pm, work);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA;
}

int launch_factors(int n, const kfac_factor_args* args, int dtype, int P, int mirror, cudaStream_t stream) {
  if (dtype == KFAC_BF16) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return KFAC_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
    const int sms = device_sm_count(dev);
    if (sms <= 0) return KFAC_ERR_CUDA;
    if (!ensure_smem_attr(dev, (const void*)syrk_tc_kernel<SyLinear>, kSySmem)) return KFAC_ERR_CUDA;
    for (int base = 0; base < n; base += kSyMaxProbs) {
      const int cnt = n - base < kSyMaxProbs ? n - base : kSyMaxProbs;
      SyParams<SyLinear> prm;
      memset(&prm, 0, sizeof(prm));
      long long units = 0;
      double work = 0.0;  // algorithmic flops of the launch
      for (int k = 0; k < cnt; ++k) {
        const kfac_factor_args& a = args[base + k];
        const long long rows_p = a.rows / P;
        cuuint64_t gdim[3] = {(cuuint64_t)a.d, (cuuint64_t)rows_p, (cuuint64_t)P};
        cuuint64_t gstride[2] = {(cuuint64_t)a.ld_x * 2, (cuuint64_t)(rows_p * a.ld_x * 2)};
        cuuint32_t box[3] = {64, kSyBK, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult cr = enc(&prm.maps[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.x), gdim, gstride,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return KFAC_ERR_INVALID_ARG;
        const int st = sy_set_output(enc, &prm.omaps[k], prm.probs[k], a.out, a.d, a.ld_out, a.stride_out, P, rows_p,
                                     a.scale, units);
        if (st != KFAC_OK) return st;
        const double d = (double)a.d;
        work += 2.0 * (double)a.rows * d * (d + 1.0) / 2.0;
      }
      prm.n_probs = cnt;
      prm.P = P;
      prm.mirror = mirror;
      prm.total_units = units;
      prm.status = device_status_ptr();
      if (!prm.status) return KFAC_ERR_CUDA;
      const int st = sy_launch(prm, sms, work, KFAC_K_SYRK, stream);
      if (st != KFAC_OK) return st;
    }
    return KFAC_OK;
  }
  // fp32 inputs on CUDA cores
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  for (int base = 0; base < n; base += kSmMaxProbs) {
    const int cnt = n - base < kSmMaxProbs ? n - base : kSmMaxProbs;
    SmParams prm;
    memset(&prm, 0, sizeof(prm));
    long long tiles = 0;
    for (int k = 0; k < cnt; ++k) {
      const kfac_factor_args& a = args[base + k];
      SmProb& pr = prm.probs[k];
      const long long T = (a.d + 127) / 128;
      pr.x = a.x;
      pr.out = a.out;
      pr.ld_x = a.ld_x;
      pr.ld_out = a.ld_out;
      pr.stride_out = a.stride_out;
      pr.d = (int)a.d;
      pr.rows_p = (int)(a.rows / P);
      pr.tiles_per_shard = (int)(T * (T + 1) / 2);
      pr.tile_begin = tiles;
      pr.scale = a.scale;
      tiles += (long long)pr.tiles_per_shard * P;
    }
    prm.n_probs = cnt;
    prm.P = P;
    prm.mirror = mirror;
    prm.total_tiles = tiles;
    if (tiles == 0) continue;
    const long long cap = (long long)sms * 4;
    const int grid = (int)(tiles < cap ? tiles : cap);
    syrk_simt_kernel<float><<<grid, 256, 0, stream>>>(prm);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

// Rows 0-63: (1, 0, ..., 0), rows 64-127: zeros (64 bf16 per row): the bias
// column of the conv patch matrix and the boxes past d.
struct SyOnesTile {
  uint16_t v[128 * 64];
};
static constexpr SyOnesTile make_ones_tile() {
  SyOnesTile t{};
  for (int r = 0; r < 64; ++r) t.v[r * 64] = 0x3F80;  // bf16 1.0
  return t;
}
__device__ __align__(128) SyOnesTile g_conv_ones = make_ones_tile();

int launch_conv_factors(int n, const kfac_conv_factor_args* args, int P, int mirror, cudaStream_t stream) {
  EncodeTiledFn enc = tensor_map_encoder();
  EncodeIm2colFn enc_i2c = tensor_map_im2col_encoder();
  if (!enc || !enc_i2c) return KFAC_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  if (!ensure_smem_attr(dev, (const void*)syrk_tc_kernel<SyConv>, kSySmem)) return KFAC_ERR_CUDA;
  void* ones = nullptr;
  if (cudaGetSymbolAddress(&ones, g_conv_ones) != cudaSuccess) return KFAC_ERR_CUDA;
  // one problem per (layer, worker)
  const long long total = (long long)n * P;
  for (long long base = 0; base < total; base += kSyMaxProbs) {
    const int cnt = (int)(total - base < kSyMaxProbs ? total - base : kSyMaxProbs);
    SyParams<SyConv> prm;
    memset(&prm, 0, sizeof(prm));
    {
      cuuint64_t gdim[2] = {64, 128};
      cuuint64_t gstride[1] = {128};
      cuuint32_t box[2] = {64, 64};
      cuuint32_t estr[2] = {1, 1};
      if (enc(&prm.in.ones, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ones, gdim, gstride, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KFAC_ERR_CUDA;
    }
    long long units = 0;
    double work = 0.0;  // algorithmic flops of the launch
    for (int k = 0; k < cnt; ++k) {
      const long long e = base + k;
      const kfac_conv_factor_args& a = args[e / P];
      const int p = (int)(e % P);
      const long long Bp = a.B / P, d = 9 * a.C + 1, rows_p = Bp * a.H * a.W;
      // this worker's images, NHWC: {C, W, H, B/P}; the bounding box of a 3 x 3,
      // padding 1 window starts one pixel before the image and ends two before its end
      const uint16_t* x = static_cast<const uint16_t*>(a.x) + (long long)p * rows_p * a.C;
      cuuint64_t gdim[4] = {(cuuint64_t)a.C, (cuuint64_t)a.W, (cuuint64_t)a.H, (cuuint64_t)Bp};
      cuuint64_t gstride[3] = {(cuuint64_t)(a.C * 2), (cuuint64_t)(a.W * a.C * 2), (cuuint64_t)(a.H * a.W * a.C * 2)};
      int lower[2] = {-1, -1}, upper[2] = {-1, -1};
      cuuint32_t estr[4] = {1, 1, 1, 1};
      if (enc_i2c(&prm.maps[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(x), gdim, gstride, lower,
                  upper, 64, kSyBK, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KFAC_ERR_INVALID_ARG;
      const int st = sy_set_output(enc, &prm.omaps[k], prm.probs[k], a.out + (long long)p * a.stride_out, d,
                                   a.ld_out, 0, 1, rows_p, a.scale, units);
      if (st != KFAC_OK) return st;
      prm.in.g[k] = make_conv_geom((int)a.C, (int)a.H, (int)a.W, kSyBK);
      work += 2.0 * (double)rows_p * (double)d * ((double)d + 1.0) / 2.0;
    }
    prm.n_probs = cnt;
    prm.P = 1;
    prm.mirror = mirror;
    prm.total_units = units;
    prm.status = device_status_ptr();
    if (!prm.status) return KFAC_ERR_CUDA;
    const int st = sy_launch(prm, sms, work, KFAC_K_CONV_SYRK, stream);
    if (st != KFAC_OK) return st;
  }
  return KFAC_OK;
}

int launch_spatial_sum(const void* g, int dtype, int64_t batch, int64_t hw, int64_t C, int64_t ld_g, float* gs,
                       int64_t ld_gs, cudaStream_t stream) {
  dim3 grid((unsigned)((C + 63) / 64), (unsigned)batch);
  if (dtype == KFAC_BF16)
    spatial_sum_kernel<uint16_t><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(g), hw, C, ld_g, gs, ld_gs);
  else
    spatial_sum_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(g), hw, C, ld_g, gs, ld_gs);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA;
}

}  // namespace kfac
