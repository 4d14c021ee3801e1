// Epilogue of the tensor-core factor SYRK (factors.cu: both its linear-layer
// and its implicit-im2col conv instantiation).
//
// One epilogue warp owns TMEM lane quarter q, i.e. rows i*128 + 32q .. +31 of
// a work unit (row block i, columns [j0, j0 + w) of the tile map in
// tilemap.cuh).  For one K-chunk it reads the 128 x w fp32 accumulator in
// 32 x 32 blocks, scales them and writes the unit's stored part (columns
// >= 128 i) of the shard's factor:
//   * upper tiles only: each block is staged in shared memory (128-byte
//     swizzle: chunk j of row t lands at chunk j ^ (t & 7), conflict-free) and
//     written by a TMA store; later K-chunks of the same unit add with a TMA
//     reduce.  A block reaching past the last full 16-byte group of a row is
//     written with plain stores (TMA writes whole groups at the inner edge);
//   * mirrored: plain stores of the block and, on the last K-chunk, of its
//     transpose into the lower triangle.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace kfac {

constexpr int kFeStageOut = 4096;  // one 32 x 32 fp32 staging block

struct FeUnit {
  float* outp;              // this shard's d x d factor
  const CUtensorMap* omap;  // the factors {d, d, P} fp32, box 32 x 32, 128-byte swizzle
  long long ld_out, j0;
  int d, i, w, p;
  float scale;
};

// `tmem_acc`: TMEM address of this warp's lane quarter in the accumulator;
// `stage2`: the warp's two staging blocks (2 * kFeStageOut bytes, 1024-aligned);
// `obuf`: which of them is next (kept across chunks and units).
__device__ __forceinline__ void factor_epilogue_chunk(uint32_t tmem_acc, int q, int lane, const FeUnit& u, bool first,
                                                      bool last, bool mirror, uint8_t* stage2, int& obuf) {
  const int nb = (u.w + 63) / 64;
  const int r = u.i * 128 + q * 32 + lane;
  float* orow = u.outp + (long long)r * u.ld_out;
  const long long jend = u.j0 + u.w;
  const long long lower_from = (long long)(u.i + 1) * 128;  // columns in lower-tile territory
  const long long store_from = (long long)u.i * 128;          // columns before it: not this unit's
  if (!mirror) {
    if (!first && lane == 0) bulk_wait<0>();  // earlier writes of this unit are done
    __syncwarp();
    const int r0 = u.i * 128 + q * 32;
    const long long d4 = (long long)(u.d / 4) * 4;
    for (int c = 0; c < nb * 2; ++c) {
      uint32_t v[32];
      tc_ld_32x32b_x32(tmem_acc + c * 32, v);
      tc_wait_ld();
      const long long col0 = u.j0 + c * 32;
      if (col0 >= jend || col0 < store_from || r0 >= u.d) continue;  // uniform over the warp
      if (col0 + 32 > d4 && d4 != u.d) {
        if (r < u.d)
          for (int t = 0; t < 32; ++t) {
            const long long col = col0 + t;
            if (col >= jend) break;
            float o = __uint_as_float(v[t]) * u.scale;
            if (!first) o += orow[col];
            orow[col] = o;
          }
        continue;
      }
      uint8_t* buf = stage2 + obuf * kFeStageOut;
      if (lane == 0) bulk_wait_read<1>();  // the store that last used `buf` has read it
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float4 o = make_float4(__uint_as_float(v[4 * j]) * u.scale, __uint_as_float(v[4 * j + 1]) * u.scale,
                               __uint_as_float(v[4 * j + 2]) * u.scale, __uint_as_float(v[4 * j + 3]) * u.scale);
        *reinterpret_cast<float4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (first)
          tma_store_3d(u.omap, buf, (int)col0, r0, u.p);
        else
          tma_reduce_add_3d(u.omap, buf, (int)col0, r0, u.p);
        bulk_commit();
      }
      obuf ^= 1;
    }
    return;
  }
  for (int c = 0; c < nb * 2; ++c) {
    uint32_t v[32];
    tc_ld_32x32b_x32(tmem_acc + c * 32, v);
    tc_wait_ld();
    const long long col0 = u.j0 + c * 32;
    if (r < u.d && col0 < jend && col0 >= store_from) {
      float o[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) o[t] = __uint_as_float(v[t]) * u.scale;
      if (col0 + 32 <= jend) {
#pragma unroll
        for (int t = 0; t < 32; t += 4) {
          float4* dst = reinterpret_cast<float4*>(orow + col0 + t);
          if (!first) {
            const float4 prev = *dst;
            o[t] += prev.x;
            o[t + 1] += prev.y;
            o[t + 2] += prev.z;
            o[t + 3] += prev.w;
          }
          *dst = make_float4(o[t], o[t + 1], o[t + 2], o[t + 3]);
        }
      } else {
        for (int t = 0; t < 32; ++t)
          if (col0 + t < jend) {
            if (!first) o[t] += orow[col0 + t];
            orow[col0 + t] = o[t];
          }
      }
      if (last) {
        for (int t = 0; t < 32; ++t) {
          const long long col = col0 + t;
          if (col < jend && col >= lower_from) u.outp[col * u.ld_out + r] = o[t];
        }
      }
    }
  }
}

}  // namespace kfac
