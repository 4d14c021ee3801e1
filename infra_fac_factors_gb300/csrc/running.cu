// Fused aggregation + running average + damping, one pass over the upper
// tiles of every factor (SPD-KFAC §II-C: the P workers' local factors are
// aggregated before inverting; §II-B: Tikhonov damping):
//
//   F       = (1/P) sum_p shards[p]
//   running = first_step ? F : decay * running + (1 - decay) * F
//   damped  = running + gamma * I
//
// HBM-bound: per element P (+1) fp32 reads and 2 fp32 writes.  One warp streams
// one row segment [128*floor(r/128), d) with 16-byte loads, two per lane per
// iteration (columns c and c + 128); the loads of up to eight shards of both
// are issued before they are summed.
#include "common.cuh"
#include "launch.h"

namespace kfac {

constexpr int kRunMaxProbs = 256;

struct RunProb {
  const float* shards;
  float* running;
  float* damped;
  long long stride, ld, row_begin;
  int d;
};
struct RunParams {
  RunProb probs[kRunMaxProbs];
  long long total_rows;
  int n_probs, P, first_step;
  float decay, gamma, inv_p;
};

__global__ void __launch_bounds__(256) update_running_kernel(const __grid_constant__ RunParams prm) {
  const int lane = threadIdx.x % 32;
  const long long warp_global = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) / 32;
  const float decay = prm.decay, keep = 1.f - prm.decay;
  int pi = 0;  // rows are visited in increasing order: the problem only advances
  for (long long g = warp_global; g < prm.total_rows; g += nwarps) {
    while (pi + 1 < prm.n_probs && prm.probs[pi + 1].row_begin <= g) ++pi;
    const RunProb& pr = prm.probs[pi];
    const long long r = g - pr.row_begin;
    const long long c_begin = (r / 128) * 128;
    const long long off_row = r * pr.ld;
    // vector part: two 16-byte groups per lane per iteration (c and c + 128)
    const long long c_vec_end = c_begin + ((pr.d - c_begin) / 4) * 4;
    for (long long cb = c_begin + lane * 4; cb < c_vec_end; cb += 256) {
      float4 f2[2];
      const bool two = cb + 128 < c_vec_end;
      // the running factor's values, loaded with the shards' (not after their sum)
      float4 old2[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
      if (!prm.first_step) {
        old2[0] = *reinterpret_cast<const float4*>(pr.running + off_row + cb);
        if (two) old2[1] = *reinterpret_cast<const float4*>(pr.running + off_row + cb + 128);
      }
      {
        float4 v[16];
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < prm.P) {
            v[p] = __ldcs(reinterpret_cast<const float4*>(pr.shards + off_row + cb + (long long)p * pr.stride));
            if (two) v[8 + p] = __ldcs(reinterpret_cast<const float4*>(pr.shards + off_row + cb + 128 + (long long)p * pr.stride));
          }
        for (int h = 0; h < 2; ++h) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int p = 0; p < 8; ++p)
            if (p < prm.P) {
              acc.x += v[8 * h + p].x; acc.y += v[8 * h + p].y; acc.z += v[8 * h + p].z; acc.w += v[8 * h + p].w;
            }
          f2[h] = acc;
        }
        for (int p0 = 8; p0 < prm.P; ++p0) {  // P > 8: the rest one by one
          const float4 a = __ldcs(reinterpret_cast<const float4*>(pr.shards + off_row + cb + (long long)p0 * pr.stride));
          f2[0].x += a.x; f2[0].y += a.y; f2[0].z += a.z; f2[0].w += a.w;
          if (two) {
            const float4 b = __ldcs(reinterpret_cast<const float4*>(pr.shards + off_row + cb + 128 + (long long)p0 * pr.stride));
            f2[1].x += b.x; f2[1].y += b.y; f2[1].z += b.z; f2[1].w += b.w;
          }
        }
      }
      for (int h = 0; h < (two ? 2 : 1); ++h) {
        const long long c = cb + 128 * h;
        const long long off = off_row + c;
        float4 f = f2[h];
        f.x *= prm.inv_p;
        f.y *= prm.inv_p;
        f.z *= prm.inv_p;
        f.w *= prm.inv_p;
        float4 rn;
        if (prm.first_step) {
          rn = f;
        } else {
          const float4 old = old2[h];
          rn.x = fmaf(decay, old.x, keep * f.x);
          rn.y = fmaf(decay, old.y, keep * f.y);
          rn.z = fmaf(decay, old.z, keep * f.z);
          rn.w = fmaf(decay, old.w, keep * f.w);
        }
        float4 dm = rn;
        if (r >= c && r < c + 4) {
          const int k = (int)(r - c);
          if (k == 0) dm.x += prm.gamma;
          if (k == 1) dm.y += prm.gamma;
          if (k == 2) dm.z += prm.gamma;
          if (k == 3) dm.w += prm.gamma;
        }
        *reinterpret_cast<float4*>(pr.running + off) = rn;
        __stcs(reinterpret_cast<float4*>(pr.damped + off), dm);
      }
    }
    // scalar tail (d not a multiple of 4)
    const long long c = c_vec_end + lane;
    if (c < pr.d) {
      const long long off = off_row + c;
      float f = 0.f;
      for (int p = 0; p < prm.P; ++p) f += pr.shards[off + (long long)p * pr.stride];
      f *= prm.inv_p;
      const float rn = prm.first_step ? f : fmaf(decay, pr.running[off], keep * f);
      pr.running[off] = rn;
      pr.damped[off] = (c == r) ? rn + prm.gamma : rn;
    }
  }
}

int launch_update_running(int n, const kfac_running_args* args, int P, float decay, float gamma, int first_step,
                          cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  for (int base = 0; base < n; base += kRunMaxProbs) {
    const int cnt = n - base < kRunMaxProbs ? n - base : kRunMaxProbs;
    RunParams prm;
    memset(&prm, 0, sizeof(prm));
    long long rows = 0;
    for (int k = 0; k < cnt; ++k) {
      const kfac_running_args& a = args[base + k];
      RunProb& pr = prm.probs[k];
      pr.shards = a.shards;
      pr.running = a.running;
      pr.damped = a.damped;
      pr.stride = a.stride_shard;
      pr.ld = a.ld;
      pr.d = (int)a.d;
      pr.row_begin = rows;
      rows += a.d;
    }
    prm.n_probs = cnt;
    prm.P = P;
    prm.first_step = first_step;
    prm.decay = decay;
    prm.gamma = gamma;
    prm.inv_p = 1.0f / (float)P;
    prm.total_rows = rows;
    if (rows == 0) continue;
    const long long want = (rows + 7) / 8;  // 8 warps per block, one row per warp
    const long long cap = (long long)sms * 8;
    const int grid = (int)(want < cap ? want : cap);
    double work = 0.0;  // algorithmic bytes: P shard reads, running read (not on a first step) and write, damped write
    for (int k = 0; k < cnt; ++k) {
      const double d = (double)args[base + k].d;
      work += (double)(P + (first_step ? 2 : 3)) * 4.0 * d * (d + 1.0) / 2.0;
    }
    ProfMark pm;
    prof_begin(stream, pm);
    update_running_kernel<<<grid, 256, 0, stream>>>(prm);
    prof_end(KFAC_K_RUNNING, stream, pm, work);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

}  // namespace kfac
