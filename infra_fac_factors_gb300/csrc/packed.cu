// Packed upper triangles of symmetric factors (SPD-KFAC §III-A: a symmetric
// d x d Kronecker factor is communicated as its d(d+1)/2 upper-triangle
// elements, and small factors are fused into one message; §IV: only the upper
// triangle of a symmetric inverse is sent).
//
// Layout: the upper triangle incl. the diagonal, row by row,
//   packed[r*d - r*(r-1)/2 + (c - r)] = M[r][c]      (0 <= r <= c < d),
// so row r is the d - r consecutive elements starting at r*d - r(r-1)/2.
//
// One launch covers every matrix of the call (the fused pass: many small
// factors move as one batch, as they would in one fused message).  One warp
// copies one row: lane l moves elements l, l + 32, ... with eight loads in
// flight before their stores, so both the row of M and the packed row are
// read and written in coalesced 128-byte runs (the two sides start at
// different offsets modulo 16 bytes, which rules out 16-byte vectors).
// Unpacking can also fill the strict lower triangle from the packed upper one
// (`mirror`): row r's columns c < r are gathered from the packed rows c.
#include "common.cuh"
#include "launch.h"

namespace kfac {

constexpr int kPkMaxProbs = 256;
constexpr int kPkUnroll = 8;

struct PkProb {
  float* mat;
  float* packed;
  long long ld, row_begin;
  int d;
};
struct PkParams {
  PkProb probs[kPkMaxProbs];
  long long total_rows;
  int n_probs, unpack, mirror;
};

__device__ __forceinline__ long long packed_row_start(long long r, long long d) { return r * d - r * (r - 1) / 2; }

__global__ void __launch_bounds__(256) packed_kernel(const __grid_constant__ PkParams prm) {
  const int lane = threadIdx.x % 32;
  const long long warp_global = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) / 32;
  int pi = 0;  // rows are visited in increasing order: the problem only advances
  for (long long g = warp_global; g < prm.total_rows; g += nwarps) {
    while (pi + 1 < prm.n_probs && prm.probs[pi + 1].row_begin <= g) ++pi;
    const PkProb& pr = prm.probs[pi];
    const long long r = g - pr.row_begin;
    const long long n = pr.d - r;  // elements of packed row r
    float* mrow = pr.mat + r * pr.ld + r;
    float* prow = pr.packed + packed_row_start(r, pr.d);
    const float* src = prm.unpack ? prow : mrow;
    float* dst = prm.unpack ? mrow : prow;
    for (long long j0 = 0; j0 < n; j0 += 32 * kPkUnroll) {
      float v[kPkUnroll];
#pragma unroll
      for (int u = 0; u < kPkUnroll; ++u) {
        const long long j = j0 + u * 32 + lane;
        if (j < n) v[u] = __ldcs(src + j);
      }
#pragma unroll
      for (int u = 0; u < kPkUnroll; ++u) {
        const long long j = j0 + u * 32 + lane;
        if (j < n) __stcs(dst + j, v[u]);
      }
    }
    if (prm.unpack && prm.mirror) {
      // M[r][c] = M[c][r] for c < r, from packed row c
      float* lrow = pr.mat + r * pr.ld;
      for (long long c = lane; c < r; c += 32) lrow[c] = pr.packed[packed_row_start(c, pr.d) + (r - c)];
    }
  }
}

int launch_packed(int n, const kfac_pack_args* args, int unpack, int mirror, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return KFAC_ERR_CUDA;
  for (int base = 0; base < n; base += kPkMaxProbs) {
    const int cnt = n - base < kPkMaxProbs ? n - base : kPkMaxProbs;
    PkParams prm;
    memset(&prm, 0, sizeof(prm));
    long long rows = 0;
    for (int k = 0; k < cnt; ++k) {
      const kfac_pack_args& a = args[base + k];
      PkProb& pr = prm.probs[k];
      pr.mat = a.mat;
      pr.packed = a.packed;
      pr.ld = a.ld;
      pr.d = (int)a.d;
      pr.row_begin = rows;
      rows += a.d;
    }
    prm.n_probs = cnt;
    prm.total_rows = rows;
    prm.unpack = unpack;
    prm.mirror = mirror;
    const long long want = (rows + 7) / 8;  // 8 warps per block, one row per warp
    const long long cap = (long long)sms * 16;
    const int grid = (int)(want < cap ? want : cap);
    packed_kernel<<<grid, 256, 0, stream>>>(prm);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

}  // namespace kfac
