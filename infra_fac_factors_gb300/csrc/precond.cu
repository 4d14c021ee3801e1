// Preconditioned gradient of each layer (SPD-KFAC §II-B, the damped update
// rule):  out = inv_g * grad * inv_a.
// Two grouped GEMM launches over all layers: tmp = grad * inv_a, then
// out = inv_g * tmp.  fp32 operands, fp32 products and accumulation on CUDA
// cores (simt.cuh).
#include "common.cuh"
#include "launch.h"
#include "simt.cuh"

namespace kfac {

constexpr int kPcMaxProbs = 256;

struct GemmProb {
  const float* A;  // M x K, row-major (K contiguous)
  const float* B;  // K x N, row-major (N contiguous)
  float* C;        // M x N
  long long lda, ldb, ldc, tile_begin;
  int M, N, K, tiles_n;
};
struct GemmParams {
  GemmProb probs[kPcMaxProbs];
  long long total_tiles;
  int n_probs;
};

__global__ void __launch_bounds__(256) gemm_nn_kernel(const __grid_constant__ GemmParams prm) {
  __shared__ __align__(16) float smem[simt_smem_bytes<float>() / sizeof(float)];
  for (long long u = blockIdx.x; u < prm.total_tiles; u += gridDim.x) {
    int pi = 0;
    while (pi + 1 < prm.n_probs && prm.probs[pi + 1].tile_begin <= u) ++pi;
    const GemmProb& g = prm.probs[pi];
    const long long t = u - g.tile_begin;
    const int tm = (int)(t / g.tiles_n), tn = (int)(t % g.tiles_n);
    Opnd<float> A{g.A + (long long)tm * 128 * g.lda, g.lda, 1, min(128, g.M - tm * 128)};
    Opnd<float> B{g.B + (long long)tn * 128, 1, g.ldb, min(128, g.N - tn * 128)};
    float acc[8][8];
    zero_acc(acc);
    simt_tile<float, float, float>(acc, A, B, g.K, smem);
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const int r = tm * 128 + ty * 8 + a;
      if (r >= g.M) continue;
      float* crow = g.C + (long long)r * g.ldc;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int cidx = tn * 128 + tx * 8 + b;
        if (cidx < g.N) crow[cidx] = acc[a][b];
      }
    }
  }
}

static long long pad4(long long v) { return (v + 3) / 4 * 4; }

size_t precondition_workspace(int n, const kfac_precond_args* args) {
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += (size_t)args[i].d_out * pad4(args[i].d_in) * sizeof(float);
  return total;
}

static int run_gemms(const GemmProb* probs, int n, cudaStream_t stream, int sms) {
  for (int base = 0; base < n; base += kPcMaxProbs) {
    const int cnt = n - base < kPcMaxProbs ? n - base : kPcMaxProbs;
    GemmParams prm;
    memset(&prm, 0, sizeof(prm));
    long long tiles = 0;
    for (int k = 0; k < cnt; ++k) {
      prm.probs[k] = probs[base + k];
      GemmProb& g = prm.probs[k];
      g.tiles_n = (g.N + 127) / 128;
      g.tile_begin = tiles;
      tiles += (long long)((g.M + 127) / 128) * g.tiles_n;
    }
    prm.n_probs = cnt;
    prm.total_tiles = tiles;
    if (tiles == 0) continue;
    const long long cap = (long long)sms * 4;
    gemm_nn_kernel<<<(unsigned)(tiles < cap ? tiles : cap), 256, 0, stream>>>(prm);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

int launch_precondition(int n, const kfac_precond_args* args, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  if (workspace_bytes < precondition_workspace(n, args) || (workspace == nullptr && n > 0)) return KFAC_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  GemmProb* g1 = new GemmProb[n > 0 ? n : 1];
  GemmProb* g2 = new GemmProb[n > 0 ? n : 1];
  float* tmp = static_cast<float*>(workspace);
  for (int i = 0; i < n; ++i) {
    const kfac_precond_args& a = args[i];
    const long long ldt = pad4(a.d_in);
    GemmProb& p1 = g1[i];
    memset(&p1, 0, sizeof(p1));
    p1.A = a.grad;
    p1.lda = a.ld_grad;
    p1.B = a.inv_a;
    p1.ldb = a.ld_a;
    p1.C = tmp;
    p1.ldc = ldt;
    p1.M = (int)a.d_out;
    p1.N = (int)a.d_in;
    p1.K = (int)a.d_in;
    GemmProb& p2 = g2[i];
    memset(&p2, 0, sizeof(p2));
    p2.A = a.inv_g;
    p2.lda = a.ld_g;
    p2.B = tmp;
    p2.ldb = ldt;
    p2.C = a.out;
    p2.ldc = a.ld_out;
    p2.M = (int)a.d_out;
    p2.N = (int)a.d_in;
    p2.K = (int)a.d_out;
    tmp += a.d_out * ldt;
  }
  int rc = run_gemms(g1, n, stream, sms);
  if (rc == KFAC_OK) rc = run_gemms(g2, n, stream, sms);
  delete[] g1;
  delete[] g2;
  return rc;
}

}  // namespace kfac
