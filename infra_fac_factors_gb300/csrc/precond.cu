// Preconditioned gradient of each layer (SPD-KFAC §II-B, the damped update
// rule):  out = inv_g * grad * inv_a, on tcgen05 tensor cores.
//
// The fp32 operands are carried as three bf16 slices (x = hi + mid + lo, all 24
// bits of fp32; six products per multiply-add, gemm_tc.cu), and every 16-wide
// k-step is summed into fp32 registers with round-to-nearest.  Less does not
// do: grad lies in the row space of the layer input while inv_a has gain up to
// 1/gamma on the other directions, so operand rounding and accumulation error
// are amplified ~1/gamma-fold (two slices, 16 bits, gave 1e-2 relative error on
// the first steps of the MLP workload, where 529 of 785 directions have gain
// 1000; one tensor-core accumulator over the whole K gave 5e-3).
//   1. split      grad, inv_a, inv_g -> bf16 slices               (one launch)
//   2. GEMM 1     tmp^T = inv_a * grad^T   (d_in x d_out), written as slices
//   3. GEMM 2     out   = inv_g * tmp      (= inv_g * (tmp^T)^T), fp32
// inv_a and inv_g are symmetric, so their rows serve as the K-major operands.
#include "common.cuh"
#include "gemm_tc.h"
#include "launch.h"

namespace kfac {

constexpr int kPcSlices = 3;

static long long pad8(long long v) { return (v + 7) / 8 * 8; }
static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct PcLayout {
  size_t grad, inv_a, inv_g, tmp, end;
};

// Workspace of layer i starting at byte `off`: four sliced operands.
static PcLayout pc_layout(const kfac_precond_args& a, size_t off) {
  const size_t s = kPcSlices * sizeof(uint16_t);
  PcLayout L;
  L.grad = off;
  off += align256(s * a.d_out * pad8(a.d_in));
  L.inv_a = off;
  off += align256(s * a.d_in * pad8(a.d_in));
  L.inv_g = off;
  off += align256(s * a.d_out * pad8(a.d_out));
  L.tmp = off;
  off += align256(s * a.d_in * pad8(a.d_out));
  L.end = off;
  return L;
}

size_t precondition_workspace(int n, const kfac_precond_args* args) {
  size_t off = 0;
  for (int i = 0; i < n; ++i) off = pc_layout(args[i], off).end;
  return off;
}

int launch_precondition(int n, const kfac_precond_args* args, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  if (workspace_bytes < precondition_workspace(n, args) || (workspace == nullptr && n > 0)) return KFAC_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SplitItem* items = new SplitItem[3 * (size_t)n];
  GtOperand* g1 = new GtOperand[n];
  GtOperand* g2 = new GtOperand[n];
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    const kfac_precond_args& a = args[i];
    const PcLayout L = pc_layout(a, off);
    off = L.end;
    uint16_t* s_grad = reinterpret_cast<uint16_t*>(ws + L.grad);
    uint16_t* s_ia = reinterpret_cast<uint16_t*>(ws + L.inv_a);
    uint16_t* s_ig = reinterpret_cast<uint16_t*>(ws + L.inv_g);
    uint16_t* s_tmp = reinterpret_cast<uint16_t*>(ws + L.tmp);
    const long long ldi = pad8(a.d_in), ldo = pad8(a.d_out);
    items[3 * i + 0] = SplitItem{a.grad, s_grad, a.d_out, a.d_in, a.ld_grad, ldi, a.d_out * ldi, 0};
    items[3 * i + 1] = SplitItem{a.inv_a, s_ia, a.d_in, a.d_in, a.ld_a, ldi, a.d_in * ldi, 0};
    items[3 * i + 2] = SplitItem{a.inv_g, s_ig, a.d_out, a.d_out, a.ld_g, ldo, a.d_out * ldo, 0};
    // tmp^T[n][m] = sum_k inv_a[n][k] grad[m][k]: M = d_in, N = d_out, K = d_in
    g1[i] = GtOperand{s_ia, s_grad, a.d_in, a.d_out, a.d_in, ldi, ldi, s_tmp, ldo, a.d_in * ldo, 1, 1.0f};
    // out[m][n] = sum_k inv_g[m][k] tmp^T[n][k]: M = d_out, N = d_in, K = d_out
    g2[i] = GtOperand{s_ig, s_tmp, a.d_out, a.d_in, a.d_out, ldo, ldo, a.out, a.ld_out, 0, 0, 1.0f};
  }
  int rc = launch_split(items, 3 * n, stream);
  if (rc == KFAC_OK) rc = launch_gemm_tc(g1, n, stream);
  if (rc == KFAC_OK) rc = launch_gemm_tc(g2, n, stream);
  delete[] items;
  delete[] g1;
  delete[] g2;
  return rc;
}

}  // namespace kfac
