// Preconditioned gradient of each layer (SPD-KFAC §II-B, the damped update
// rule):  out = inv_g * grad * inv_a, on tcgen05 tensor cores.
//
// The fp32 operands are carried as bf16 slices (x = hi + mid + lo, all 24 bits
// of fp32, gemm_tc.cu), and every twelve MMAs are summed into fp32 registers
// with round-to-nearest.  grad lies in the row space of the layer input while
// inv_a has gain up to 1/gamma on the other directions, so operand rounding is
// amplified up to ~1/gamma-fold: with 16-bit operands (two slices, three MMAs
// per multiply-add) the relative error of out is 6e-6 on the BERT QKV layer
// and 1.4e-4 on its FFN-out layer, but 9e-3 on the first steps of the MLP
// workload (529 of 785 directions have gain 1000) and 3.5e-3 on the C = 512
// ResNet conv.  With all 24 bits (three slices, six MMAs) it stays near 1e-5.
//
// KFAC_PRECOND_FP32: six MMAs per multiply-add for every layer.
//   1. split      grad, inv_a, inv_g -> three bf16 slices            (one launch)
//   2. GEMM 1     tmp^T = inv_a * grad^T   (d_in x d_out), written as slices
//   3. GEMM 2     out   = inv_g * tmp      (= inv_g * (tmp^T)^T), fp32
// KFAC_PRECOND_AUTO: the same with three MMAs per multiply-add, then an
// a-posteriori check of every layer, and the six-MMA pass (steps 1-3, three
// slices) for the layers the check flags only:
//   1'. split (two slices), fused with y = inv_a Z and s = inv_g Z' for eight
//       Rademacher probes on each side (Z: d_in x 8, Z': d_out x 8)
//   2', 3'. GEMMs with two slices
//   4. check: per layer, the 8 x 8 bilinear forms Z'^T out Z and
//      s^T grad y = Z'^T inv_g grad inv_a Z in one pass over grad and out;
//      the estimate ||Z'^T (out - inv_g grad inv_a) Z||_F / ||Z'^T inv_g grad
//      inv_a Z||_F tracks the relative Frobenius error of out (each bilinear
//      form of independent Rademacher vectors has mean square ||.||_F^2)
//   5. flag the layers whose estimate exceeds kPcAutoTol (or is not finite)
//   6. steps 1-3 with three slices for the flagged layers (device-side flags:
//      the launches skip the other layers' work)
// The optional weight step (weight -= lr * out) runs in the epilogue of the
// GEMM 2 launch that produces the final out (FP32: the only one; AUTO: the
// recomputation, for the flagged layers), and for the layers AUTO keeps at 16
// bits in pc_weight_kernel, from the stored out, after the check.
// inv_a and inv_g are symmetric, so their rows serve as the K-major operands,
// and s = inv_g Z' = (Z'^T inv_g)^T.
#include <mutex>

#include "common.cuh"
#include "gemm_tc.h"
#include "launch.h"
#include "split.cuh"

namespace kfac {

// Largest accepted estimate of the 16-bit result's relative error: 5x under
// the 2e-3 bar.  On the workloads the estimate falls within 0.79x..1.28x of
// the true error.
constexpr float kPcAutoTol = 4e-4f;
constexpr int kChkRows = 32;    // rows of out / grad per warp unit of the check
constexpr int kChkMax = 256;    // layers per check launch (parameter space)

static long long pad8(long long v) { return (v + 7) / 8 * 8; }
static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct PcLayout {
  size_t grad, inv_a, inv_g, tmp, end;
};

// Workspace of layer i starting at byte `off`: four sliced operands.
static PcLayout pc_layout(const kfac_precond_args& a, size_t off) {
  const size_t s = kSlices * sizeof(uint16_t);
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

// After all layers' slices: the probe region (zeroed by every AUTO call), then
// the flags.  Per layer: y [d_in][8] and s [d_out][8] fp32; then per layer 128
// doubles (Z'^T out Z and s^T grad y, 8 x 8 each).
struct PcProbeLayout {
  size_t begin, acc, flags, end;
};

static PcProbeLayout pc_probe_layout(int n, const kfac_precond_args* args, size_t off) {
  PcProbeLayout P;
  P.begin = off;
  for (int i = 0; i < n; ++i) off += align256(sizeof(float) * kProbeN * (args[i].d_in + args[i].d_out));
  P.acc = off;
  off += align256(sizeof(double) * 2 * kProbeN * kProbeN * (size_t)n);
  P.flags = off;
  off += align256(sizeof(int) * (size_t)n);
  P.end = off;
  return P;
}

size_t precondition_workspace(int n, const kfac_precond_args* args) {
  size_t off = 0;
  for (int i = 0; i < n; ++i) off = pc_layout(args[i], off).end;
  return pc_probe_layout(n, args, off).end;
}

// ------------------------------------------------------------------ check
struct PcChkItem {
  const float* grad;
  const float* out;
  const float* y;  // [d_in][8]
  const float* s;  // [d_out][8]
  double* acc;     // [2][8][8]: Z'^T out Z, s^T grad y
  long long ld_grad, ld_out, d_out, d_in, unit_begin;
};

struct PcChkParams {
  PcChkItem items[kChkMax];
  long long total_units;
  int n;
};

// left probe l at row r (the probes of gemm_tc.h with bit offset 8)
__device__ __forceinline__ float left_sign(long long r, int l) {
  const uint32_t hh = probe_hash((uint32_t)(r >> 3)), h = hh >> 8;
  const int e = (int)(r & 7);
  const int b = e ^ probe_class_offset(hh, 8);
  return ((__popc(l & b) + (int)((h >> e) & 1u)) & 1) ? -1.f : 1.f;
}

// p[k] = sum_e z_k[c0 + e] x[e]: the right probes (bit offset 0)
__device__ __forceinline__ void right_probe8(const float (&x)[8], long long c0, float (&p)[8]) {
  const uint32_t h = probe_hash((uint32_t)(c0 >> 3));
  const int t = probe_class_offset(h, 0);
#pragma unroll
  for (int e = 0; e < 8; ++e) p[e] = ((h >> e) & 1u) ? -x[e] : x[e];
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

// Warp unit: one 256-column segment (8 columns per lane) of kChkRows rows.
// Per row the lanes' partial sums w_k = (grad y_k)_r and q_k = (out z_k)_r
// (16 values) are reduce-scattered in 16 shuffles; lane pairs (2j, 2j + 1)
// then hold value j (q_0..7 for j < 8, w_0..7 after) and multiply it by
// z'_l[r] (for q) or s_l[r] (for w), each lane of the pair for four l.
// NW warps per block: eight (the check running alone) or two (one block per
// NW units, 64 threads and 8 K registers: it fits beside a preconditioning
// GEMM block on one SM).
template <int NW>
__global__ void __launch_bounds__(NW * 32, 16 / NW) pc_check_kernel(const __grid_constant__ PcChkParams prm) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // value this lane holds after the reduce-scatter: bits 4..1 of the lane
  const int j = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
  const int is_w = j >> 3, kj = j & 7, l0 = (lane & 1) * 4;
  for (long long u = (long long)blockIdx.x * NW + warp; u < prm.total_units; u += (long long)gridDim.x * NW) {
    int lo = 0, hi = prm.n;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prm.items[mid].unit_begin <= u)
        lo = mid;
      else
        hi = mid;
    }
    const PcChkItem& it = prm.items[lo];
    const long long segs = (it.d_in + 255) / 256;
    const long long local = u - it.unit_begin;
    const long long rg = local / segs;
    const long long c0 = (local - rg * segs) * 256 + lane * 8;
    float yv[8][8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (c0 + e < it.d_in) {
        const float4 a = *reinterpret_cast<const float4*>(it.y + (c0 + e) * kProbeN);
        const float4 b = *reinterpret_cast<const float4*>(it.y + (c0 + e) * kProbeN + 4);
        yv[e][0] = a.x; yv[e][1] = a.y; yv[e][2] = a.z; yv[e][3] = a.w;
        yv[e][4] = b.x; yv[e][5] = b.y; yv[e][6] = b.z; yv[e][7] = b.w;
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) yv[e][k] = 0.f;
      }
    }
    float acc4[4] = {0.f, 0.f, 0.f, 0.f};
    const long long r_end = (rg + 1) * kChkRows < it.d_out ? (rg + 1) * kChkRows : it.d_out;
    // this lane's 8 columns of row r of grad and out (zero past d_in)
    auto fetch = [&](long long r, float (&g8)[8], float (&o8)[8]) {
      if (c0 + 8 <= it.d_in) {
        const float4 a = *reinterpret_cast<const float4*>(it.grad + r * it.ld_grad + c0);
        const float4 b = *reinterpret_cast<const float4*>(it.grad + r * it.ld_grad + c0 + 4);
        const float4 c = *reinterpret_cast<const float4*>(it.out + r * it.ld_out + c0);
        const float4 d = *reinterpret_cast<const float4*>(it.out + r * it.ld_out + c0 + 4);
        g8[0] = a.x; g8[1] = a.y; g8[2] = a.z; g8[3] = a.w; g8[4] = b.x; g8[5] = b.y; g8[6] = b.z; g8[7] = b.w;
        o8[0] = c.x; o8[1] = c.y; o8[2] = c.z; o8[3] = c.w; o8[4] = d.x; o8[5] = d.y; o8[6] = d.z; o8[7] = d.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const bool in = c0 + e < it.d_in;
          g8[e] = in ? it.grad[r * it.ld_grad + c0 + e] : 0.f;
          o8[e] = in ? it.out[r * it.ld_out + c0 + e] : 0.f;
        }
      }
    };
    // the next row is fetched while the current one is reduced
    float gn[8], on[8];
    if (rg * kChkRows < r_end) fetch(rg * kChkRows, gn, on);
    for (long long r = rg * kChkRows; r < r_end; ++r) {
      float g8[8], o8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        g8[e] = gn[e];
        o8[e] = on[e];
      }
      if (r + 1 < r_end) fetch(r + 1, gn, on);
      float v[16], q[8];
      right_probe8(o8, c0, q);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[k] = q[k];
        float w = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) w = fmaf(g8[e], yv[e][k], w);
        v[8 + k] = w;
      }
      // reduce-scatter over the warp: offsets 16, 8, 4, 2 halve the values
      // held, offset 1 completes the sum (lanes 2j and 2j + 1 agree)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool up = lane & 16;
        const float send = up ? v[i] : v[i + 8], keep = up ? v[i + 8] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool up = lane & 8;
        const float send = up ? v[i] : v[i + 4], keep = up ? v[i + 4] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bool up = lane & 4;
        const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
      {
        const bool up = lane & 2;
        const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
      }
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      if (is_w) {
        const float4 sl = *reinterpret_cast<const float4*>(it.s + r * kProbeN + l0);
        acc4[0] = fmaf(sl.x, v[0], acc4[0]);
        acc4[1] = fmaf(sl.y, v[0], acc4[1]);
        acc4[2] = fmaf(sl.z, v[0], acc4[2]);
        acc4[3] = fmaf(sl.w, v[0], acc4[3]);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) acc4[t] = fmaf(left_sign(r, l0 + t), v[0], acc4[t]);
      }
    }
    // acc[is_w][k][l]: Z'^T out Z (is_w = 0) and s^T grad y (is_w = 1)
#pragma unroll
    for (int t = 0; t < 4; ++t) atomicAdd(it.acc + is_w * 64 + kj * 8 + l0 + t, (double)acc4[t]);
  }
}

// Per layer: flag when ||Z'^T out Z - s^T grad y||_F > tol ||s^T grad y||_F
// (or when either is not finite); route = products per multiply-add used.
__global__ void pc_flag_kernel(const double* acc, int n, float tol, int* flags, int* route) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const double* a = acc + (size_t)i * 2 * kProbeN * kProbeN;
    double num = 0.0, den = 0.0;
    for (int t = 0; t < kProbeN * kProbeN; ++t) {
      const double d = a[t] - a[64 + t];
      num += d * d;
      den += a[64 + t] * a[64 + t];
    }
    const bool ok = num <= (double)tol * (double)tol * den;  // false for NaN
    flags[i] = ok ? 0 : 1;
    if (route) route[i] = ok ? 3 : 6;
  }
}

// weight -= lr * out for the layers whose flag is 0 (kept at 16 bits): one
// warp per 128-column row segment, four consecutive columns per lane
struct PcWItem {
  const float* out;
  float* w;
  long long ld_out, ld_w, d_out, d_in, unit_begin;
  float lr;
  int flag_idx;
};
constexpr int kPcWMax = 256;
struct PcWParams {
  PcWItem items[kPcWMax];
  const int* flags;
  long long total_units;
  int n;
};

__global__ void __launch_bounds__(256) pc_weight_kernel(const __grid_constant__ PcWParams prm) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (long long u = (long long)blockIdx.x * 8 + warp; u < prm.total_units; u += (long long)gridDim.x * 8) {
    int lo = 0, hi = prm.n;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prm.items[mid].unit_begin <= u)
        lo = mid;
      else
        hi = mid;
    }
    const PcWItem& it = prm.items[lo];
    if (prm.flags[it.flag_idx] != 0) continue;  // recomputed: stepped in the GEMM epilogue
    const long long segs = (it.d_in + 127) / 128;
    const long long local = u - it.unit_begin;
    const long long r = local / segs;
    const long long c = (local - r * segs) * 128 + lane * 4;
    const float* src = it.out + r * it.ld_out + c;
    float* w = it.w + r * it.ld_w + c;
    if (c + 4 <= it.d_in) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      float4 x = *reinterpret_cast<const float4*>(w);
      x.x = __fmaf_rn(-it.lr, v.x, x.x);
      x.y = __fmaf_rn(-it.lr, v.y, x.y);
      x.z = __fmaf_rn(-it.lr, v.z, x.z);
      x.w = __fmaf_rn(-it.lr, v.w, x.w);
      *reinterpret_cast<float4*>(w) = x;
    } else {
      for (int t = 0; t < 4 && c + t < it.d_in; ++t) w[t] = __fmaf_rn(-it.lr, src[t], w[t]);
    }
  }
}

static int launch_weight_step(int n, const kfac_precond_args* args, const int* flags, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  PcWParams* prm = new PcWParams;
  int rc = KFAC_OK;
  int cnt = 0;
  long long total = 0;
  auto flush = [&]() {
    if (cnt == 0 || rc != KFAC_OK) return;
    prm->n = cnt;
    prm->flags = flags;
    prm->total_units = total;
    const long long blocks = (total + 7) / 8, cap = (long long)sms * 8;
    pc_weight_kernel<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, stream>>>(*prm);
    count_launch();
    if (cudaGetLastError() != cudaSuccess) rc = KFAC_ERR_CUDA;
    cnt = 0;
    total = 0;
  };
  for (int i = 0; i < n && rc == KFAC_OK; ++i) {
    const kfac_precond_args& a = args[i];
    if (!a.weight) continue;
    prm->items[cnt] = PcWItem{a.out, a.weight, a.ld_out, a.ld_weight, a.d_out, a.d_in, total, a.lr, i};
    total += a.d_out * ((a.d_in + 127) / 128);
    if (++cnt == kPcWMax) flush();
  }
  flush();
  delete prm;
  return rc;
}

__global__ void pc_route_fill_kernel(int* route, int n, int v) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) route[i] = v;
}

static int launch_check(int n, const PcChkItem* items, cudaStream_t stream, bool compact = false) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  const int sms = device_sm_count(dev);
  PcChkParams* prm = new PcChkParams;
  int rc = KFAC_OK;
  for (int base = 0; base < n && rc == KFAC_OK; base += kChkMax) {
    const int cnt = n - base < kChkMax ? n - base : kChkMax;
    long long total = 0;
    for (int i = 0; i < cnt; ++i) {
      prm->items[i] = items[base + i];
      prm->items[i].unit_begin = total;
      const PcChkItem& it = prm->items[i];
      total += ((it.d_in + 255) / 256) * ((it.d_out + kChkRows - 1) / kChkRows);
    }
    prm->n = cnt;
    prm->total_units = total;
    if (total == 0) continue;
    if (compact) {
      pc_check_kernel<2><<<(unsigned)((total + 1) / 2), 64, 0, stream>>>(*prm);
    } else {
      const long long blocks = (total + 7) / 8, cap = (long long)sms * 8;
      pc_check_kernel<8><<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, stream>>>(*prm);
    }
    count_launch();
    if (cudaGetLastError() != cudaSuccess) rc = KFAC_ERR_CUDA;
  }
  delete prm;
  return rc;
}

// ------------------------------------------------------------------ layer groups
// A large AUTO call runs its layers in groups (contiguous, of about equal GEMM
// work): the GEMMs of group g on a highest-priority stream of the library
// while the split of group g + 1 and the check of group g - 1 run on two
// lowest-priority streams, in blocks small enough to share an SM with a GEMM
// block (the GEMMs are bound by the tensor pipe, the split and the check by
// memory).  Only the first group's split and the last group's check run alone.
constexpr int kPcMaxGroups = 8;
constexpr double kPcGroupWork = 7.0e11;  // GEMM flops (2 M N K) per group, about

struct PcStreams {
  cudaStream_t hi = nullptr, lo = nullptr, lo2 = nullptr;
  cudaEvent_t fork = nullptr, split_done[kPcMaxGroups] = {}, gemm_done[kPcMaxGroups] = {}, hi_done = nullptr,
              chk_done = nullptr;
};

// The streams and events of the caller stream's set, created once (up to four
// caller streams per device); false when no set is free: the call then runs
// in one group on the caller's stream.  A set is not meant for concurrent
// calls from several host threads on the same caller stream.
static bool pc_streams(int dev, cudaStream_t caller, PcStreams* out) {
  constexpr int kSets = 4;
  static std::mutex mu;
  static PcStreams table[64][kSets];
  static cudaStream_t owner[64][kSets];
  if (dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  int slot = -1;
  for (int i = 0; i < kSets && slot < 0; ++i)
    if (table[dev][i].hi && owner[dev][i] == caller) slot = i;
  for (int i = 0; i < kSets && slot < 0; ++i)
    if (!table[dev][i].hi) slot = i;
  if (slot < 0) return false;
  PcStreams& t = table[dev][slot];
  if (!t.hi) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return false;
    PcStreams n;
    cudaEvent_t* evs[] = {&n.fork, &n.hi_done, &n.chk_done};
    for (cudaEvent_t* e : evs)
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    for (int g = 0; g < kPcMaxGroups; ++g)
      if (cudaEventCreateWithFlags(&n.split_done[g], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&n.gemm_done[g], cudaEventDisableTiming) != cudaSuccess)
        return false;
    if (cudaStreamCreateWithPriority(&n.lo, cudaStreamNonBlocking, least) != cudaSuccess ||
        cudaStreamCreateWithPriority(&n.lo2, cudaStreamNonBlocking, least) != cudaSuccess ||
        cudaStreamCreateWithPriority(&n.hi, cudaStreamNonBlocking, greatest) != cudaSuccess)
      return false;
    t = n;
    owner[dev][slot] = caller;
  }
  *out = t;
  return true;
}

// Group boundaries: first[g] .. first[g + 1] - 1; returns the group count.
static int pc_groups(int n, const kfac_precond_args* args, int (&first)[kPcMaxGroups + 1]) {
  double total = 0.0;
  for (int i = 0; i < n; ++i)
    total += 2.0 * (double)args[i].d_in * args[i].d_out * (double)(args[i].d_in + args[i].d_out);
  int G = (int)(total / kPcGroupWork + 0.5);
  G = G < 1 ? 1 : G > kPcMaxGroups ? kPcMaxGroups : G;
  if (G > n) G = n;
  first[0] = 0;
  int g = 1;
  double run = 0.0;
  for (int i = 0; i < n && g < G; ++i) {
    run += 2.0 * (double)args[i].d_in * args[i].d_out * (double)(args[i].d_in + args[i].d_out);
    if (run >= total * g / G && i + 1 < n) first[g++] = i + 1;
  }
  G = g;
  first[G] = n;
  return G;
}

// The 16-bit pass of AUTO (split with probes, both GEMMs, check) in groups;
// on return everything is ordered before the caller's stream's next work.
static int pc_auto_pass_grouped(int G, const int (&first)[kPcMaxGroups + 1], const SplitItem* items,
                                const GtOperand* g1, const GtOperand* g2, const PcChkItem* chk,
                                const PcStreams& ps, cudaStream_t stream) {
  int rc = KFAC_OK;
  auto ok = [&](cudaError_t e) {
    if (e != cudaSuccess && rc == KFAC_OK) rc = KFAC_ERR_CUDA;
    return rc == KFAC_OK;
  };
  if (!ok(cudaEventRecord(ps.fork, stream))) return rc;
  ok(cudaStreamWaitEvent(ps.hi, ps.fork, 0));
  ok(cudaStreamWaitEvent(ps.lo, ps.fork, 0));
  ok(cudaStreamWaitEvent(ps.lo2, ps.fork, 0));
  // the first group's split alone, on the GEMM stream
  if (rc == KFAC_OK) rc = launch_split(items, 3 * first[1], 2, nullptr, ps.hi);
  ok(cudaEventRecord(ps.split_done[0], ps.hi));
  // the other groups' splits, from the first GEMM on
  ok(cudaStreamWaitEvent(ps.lo, ps.split_done[0], 0));
  for (int g = 1; g < G && rc == KFAC_OK; ++g) {
    rc = launch_split(items + 3 * first[g], 3 * (first[g + 1] - first[g]), 2, nullptr, ps.lo, true);
    ok(cudaEventRecord(ps.split_done[g], ps.lo));
  }
  // GEMM launches: GEMM 1 of group 0; then GEMM 2 of group g - 1 together
  // with GEMM 1 of group g (independent problems, one persistent grid); last,
  // GEMM 2 of the last group.  The check of group g follows GEMM 2 of group g.
  GtOperand* ops = new GtOperand[first[G] > 0 ? first[G] : 1];
  for (int g = 0; g <= G && rc == KFAC_OK; ++g) {
    int cnt = 0;
    if (g > 0)
      for (int i = first[g - 1]; i < first[g]; ++i) ops[cnt++] = g2[i];
    if (g < G) {
      for (int i = first[g]; i < first[g + 1]; ++i) ops[cnt++] = g1[i];
      if (g > 0) ok(cudaStreamWaitEvent(ps.hi, ps.split_done[g], 0));
    }
    if (rc == KFAC_OK) rc = launch_gemm_tc(ops, cnt, 2, nullptr, ps.hi);
    if (g > 0) {
      ok(cudaEventRecord(ps.gemm_done[g - 1], ps.hi));
      ok(cudaStreamWaitEvent(ps.lo2, ps.gemm_done[g - 1], 0));
      const int a = first[g - 1];
      if (rc == KFAC_OK) rc = launch_check(first[g] - a, chk + a, ps.lo2, g < G);
    }
  }
  delete[] ops;
  // join (also on failure, so that no side stream is left forked)
  cudaEventRecord(ps.hi_done, ps.hi);
  cudaEventRecord(ps.chk_done, ps.lo2);
  cudaStreamWaitEvent(stream, ps.hi_done, 0);
  cudaStreamWaitEvent(stream, ps.chk_done, 0);
  return rc;
}

// ------------------------------------------------------------------ driver
int launch_precondition(int n, const kfac_precond_args* args, int precision, int* route, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  if (workspace_bytes < precondition_workspace(n, args) || (workspace == nullptr && n > 0)) return KFAC_ERR_WORKSPACE;
  const bool autop = precision == KFAC_PRECOND_AUTO;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SplitItem* items = new SplitItem[3 * (size_t)n];
  GtOperand* g1 = new GtOperand[n];
  GtOperand* g2 = new GtOperand[n];
  PcChkItem* chk = new PcChkItem[n];
  size_t off = 0;
  for (int i = 0; i < n; ++i) off = pc_layout(args[i], off).end;
  const PcProbeLayout PL = pc_probe_layout(n, args, off);
  double* acc = reinterpret_cast<double*>(ws + PL.acc);
  int* flags = reinterpret_cast<int*>(ws + PL.flags);
  off = 0;
  size_t poff = PL.begin;
  for (int i = 0; i < n; ++i) {
    const kfac_precond_args& a = args[i];
    const PcLayout L = pc_layout(a, off);
    off = L.end;
    uint16_t* s_grad = reinterpret_cast<uint16_t*>(ws + L.grad);
    uint16_t* s_ia = reinterpret_cast<uint16_t*>(ws + L.inv_a);
    uint16_t* s_ig = reinterpret_cast<uint16_t*>(ws + L.inv_g);
    uint16_t* s_tmp = reinterpret_cast<uint16_t*>(ws + L.tmp);
    float* y = reinterpret_cast<float*>(ws + poff);
    float* sv = y + kProbeN * a.d_in;
    poff += align256(sizeof(float) * kProbeN * (a.d_in + a.d_out));
    const long long ldi = pad8(a.d_in), ldo = pad8(a.d_out);
    items[3 * i + 0] = SplitItem{a.grad, s_grad, a.d_out, a.d_in, a.ld_grad, ldi, a.d_out * ldi, 0, nullptr, 0, i};
    items[3 * i + 1] = SplitItem{a.inv_a, s_ia, a.d_in, a.d_in, a.ld_a, ldi, a.d_in * ldi, 0, autop ? y : nullptr, 0, i};
    items[3 * i + 2] =
        SplitItem{a.inv_g, s_ig, a.d_out, a.d_out, a.ld_g, ldo, a.d_out * ldo, 0, autop ? sv : nullptr, 8, i};
    // tmp^T[n][m] = sum_k inv_a[n][k] grad[m][k]: M = d_in, N = d_out, K = d_in
    g1[i] = GtOperand{s_ia, s_grad, a.d_in, a.d_out, a.d_in, ldi, ldi, s_tmp, ldo, a.d_in * ldo, 1, 1.0f, i};
    // out[m][n] = sum_k inv_g[m][k] tmp^T[n][k]: M = d_out, N = d_in, K = d_out
    g2[i] = GtOperand{s_ig, s_tmp, a.d_out, a.d_in, a.d_out, ldo, ldo, a.out, a.ld_out, 0, 0, 1.0f, i};
    chk[i] = PcChkItem{a.grad, a.out, y, sv, acc + (size_t)i * 2 * kProbeN * kProbeN,
                       a.ld_grad, a.ld_out, a.d_out, a.d_in, 0};
  }
  GtOperand* g2w = new GtOperand[n];  // GEMM 2 with the weight step
  for (int i = 0; i < n; ++i) {
    g2w[i] = g2[i];
    g2w[i].w = args[i].weight;
    g2w[i].ldw = args[i].ld_weight;
    g2w[i].lr = args[i].lr;
  }
  int rc = KFAC_OK;
  if (!autop) {
    rc = launch_split(items, 3 * n, 3, nullptr, stream);
    if (rc == KFAC_OK) rc = launch_gemm_tc(g1, n, 3, nullptr, stream);
    if (rc == KFAC_OK) rc = launch_gemm_tc(g2w, n, 3, nullptr, stream);
    if (rc == KFAC_OK && route && n > 0) {
      pc_route_fill_kernel<<<(n + 255) / 256, 256, 0, stream>>>(route, n, 6);
      count_launch();
      if (cudaGetLastError() != cudaSuccess) rc = KFAC_ERR_CUDA;
    }
  } else {
    if (cudaMemsetAsync(ws + PL.begin, 0, PL.flags - PL.begin, stream) != cudaSuccess) rc = KFAC_ERR_CUDA;
    int first[kPcMaxGroups + 1];
    const int G = pc_groups(n, args, first);
    int dev = 0;
    PcStreams ps;
    if (rc == KFAC_OK && G > 1 && cudaGetDevice(&dev) == cudaSuccess && pc_streams(dev, stream, &ps)) {
      rc = pc_auto_pass_grouped(G, first, items, g1, g2, chk, ps, stream);
    } else {
      if (rc == KFAC_OK) rc = launch_split(items, 3 * n, 2, nullptr, stream);
      if (rc == KFAC_OK) rc = launch_gemm_tc(g1, n, 2, nullptr, stream);
      if (rc == KFAC_OK) rc = launch_gemm_tc(g2, n, 2, nullptr, stream);
      if (rc == KFAC_OK) rc = launch_check(n, chk, stream);
    }
    if (rc == KFAC_OK) {
      pc_flag_kernel<<<(n + 127) / 128, 128, 0, stream>>>(acc, n, kPcAutoTol, flags, route);
      count_launch();
      if (cudaGetLastError() != cudaSuccess) rc = KFAC_ERR_CUDA;
    }
    for (int i = 0; i < 3 * n; ++i) items[i].probe = nullptr;  // the probes are taken
    if (rc == KFAC_OK) rc = launch_split(items, 3 * n, 3, flags, stream);
    if (rc == KFAC_OK) rc = launch_gemm_tc(g1, n, 3, flags, stream);
    if (rc == KFAC_OK) rc = launch_gemm_tc(g2w, n, 3, flags, stream);
    if (rc == KFAC_OK) rc = launch_weight_step(n, args, flags, stream);
  }
  delete[] items;
  delete[] g1;
  delete[] g2;
  delete[] g2w;
  delete[] chk;
  return rc;
}

}  // namespace kfac
