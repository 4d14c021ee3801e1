// extern "C" entry points of kfac.h: host-side argument validation, then the
// launchers.  Nothing here allocates device memory or synchronises the host
// (except kfac_device_status, which documents its synchronisation).
#include <math.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <initializer_list>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tilemap.cuh"

namespace kfac {

namespace {
constexpr int kMaxDev = 64;
std::mutex g_mu;
int g_sms[kMaxDev];
int g_cc_ok[kMaxDev];  // 0 unknown, 1 sm_103, -1 other
int g_smem_set[kMaxDev][16];
const void* g_smem_fn[kMaxDev][16];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool finite(float v) { return isfinite(v) != 0; }
}  // namespace

int device_sm_count(int dev) {
  if (dev < 0 || dev >= kMaxDev) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = v;
  }
  return g_sms[dev];
}

bool ensure_smem_attr(int dev, const void* fn, int bytes) {
  if (dev < 0 || dev >= kMaxDev) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < 16; ++i) {
    if (g_smem_fn[dev][i] == fn && g_smem_set[dev][i] >= bytes) return true;
    if (g_smem_fn[dev][i] == nullptr) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
      g_smem_fn[dev][i] = fn;
      g_smem_set[dev][i] = bytes;
      return true;
    }
  }
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
}

static void* driver_entry(const char* name) {
  cudaDriverEntryPointQueryResult q;
  void* p = nullptr;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return p;
  return nullptr;
}

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(driver_entry("cuTensorMapEncodeTiled"));
  return fn;
}

EncodeIm2colFn tensor_map_im2col_encoder() {
  static EncodeIm2colFn fn = reinterpret_cast<EncodeIm2colFn>(driver_entry("cuTensorMapEncodeIm2col"));
  return fn;
}

// The kernels are built for sm_103a only.
static int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) return KFAC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_cc_ok[dev] == 0) {
    int ma = 0, mi = 0;
    if (cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return KFAC_ERR_CUDA;
    g_cc_ok[dev] = (ma == 10 && mi == 3) ? 1 : -1;
  }
  return g_cc_ok[dev] == 1 ? KFAC_OK : KFAC_ERR_UNSUPPORTED;
}

// Every data pointer of a call must lie in device memory of the current device:
// the tensor maps the kernels load through (some with cluster multicast) must
// cover this GPU's own memory only, and no kernel may touch host-mapped,
// managed or peer memory.  Checked on the host before any launch.
static bool on_device(const void* p, int dev) {
  if (!p) return true;  // optional pointers; required ones are checked for NULL before
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // do not leave the query's error behind for the launch checks
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

static int check_pointers(std::initializer_list<const void*> ptrs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  for (const void* p : ptrs)
    if (!on_device(p, dev)) return KFAC_ERR_INVALID_ARG;
  return KFAC_OK;
}

int supported_device() { return check_device(); }

// An NVTX range around the host side of one call, named after the time
// categories the pages break an iteration into (FactorComp: the Kronecker
// factors; InverseComp: the inverses; and, on one GPU, EMAReduce for the shard
// mean that stands in for the factor all-reduce, with the running average and
// damping, and Precond for the preconditioned gradient).  Profilers show the
// launches of the call under it; without a profiler attached it costs a
// branch.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

int* device_status_ptr();

static std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace kfac

using namespace kfac;

extern "C" {

const char* kfac_status_string(int status) {
  switch (status) {
    case KFAC_OK: return "KFAC_OK";
    case KFAC_ERR_INVALID_ARG: return "KFAC_ERR_INVALID_ARG";
    case KFAC_ERR_NOT_SPD: return "KFAC_ERR_NOT_SPD";
    case KFAC_ERR_CUDA: return "KFAC_ERR_CUDA";
    case KFAC_ERR_UNSUPPORTED: return "KFAC_ERR_UNSUPPORTED";
    case KFAC_ERR_TIMEOUT: return "KFAC_ERR_TIMEOUT";
    case KFAC_ERR_WORKSPACE: return "KFAC_ERR_WORKSPACE";
    default: return "KFAC_ERR_UNKNOWN";
  }
}

int kfac_version(void) { return 100; }

unsigned long long kfac_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

namespace kfac {
// One CTA waits, with the kernels' bounded wait, on an mbarrier that nothing
// arrives on: the wait must give up after `limit` cycles, record
// KFAC_ERR_TIMEOUT in the status word and let the kernel return.
__global__ void wait_selftest_kernel(int* status, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, limit);
  __syncthreads();
}
}  // namespace kfac

extern "C" {

int kfac_wait_selftest(int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1000 || limit_cycles > kfac::kWaitLimitCycles) return KFAC_ERR_INVALID_ARG;
  const int dc = kfac::check_device();
  if (dc != KFAC_OK) return dc;
  int* p = kfac::device_status_ptr();
  if (!p) return KFAC_ERR_CUDA;
  kfac::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(p, (long long)limit_cycles);
  kfac::count_launch();
  return cudaGetLastError() == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA;
}

int kfac_device_status(int* status_out, int clear, void* stream) {
  if (!status_out) return KFAC_ERR_INVALID_ARG;
  int* p = device_status_ptr();
  if (!p) return KFAC_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KFAC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KFAC_ERR_CUDA;
  *status_out = v;
  if (clear && v != 0) {
    if (cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess) return KFAC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return KFAC_OK;
}

int kfac_factors(int n, const kfac_factor_args* args, int dtype, int P, int mirror, void* stream) {
  if (n < 0 || n > 4096 || (n > 0 && !args)) return KFAC_ERR_INVALID_ARG;
  if (dtype != KFAC_BF16 && dtype != KFAC_FP32) return KFAC_ERR_INVALID_ARG;
  if (P < 1 || P > 65535) return KFAC_ERR_INVALID_ARG;
  const int64_t vec = dtype == KFAC_BF16 ? 8 : 4;
  for (int i = 0; i < n; ++i) {
    const kfac_factor_args& a = args[i];
    if (!a.x || !a.out || !aligned16(a.x) || !aligned16(a.out)) return KFAC_ERR_INVALID_ARG;
    if (a.d < 1 || a.d > 65536 || a.rows < P || a.rows % P != 0) return KFAC_ERR_INVALID_ARG;
    if (a.rows / P > (int64_t)1 << 30) return KFAC_ERR_INVALID_ARG;
    if (a.ld_x < a.d || a.ld_x % vec != 0) return KFAC_ERR_INVALID_ARG;
    if (a.ld_out < a.d || a.ld_out % 4 != 0) return KFAC_ERR_INVALID_ARG;
    if (P > 1 && (a.stride_out < a.d * a.ld_out || a.stride_out % 4 != 0)) return KFAC_ERR_INVALID_ARG;
    if (!finite(a.scale)) return KFAC_ERR_INVALID_ARG;
  }
  if (n == 0) return KFAC_OK;
  const int dc = check_device();
  if (dc != KFAC_OK) return dc;
  for (int i = 0; i < n; ++i) {
    const int pc = check_pointers({args[i].x, args[i].out});
    if (pc != KFAC_OK) return pc;
  }
  NvtxRange range("FactorComp");
  return launch_factors(n, args, dtype, P, mirror, static_cast<cudaStream_t>(stream));
}

int kfac_conv_factors(int n, const kfac_conv_factor_args* args, int P, int mirror, void* stream) {
  if (n < 0 || n > 4096 || (n > 0 && !args)) return KFAC_ERR_INVALID_ARG;
  if (P < 1 || P > 65535) return KFAC_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const kfac_conv_factor_args& a = args[i];
    if (!a.x || !a.out || !aligned16(a.x) || !aligned16(a.out)) return KFAC_ERR_INVALID_ARG;
    if (a.C < 64 || a.C > 7232 || a.C % 64 != 0) return KFAC_ERR_INVALID_ARG;
    if (a.B < P || a.B % P != 0 || a.H < 1 || a.W < 1) return KFAC_ERR_INVALID_ARG;
    if (a.H > 0x7fffffff / a.W || a.B > 0x7fffffff / (a.H * a.W)) return KFAC_ERR_INVALID_ARG;
    const int64_t d = 9 * a.C + 1;
    if (a.ld_out < d || a.ld_out % 4 != 0) return KFAC_ERR_INVALID_ARG;
    if (P > 1 && (a.stride_out < d * a.ld_out || a.stride_out % 4 != 0)) return KFAC_ERR_INVALID_ARG;
    if (!finite(a.scale)) return KFAC_ERR_INVALID_ARG;
  }
  if (n == 0) return KFAC_OK;
  const int dc = check_device();
  if (dc != KFAC_OK) return dc;
  for (int i = 0; i < n; ++i) {
    const int pc = check_pointers({args[i].x, args[i].out});
    if (pc != KFAC_OK) return pc;
  }
  NvtxRange range("FactorComp");
  return launch_conv_factors(n, args, P, mirror, static_cast<cudaStream_t>(stream));
}

int kfac_spatial_sum(const void* g, int dtype, int64_t batch, int64_t hw, int64_t C, int64_t ld_g, float* gs,
                     int64_t ld_gs, void* stream) {
  if (dtype != KFAC_BF16 && dtype != KFAC_FP32) return KFAC_ERR_INVALID_ARG;
  const int64_t vec = dtype == KFAC_BF16 ? 8 : 4;
  if (!g || !gs || !aligned16(g) || !aligned16(gs)) return KFAC_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535 || hw < 1 || C < 1) return KFAC_ERR_INVALID_ARG;
  if (ld_g < C || ld_g % vec != 0 || ld_gs < C || ld_gs % 4 != 0) return KFAC_ERR_INVALID_ARG;
  const int dc = check_device();
  if (dc != KFAC_OK) return dc;
  const int pc = check_pointers({g, gs});
  if (pc != KFAC_OK) return pc;
  NvtxRange range("FactorComp");
  return launch_spatial_sum(g, dtype, batch, hw, C, ld_g, gs, ld_gs, static_cast<cudaStream_t>(stream));
}

int kfac_update_running(int n, const kfac_running_args* args, int P, float decay, float gamma, int first_step,
                        void* stream) {
  if (n < 0 || n > 4096 || (n > 0 && !args)) return KFAC_ERR_INVALID_ARG;
  if (P < 1 || P > 65535) return KFAC_ERR_INVALID_ARG;
  if (!finite(decay) || decay < 0.f || decay >= 1.f) return KFAC_ERR_INVALID_ARG;
  if (!finite(gamma) || gamma < 0.f) return KFAC_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const kfac_running_args& a = args[i];
    if (!a.shards || !a.running || !a.damped) return KFAC_ERR_INVALID_ARG;
    if (!aligned16(a.shards) || !aligned16(a.running) || !aligned16(a.damped)) return KFAC_ERR_INVALID_ARG;
    if (a.running == a.damped) return KFAC_ERR_INVALID_ARG;
    if (a.d < 1 || a.d > 65536 || a.ld < a.d || a.ld % 4 != 0) return KFAC_ERR_INVALID_ARG;
    if (P > 1 && (a.stride_shard < a.d * a.ld || a.stride_shard % 4 != 0)) return KFAC_ERR_INVALID_ARG;
  }
  if (n == 0) return KFAC_OK;
  const int dc = check_device();
  if (dc != KFAC_OK) return dc;
  for (int i = 0; i < n; ++i) {
    const int pc = check_pointers({args[i].shards, args[i].running, args[i].damped});
    if (pc != KFAC_OK) return pc;
  }
  NvtxRange range("EMAReduce");
  return launch_update_running(n, args, P, decay, gamma, first_step, static_cast<cudaStream_t>(stream));
}

static bool inverse_args_ok(int n, const kfac_inverse_args* args, int refine) {
  if (n < 0 || n > 4096 || (n > 0 && !args)) return false;
  if (refine < KFAC_REFINE_NONE || refine > KFAC_REFINE_ALWAYS) return false;
  for (int i = 0; i < n; ++i) {
    const kfac_inverse_args& a = args[i];
    if (!a.damped || !a.inv || !aligned16(a.damped) || !aligned16(a.inv)) return false;
    if ((const void*)a.damped == (const void*)a.inv) return false;
    if (a.d < 1 || a.d > 65536) return false;
    if (a.ld_in < a.d || a.ld_in % 4 != 0 || a.ld_out < a.d || a.ld_out % 4 != 0) return false;
  }
  return true;
}

size_t kfac_damped_inverse_workspace(int n, const kfac_inverse_args* args, int refine) {
  if (!inverse_args_ok(n, args, refine)) return 0;
  return inverse_workspace(n, args, refine);
}

int kfac_damped_inverse(int n, const kfac_inverse_args* args, float gamma_extra, int refine, int* info, int* route,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!inverse_args_ok(n, args, refine)) return KFAC_ERR_INVALID_ARG;
  if (!finite(gamma_extra) || gamma_extra < 0.f) return KFAC_ERR_INVALID_ARG;
  if (n > 0 && (!info || (reinterpret_cast<uintptr_t>(info) & 3))) return KFAC_ERR_INVALID_ARG;
  if (route && (reinterpret_cast<uintptr_t>(route) & 3)) return KFAC_ERR_INVALID_ARG;
  if (n == 0) return KFAC_OK;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return KFAC_ERR_WORKSPACE;
  if (workspace_bytes < inverse_workspace(n, args, refine)) return KFAC_ERR_WORKSPACE;
  const int dc = check_device();
  if (dc != KFAC_OK) return dc;
  int pc = check_pointers({info, route, workspace});
  for (int i = 0; i < n && pc == KFAC_OK; ++i) pc = check_pointers({args[i].damped, args[i].inv});
  if (pc != KFAC_OK) return pc;
  NvtxRange range("InverseComp");
  return launch_damped_inverse(n, args, gamma_extra, refine, info, route, workspace, workspace_bytes,
                               static_cast<cudaStream_t>(stream));
}

static bool precond_args_ok(int n, const kfac_precond_args* args) {
  if (n < 0 || n > 4096 || (n > 0 && !args)) return false;
  for (int i = 0; i < n; ++i) {
    const kfac_precond_args& a = args[i];
    if (!a.inv_g || !a.grad || !a.inv_a || !a.out) return false;
    if (!aligned16(a.inv_g) || !aligned16(a.grad) || !aligned16(a.inv_a) || !aligned16(a.out)) return false;
    if (a.d_out < 1 || a.d_in < 1 || a.d_out > 65536 || a.d_in > 65536) return false;
    if (a.ld_g < a.d_out || a.ld_grad < a.d_in || a.ld_a < a.d_in || a.ld_out < a.d_in) return false;
    if (a.ld_g % 4 || a.ld_grad % 4 || a.ld_a % 4 || a.ld_out % 4) return false;
    if ((const void*)a.out == (const void*)a.grad || (const void*)a.out == (const void*)a.inv_a ||
        (const void*)a.out == (const void*)a.inv_g)
      return false;
    if (a.weight) {
      if (!aligned16(a.weight) || a.ld_weight < a.d_in || a.ld_weight % 4) return false;
      const void* w = a.weight;
      if (w == (const void*)a.out || w == (const void*)a.grad || w == (const void*)a.inv_a ||
          w == (const void*)a.inv_g)
        return false;
    }
  }
  return true;
}

size_t kfac_precondition_workspace(int n, const kfac_precond_args* args) {
  if (!precond_args_ok(n, args)) return 0;
  return precondition_workspace(n, args);
}

int kfac_precondition(int n, const kfac_precond_args* args, int precision, int* route, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!precond_args_ok(n, args)) return KFAC_ERR_INVALID_ARG;
  if (precision != KFAC_PRECOND_FP32 && precision != KFAC_PRECOND_AUTO) return KFAC_ERR_INVALID_ARG;
  if (route && (reinterpret_cast<uintptr_t>(route) & 3)) return KFAC_ERR_INVALID_ARG;
  if (n == 0) return KFAC_OK;
  if (!workspace || !aligned16(workspace)) return KFAC_ERR_WORKSPACE;
  if (workspace_bytes < precondition_workspace(n, args)) return KFAC_ERR_WORKSPACE;
  const int dc = check_device();
  if (dc != KFAC_OK) return dc;
  int pc = check_pointers({route, workspace});
  for (int i = 0; i < n && pc == KFAC_OK; ++i)
    pc = check_pointers({args[i].inv_g, args[i].grad, args[i].inv_a, args[i].out, args[i].weight});
  if (pc != KFAC_OK) return pc;
  NvtxRange range("Precond");
  return launch_precondition(n, args, precision, route, workspace, workspace_bytes,
                             static_cast<cudaStream_t>(stream));
}

static int packed_call(int n, const kfac_pack_args* args, int unpack, int mirror, void* stream) {
  if (n < 0 || n > 4096 || (n > 0 && !args)) return KFAC_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const kfac_pack_args& a = args[i];
    if (!a.mat || !a.packed || !aligned16(a.mat) || (reinterpret_cast<uintptr_t>(a.packed) & 3))
      return KFAC_ERR_INVALID_ARG;
    if (a.d < 1 || a.d > 65536 || a.ld < a.d || a.ld % 4 != 0) return KFAC_ERR_INVALID_ARG;
    // the two buffers must not overlap: [mat, mat + (d-1) ld + d) and [packed, packed + d(d+1)/2)
    const uintptr_t m0 = reinterpret_cast<uintptr_t>(a.mat), p0 = reinterpret_cast<uintptr_t>(a.packed);
    const uintptr_t m1 = m0 + (uintptr_t)((a.d - 1) * a.ld + a.d) * 4, p1 = p0 + (uintptr_t)(a.d * (a.d + 1) / 2) * 4;
    if (m0 < p1 && p0 < m1) return KFAC_ERR_INVALID_ARG;
  }
  if (n == 0) return KFAC_OK;
  const int dc = check_device();
  if (dc != KFAC_OK) return dc;
  for (int i = 0; i < n; ++i) {
    const int pc = check_pointers({args[i].mat, args[i].packed});
    if (pc != KFAC_OK) return pc;
  }
  NvtxRange range(unpack ? "UnpackUpper" : "PackUpper");
  return launch_packed(n, args, unpack, mirror, static_cast<cudaStream_t>(stream));
}

int kfac_pack_upper(int n, const kfac_pack_args* args, void* stream) { return packed_call(n, args, 0, 0, stream); }

int kfac_unpack_upper(int n, const kfac_pack_args* args, int mirror, void* stream) {
  return packed_call(n, args, 1, mirror != 0, stream);
}

int kfac_factor_tile_map(int64_t d, int64_t capacity, int32_t* row_block, int64_t* col_start, int32_t* width,
                         int64_t* count) {
  if (d < 1 || d > 65536 || capacity < 0 || !count) return KFAC_ERR_INVALID_ARG;
  if (capacity > 0 && (!row_block || !col_start || !width)) return KFAC_ERR_INVALID_ARG;
  const int64_t total = factor_units(d);
  *count = total;
  const int64_t n = total < capacity ? total : capacity;
  for (int64_t t = 0; t < n; ++t) {
    int i, w;
    int64_t j0;
    factor_unit(d, t, i, j0, w);
    row_block[t] = i;
    col_start[t] = j0;
    width[t] = w;
  }
  return KFAC_OK;
}

}  // extern "C"
