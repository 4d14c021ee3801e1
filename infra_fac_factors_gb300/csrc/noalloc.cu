// kfac_precondition_static: the preconditioning step with its scratch memory
// inside the library, for callers that cannot allocate device memory.
//
// kfac_precondition needs a caller-provided workspace (the bf16 slices of its
// operands).  Some callers cannot provide one: their device memory is owned by
// another allocator (for example a framework's caching allocator that must
// account for every byte), or their hot path must not allocate at all, since
// cudaMalloc can synchronise the device and can fail.  This entry point uses a
// fixed scratch array that the library itself holds instead.
//
// The array (kStaticScratchBytes = 64 MiB) is a file-scope __device__
// variable: every GPU that loads the library holds it until the process exits.
// Its device address is looked up once per device (cudaGetSymbolAddress, with
// that device current) by the first call on that device; that first call
// should therefore come before any stream capture.  The address is kept for
// the life of the process: after cudaDeviceReset the library's module is
// loaded again and the kept address no longer holds, so a process that resets
// a device must not call this entry point on it afterwards.  Every call shares the
// array and it keeps the previous call's contents (nothing in it has to start
// at zero: each call writes its scratch before reading it), so calls that
// overlap on the GPU (for example on two streams at once) race.
#include <mutex>

#include "launch.h"

namespace kfac {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)64 << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_precond_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (nullptr on failure).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_precond_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace kfac

extern "C" {

size_t kfac_precondition_static_capacity(void) { return kfac::kStaticScratchBytes; }

int kfac_precondition_static(int n, const kfac_precond_args* args, int precision, int* route, void* stream) {
  if (n < 0 || (n > 0 && !args)) return KFAC_ERR_INVALID_ARG;
  if (n == 0) return kfac_precondition(0, args, precision, route, nullptr, 0, stream);
  const size_t need = kfac_precondition_workspace(n, args);
  if (need == 0) return KFAC_ERR_INVALID_ARG;  // the query rejects invalid arguments
  if (need > kfac::kStaticScratchBytes) return KFAC_ERR_WORKSPACE;
  const int dc = kfac::supported_device();  // before the symbol lookup: a non-sm_103 device has no kernels
  if (dc != KFAC_OK) return dc;
  void* scratch = kfac::scratch_address();
  if (!scratch) return KFAC_ERR_CUDA;
  return kfac_precondition(n, args, precision, route, scratch, kfac::kStaticScratchBytes, stream);
}

}  // extern "C"
