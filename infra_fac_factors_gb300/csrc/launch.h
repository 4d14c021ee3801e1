// Internal launchers (host side) behind the C ABI of kfac.h.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "kfac.h"

namespace kfac {

int device_sm_count(int dev);
// KFAC_OK when the current device is an sm_103 part, else KFAC_ERR_UNSUPPORTED
// (or KFAC_ERR_CUDA when the runtime cannot tell).
int supported_device();
int* device_status_ptr();
// Counts every kernel launch of the library (reported by kfac_launch_count).
void count_launch();
bool ensure_smem_attr(int dev, const void* fn, int bytes);
// The driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (nullptr when the driver does not provide it).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();
// The driver's cuTensorMapEncodeIm2col (nullptr when not provided).
typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeIm2colFn tensor_map_im2col_encoder();

// Per-launch timing of the main kernels, for kfac_profile / kfac_profile_read:
// when recording is on, prof_begin records an event on the launch's stream
// and prof_end a second one after the launch, with the launch's work.
struct ProfMark {
  cudaEvent_t start = nullptr;
};
void prof_begin(cudaStream_t stream, ProfMark& m);
// Whether kfac_profile is recording (its events cannot be captured in a graph).
bool prof_recording();
void prof_end(int kind, cudaStream_t stream, const ProfMark& m, double work);

int launch_factors(int n, const kfac_factor_args* args, int dtype, int P, int mirror, cudaStream_t stream);
int launch_conv_factors(int n, const kfac_conv_factor_args* args, int P, int mirror, cudaStream_t stream);
int launch_spatial_sum(const void* g, int dtype, int64_t batch, int64_t hw, int64_t C, int64_t ld_g, float* gs,
                       int64_t ld_gs, cudaStream_t stream);
int launch_update_running(int n, const kfac_running_args* args, int P, float decay, float gamma, int first_step,
                          cudaStream_t stream);
size_t inverse_workspace(int n, const kfac_inverse_args* args, int refine);
// The high-priority stream of the caller's auxiliary set (the fp32 sweep's)
// and four of its events, for the fp64 pass that follows the fp32 pass in
// the same call on the same caller stream.
bool fp64_chain_stream(int dev, cudaStream_t caller, cudaStream_t* chain, cudaEvent_t (&ev)[4]);
int launch_damped_inverse(int n, const kfac_inverse_args* args, float gamma_extra, int refine, int* info, int* route,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);
int launch_packed(int n, const kfac_pack_args* args, int unpack, int mirror, cudaStream_t stream);
size_t precondition_workspace(int n, const kfac_precond_args* args);
int launch_precondition(int n, const kfac_precond_args* args, int precision, int* route, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

}  // namespace kfac
