/*
 * kfac.h -- C ABI of the GB300 (sm_103a) K-FAC preconditioning step.
 *
 * The step follows "Accelerating Distributed K-FAC with Smart Parallelism of
 * Computing and Communication Tasks" (SPD-KFAC):
 *   1. kfac_factors        per-worker Kronecker factors A^p = a_p^T a_p / rows_p
 *                          and G^p = g_p^T g_p / rows_p            (§II-B, Eq. (7), (8))
 *   2. kfac_update_running mean over the P workers (the D-KFAC aggregation,
 *                          §II-C), running average over steps, Tikhonov
 *                          damping R + gamma*I                      (§II-B damped update rule)
 *   3. kfac_damped_inverse (A + gamma I)^-1, (G + gamma I)^-1 through a
 *                          Cholesky decomposition                   (§III-B, §IV)
 *   4. kfac_precondition   (G + gamma I)^-1 grad (A + gamma I)^-1   (§II-B damped update rule)
 *
 * Conventions shared by every call
 *   - All matrices are row-major.  "ld" is the leading dimension in elements.
 *   - Every data pointer is a DEVICE pointer into memory of the CURRENT
 *     device (cudaMemoryTypeDevice), 16-byte aligned; host, host-mapped,
 *     managed and peer pointers are refused with KFAC_ERR_INVALID_ARG before
 *     any launch.  Every array of argument structs is a HOST array that is
 *     read during the call only.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream), never synchronise the host, and never
 *     allocate device memory.  Scratch memory is caller-provided ("workspace")
 *     and sized by the matching *_workspace query.
 *   - The caller owns every buffer.  Nothing is retained between calls, so the
 *     K-FAC state (the running factors) lives in caller buffers.
 *   - Argument errors are detected on the host before any launch and return
 *     KFAC_ERR_INVALID_ARG; a failed launch returns KFAC_ERR_CUDA.  Numerical
 *     failure of an inverse is reported per matrix in a device `info` array.
 *   - Symmetric factors are produced and consumed as UPPER TILES: with the
 *     128-row tile grid, element (r, c) belongs to an upper tile when
 *     c >= 128 * floor(r / 128).  Elements of lower tiles are not written by
 *     kfac_factors / kfac_update_running (unless `mirror` is set) and are
 *     never read by kfac_update_running / kfac_damped_inverse.
 *   - Device kernels never trap.  A device-side wait that runs past its limit
 *     (a scheduling bug, never expected) records KFAC_ERR_TIMEOUT in a device
 *     status word, read and cleared with kfac_device_status().
 *
 * Not thread-safe for concurrent calls on the same stream's buffers (the
 * caller orders its own buffers); calls on independent buffers may run on
 * different streams.
 */
#ifndef KFAC_GB300_H
#define KFAC_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status */
enum kfac_status {
  KFAC_OK = 0,
  KFAC_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or parameter      */
  KFAC_ERR_NOT_SPD = 2,     /* only as a value of info[] semantics, see below */
  KFAC_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed    */
  KFAC_ERR_UNSUPPORTED = 4, /* device is not sm_103 / feature unavailable     */
  KFAC_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (device status)  */
  KFAC_ERR_WORKSPACE = 6    /* workspace NULL or smaller than the query       */
};

enum kfac_dtype { KFAC_BF16 = 0, KFAC_FP32 = 1 };

/* Human-readable name of a status code (static string, never NULL). */
const char* kfac_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int kfac_version(void);

/* Number of CUDA kernels this library has launched in this process so far
 * (all devices, all streams).  For accounting only; host only. */
unsigned long long kfac_launch_count(void);

/* Read the device status word (KFAC_OK or KFAC_ERR_TIMEOUT) recorded by any
 * kernel of this library on the current device; clears it when `clear` != 0.
 * Synchronises `stream`. */
int kfac_device_status(int* status_out, int clear, void* stream);

/* Per-launch timing of the library's main kernels (no counterpart on the
 * pages; a measurement aid).  kfac_profile(1) clears the record and starts
 * recording: every later launch of the kernels below gets a CUDA event on
 * its stream just before and just after it, and its work is noted;
 * kfac_profile(0) stops recording.  kfac_profile_read synchronises on the
 * recorded events and returns, for one kind, the number of launches, the sum
 * of their durations (ms; launches on concurrent streams overlap other work)
 * and the sum of their work:
 *   KFAC_K_SYRK        factor SYRK (tensor cores)      work: algorithmic flops, 2 rows d(d+1)/2 per shard
 *   KFAC_K_RUNNING     running average + damping       work: algorithmic bytes, (P+3) 4 d(d+1)/2 per factor
 *   KFAC_K_INV_PANEL   inverse panel products          work: flops of the tile products (2 per multiply-add)
 *   KFAC_K_INV_UPDATE  inverse trailing updates        work: as above
 *   KFAC_K_INV_LAUUM   inverse X = U U^T               work: as above
 *   KFAC_K_GEMM16      preconditioning GEMMs, 16-bit   work: 2 M N K per problem
 *   KFAC_K_GEMM24      preconditioning GEMMs, 24-bit   work: 2 M N K per problem run
 *   KFAC_K_CONV_SYRK   conv factor SYRK (implicit im2col) work: as KFAC_K_SYRK, rows = patch rows
 *   KFAC_K_INV_DIAG    inverse: 128 x 128 diagonal blocks (CUDA cores)  work: 0
 *   KFAC_K_INV_PREP    inverse: block-column slicing (CUDA cores)       work: 0
 *   KFAC_K_INV_AUX     inverse: load, operand width, norms, residual probe, flags (CUDA cores)  work: 0
 *   KFAC_K_INV_NEWTON  inverse: the Newton step of AUTO (slicing, exact products, symmetrisation)  work: 0
 * Recording holds at most 65536 launches (later ones are not recorded).
 * Invalid kind: KFAC_ERR_INVALID_ARG.
 * kfac_profile_count gives the number of recorded launches and
 * kfac_profile_launch the i-th of them (in the order they were issued): its
 * kind, its start and end (ms after the start of the first recorded launch,
 * so launches on concurrent streams line up on one time axis) and its work;
 * both synchronise on the recorded events.  i out of range:
 * KFAC_ERR_INVALID_ARG.                                                      */
typedef enum {
  KFAC_K_SYRK = 0, KFAC_K_RUNNING = 1, KFAC_K_INV_PANEL = 2, KFAC_K_INV_UPDATE = 3,
  KFAC_K_INV_LAUUM = 4, KFAC_K_GEMM16 = 5, KFAC_K_GEMM24 = 6, KFAC_K_CONV_SYRK = 7,
  KFAC_K_INV_DIAG = 8, KFAC_K_INV_PREP = 9, KFAC_K_INV_AUX = 10, KFAC_K_INV_NEWTON = 11,
  KFAC_K_COUNT = 12
} kfac_kernel_kind;
int kfac_profile(int enable);
int kfac_profile_read(int kind, int64_t* launches, double* ms, double* work);
int kfac_profile_count(int64_t* count);
int kfac_profile_launch(int64_t i, int* kind, double* start_ms, double* end_ms, double* work);

/* Failure-detection self-test (no counterpart on the pages; a property of the
 * library): launches one CTA that waits, with the same bounded wait every
 * tcgen05 kernel of the library uses, on an mbarrier that nothing arrives on.
 * After limit_cycles SM clock cycles the wait gives up, the kernel records
 * KFAC_ERR_TIMEOUT in the device status word (see kfac_device_status) and
 * returns; the context stays usable.  limit_cycles in [1000, 4e9] (the
 * kernels' own limit), else KFAC_ERR_INVALID_ARG.  Asynchronous on stream.  */
int kfac_wait_selftest(int64_t limit_cycles, void* stream);

/* -------------------------------------------------------- 1. factors (a1, a2)
 * Per-worker Kronecker factors (§II-B, Eq. (7)/(8); §II-C local factors).
 * For each problem, x holds `rows` rows split into P equal contiguous shards
 * of rows_p = rows / P rows (worker p owns rows [p*rows_p, (p+1)*rows_p)):
 *
 *     out[p] = scale * x_p^T x_p          (d x d, fp32, p = 0..P-1)
 *
 * with out[p] = out + p * stride_out.  Use scale = 1/rows_p for the mean of
 * the paper's factors.  Only upper tiles are written (see conventions); with
 * mirror != 0 the lower tiles are written too, giving full symmetric output.
 *
 * x: KFAC_BF16 -> tcgen05 tensor cores (bf16 products, fp32 accumulation),
 *               ld_x % 8 == 0;
 *    KFAC_FP32 -> fp32 CUDA-core path (exact fp32 products), ld_x % 4 == 0.
 * out: ld_out % 4 == 0, ld_out >= d, stride_out >= d * ld_out (or 0 if P == 1).
 * Limits per call: n <= 4096 problems, 1 <= d <= 65536, rows % P == 0.
 */
typedef struct {
  const void* x;       /* device, rows x d, element type = dtype */
  int64_t rows;        /* total rows of all P shards             */
  int64_t d;           /* factor dimension                       */
  int64_t ld_x;        /* leading dimension of x (elements)      */
  float* out;          /* device, P fp32 matrices d x d          */
  int64_t ld_out;      /* leading dimension of out (elements)    */
  int64_t stride_out;  /* elements between out[p] and out[p+1]   */
  float scale;         /* multiplies x_p^T x_p                   */
} kfac_factor_args;

int kfac_factors(int n, const kfac_factor_args* args, int dtype, int P,
                 int mirror, void* stream);

/* Conv helper for the G factor of a conv layer (the pages do not describe
 * conv factors; the per-sample spatial sum is the reading taken):
 *     gs[b, c] = sum_{s < hw} g[b*hw + s, c]     (fp32 accumulate and out)
 * g: batch*hw x C, dtype bf16 (ld_g % 8 == 0) or fp32 (ld_g % 4 == 0);
 * gs: batch x C fp32, ld_gs % 4 == 0.                                       */
int kfac_spatial_sum(const void* g, int dtype, int64_t batch, int64_t hw,
                     int64_t C, int64_t ld_g, float* gs, int64_t ld_gs,
                     void* stream);

/* Conv factor A straight from the activations (implicit im2col; the pages do
 * not describe conv factors: the reading taken is the Kronecker factor of a
 * 3 x 3 convolution, stride 1, zero padding 1, with bias, whose per-position
 * input is its 3 x 3 x C patch, §II-B Eq. (7)).  For each problem the patch
 * matrix X has one row per output position (b, h, w), in that order, and
 * d = 9 C + 1 columns:
 *     X[(b,h,w), (dh*3 + dw)*C + c] = x[b, h+dh-1, w+dw-1, c]  (0 outside),
 *     X[(b,h,w), 9C] = 1.
 * Worker p owns images [p*B/P, (p+1)*B/P), i.e. patch rows
 * [p*rows_p, (p+1)*rows_p) with rows_p = (B/P) H W, and
 *     out[p] = scale * X_p^T X_p          (d x d, fp32)
 * exactly as kfac_factors would give on the materialised X (bf16 products,
 * fp32 accumulation, the same upper tiles written, `mirror` as there); X is
 * never formed in memory.
 * x: device, bf16, NHWC [B][H][W][C] contiguous, 16-byte aligned, C % 64 == 0,
 *    64 <= C <= 7232 (d <= 65089); B % P == 0; B H W <= 2^31 - 1.
 * out: as kfac_factors (ld_out % 4 == 0, ld_out >= d, stride_out >= d ld_out
 *    and % 4 == 0 when P > 1).  n <= 4096.  Errors: KFAC_ERR_INVALID_ARG.   */
typedef struct {
  const void* x;       /* device, bf16 NHWC activations of all P workers  */
  int64_t B, H, W, C;  /* images, height, width, channels                 */
  float* out;          /* device, P fp32 matrices d x d, d = 9 C + 1      */
  int64_t ld_out;      /* leading dimension of out (elements)             */
  int64_t stride_out;  /* elements between out[p] and out[p+1]            */
  float scale;         /* multiplies X_p^T X_p                            */
} kfac_conv_factor_args;

int kfac_conv_factors(int n, const kfac_conv_factor_args* args, int P,
                      int mirror, void* stream);

/* --------------------------------------- 2. reduce + running average + damp (a3)
 * One fused pass over the upper tiles of each factor (§II-C aggregation,
 * §II-B damping):
 *     F = (1/P) sum_p shards[p]
 *     running = first_step ? F : decay * running + (1 - decay) * F
 *     damped  = running + gamma * I
 * shards[p] = shards + p * stride_shard.  shards, running and damped share
 * `ld` (ld % 4 == 0, ld >= d).  running is read only when first_step == 0.
 * 0 <= decay < 1, gamma >= 0.  n <= 4096.                                    */
typedef struct {
  const float* shards;  /* device, P fp32 d x d matrices (upper tiles read) */
  int64_t stride_shard; /* elements between shards[p] and shards[p+1]       */
  float* running;       /* device, in/out running average (upper tiles)     */
  float* damped;        /* device, out running + gamma I (upper tiles)      */
  int64_t d;
  int64_t ld;
} kfac_running_args;

int kfac_update_running(int n, const kfac_running_args* args, int P,
                        float decay, float gamma, int first_step, void* stream);

/* ------------------------------------------------------ 3. damped inverse (a4)
 * Batched inverse of damped SPD factors through a Cholesky decomposition
 * (§IV: cuSolver-style Cholesky-based inverse; §III-B: the damped inverses):
 *     D_i + gamma_extra * I = L L^T,   inv_i = L^-T L^-1
 * computed with a blocked right-looking Cholesky (128-wide panels) fused with
 * the blocked triangular inverse, then inv = W^T W with W = L^-1.  Only the
 * upper triangle (incl. diagonal) of D_i is read.  inv_i is written as a full,
 * exactly symmetric matrix (§IV: the inverse of a symmetric factor is
 * symmetric).  Matrices may have different sizes.
 *
 * refine: KFAC_REFINE_NONE   fp32 arithmetic for every matrix (tile products
 *                            on tensor cores with 24-bit operands: three bf16
 *                            slices, six MMAs per multiply-add);
 *         KFAC_REFINE_AUTO   fp32, with 16-bit operands (two slices, three
 *                            MMAs) for a matrix whose Gershgorin discs bound its
 *                            condition number by 16 and 24-bit ones otherwise;
 *                            a matrix whose residual ||inv D - I||_F / sqrt(d),
 *                            estimated with four random +-1 probes, exceeds
 *                            2.5e-4, or whose ||D||_1 / min_j L_jj^2 exceeds
 *                            3e5, then gets one Newton step
 *                            inv + inv (I - D inv) on tensor cores, its
 *                            residual formed exactly (error-free bf16 slices),
 *                            and is recomputed in fp64 when the step's
 *                            estimated residual still exceeds 5e-4 or when its
 *                            fp32 factorisation failed;
 *         KFAC_REFINE_ALWAYS fp64 arithmetic for every matrix.
 * info: device int[n]; info[i] = 0 on success, k > 0 when the k-th pivot
 *       (1-based) is not positive (LAPACK potrf convention); inv_i is then
 *       unspecified.  route (device int[n], may be NULL): 0 when inv_i came
 *       from the fp32 pass with 24-bit operands, 2 with 16-bit operands, 3
 *       from the Newton step after it, 1 from the fp64 pass.
 * ld_in, ld_out % 4 == 0.  n <= 4096, 1 <= d <= 65536.
 * Workspace: kfac_damped_inverse_workspace(n, args, refine) bytes, 256-byte
 * aligned, fully overwritten (no initialisation needed).
 * Streams: part of the work runs on streams that the library creates once
 * (two of highest and one of lowest priority, with their events), forked
 * from `stream` after the work already queued there and joined back into
 * `stream` before the call returns, so ordering on `stream` is as for a
 * single-stream call.  Each caller stream gets its own set (up to four per
 * device), so inverses issued on different streams overlap; calls on further
 * caller streams run on their own stream alone (the same results, without the
 * look-ahead).  A set is not meant for concurrent calls from several host
 * threads on the same caller stream.
 * Graphs: with KFAC_REFINE_AUTO the Newton step and the fp64 pass are
 * launched as one CUDA graph whose conditional nodes skip them when no matrix
 * is flagged (device-side decision, no host synchronisation).  The library
 * builds it on the first call for a given batch size, largest block count and
 * workspace address, and keeps it for the process (up to 64 such graphs per
 * process; further calls, calls while kfac_profile records, and calls on a
 * stream that is being captured launch the passes one by one, with the same
 * results).                                                                  */
enum kfac_refine { KFAC_REFINE_NONE = 0, KFAC_REFINE_AUTO = 1, KFAC_REFINE_ALWAYS = 2 };

typedef struct {
  const float* damped;  /* device, d x d fp32 (upper triangle read) */
  float* inv;           /* device, d x d fp32 out (full symmetric)  */
  int64_t d;
  int64_t ld_in;
  int64_t ld_out;
} kfac_inverse_args;

size_t kfac_damped_inverse_workspace(int n, const kfac_inverse_args* args, int refine);

int kfac_damped_inverse(int n, const kfac_inverse_args* args, float gamma_extra,
                        int refine, int* info, int* route, void* workspace,
                        size_t workspace_bytes, void* stream);

/* -------------------------------------------------------- 4. precondition (a5)
 * Preconditioned gradient of each layer (§II-B damped update rule):
 *     out = inv_g * grad * inv_a        (d_out x d_out)(d_out x d_in)(d_in x d_in)
 * inv_g and inv_a must be full symmetric matrices (as kfac_damped_inverse
 * writes them).  All fp32; every ld % 4 == 0.  out must not alias an input.
 * Workspace: kfac_precondition_workspace(n, args) bytes (bf16 slices of the
 * operands and of grad * inv_a, probe vectors, flags), 16-byte aligned.
 *
 * precision: the products run on bf16 tensor cores with each fp32 operand
 * cut into bf16 slices, summed in fp32 with round-to-nearest every twelve MMAs.
 *   KFAC_PRECOND_FP32  all 24 bits of every operand (six MMAs per multiply-add)
 *                      for every layer: close to an fp32 FMA loop.
 *   KFAC_PRECOND_AUTO  16-bit operands (three MMAs), then every layer's result
 *                      is checked with eight random +-1 probes on each side
 *                      (the 8 x 8 bilinear forms Z'^T out Z against
 *                      (inv_g Z')^T grad (inv_a Z), which estimate the relative
 *                      Frobenius error of out); a layer whose estimate exceeds
 *                      4e-4, or is not finite, is recomputed as with FP32.
 * route: NULL, or a device int[n] receiving, per layer, the MMAs per
 * multiply-add its result came from (3 or 6).  Invalid precision, or a route
 * pointer not 4-byte aligned, returns KFAC_ERR_INVALID_ARG.
 * Streams: an AUTO call with more than about 1 TFLOP of GEMM work runs its
 * 16-bit pass in groups of layers on three streams that the library creates
 * once per caller stream (up to four caller streams per device; further ones
 * run the call on `stream` alone), forked from `stream` and joined back into
 * it before the call returns: ordering on `stream` is as for a single-stream
 * call.  A set is not meant for concurrent calls from several host threads on
 * the same caller stream.                                                    */
typedef struct {
  const float* inv_g;  int64_t ld_g;
  const float* grad;   int64_t ld_grad;
  const float* inv_a;  int64_t ld_a;
  float* out;          int64_t ld_out;
  int64_t d_out;
  int64_t d_in;
  /* Optional fused weight step (§II-B, the damped update rule: the weights move
   * by -lr times the preconditioned gradient).  When `weight` is not NULL the
   * call also performs weight[r][c] -= lr * out[r][c] (one fp32 fused
   * multiply-add per element) for r < d_out, c < d_in, once per call with the
   * final out: in the epilogue of the GEMM that produces it (FP32, and the
   * layers AUTO recomputes), or in an elementwise pass over the stored out
   * after the check (the layers AUTO keeps at 16 bits).  weight is fp32
   * d_out x d_in row-major, ld_weight >= d_in, ld_weight % 4 == 0, 16-byte
   * aligned, and must not alias out or an input.  NULL: no weight step.     */
  float* weight;       int64_t ld_weight;
  float lr;
} kfac_precond_args;

size_t kfac_precondition_workspace(int n, const kfac_precond_args* args);

typedef enum { KFAC_PRECOND_FP32 = 0, KFAC_PRECOND_AUTO = 1 } kfac_precond_precision;

int kfac_precondition(int n, const kfac_precond_args* args, int precision, int* route,
                      void* workspace, size_t workspace_bytes, void* stream);

/* The same preconditioning with no caller-provided workspace and no device
 * allocation, for callers that cannot allocate device memory (their device
 * memory is owned by another allocator, or their hot path must not allocate:
 * cudaMalloc can synchronise the device and can fail).  The paper has no
 * counterpart; this is a property of the library.
 * The scratch is a fixed array inside the library of
 * kfac_precondition_static_capacity() bytes (64 MiB), held by every GPU that
 * loads the library until the process exits.  A call whose
 * kfac_precondition_workspace() exceeds it returns KFAC_ERR_WORKSPACE before
 * any launch.  The first call on a device looks up the array's address on
 * that device (cudaGetSymbolAddress), so make it before any stream capture;
 * the address is kept for the process, so do not call this entry point on a
 * device after cudaDeviceReset of that device.
 * All calls share the array and it keeps the last call's contents; calls that
 * overlap on the GPU (e.g. on two streams at once) race.  Otherwise as
 * kfac_precondition.                                                         */
size_t kfac_precondition_static_capacity(void);
int kfac_precondition_static(int n, const kfac_precond_args* args, int precision,
                             int* route, void* stream);

/* --------------------------------------------------- packed upper triangles
 * A symmetric factor or inverse travels as its d(d+1)/2 upper-triangle
 * elements, and small factors are fused into one message (§III-A: the
 * communicated elements of a symmetric Kronecker factor, tensor fusion of
 * factors, Eq. (14)/(15), Fig. 4; §IV: only the upper triangle of the
 * symmetric inverse is sent).  Layout: row-major packed upper triangle,
 *     packed[r*d - r*(r-1)/2 + (c - r)] = M[r][c]      0 <= r <= c < d,
 * i.e. row r holds the d - r elements M[r][r..d-1].
 * kfac_pack_upper   packed <- upper triangle of mat (reads c >= r only);
 * kfac_unpack_upper upper triangle of mat <- packed; with mirror != 0 the
 *                   strict lower triangle of mat too (M[c][r] = M[r][c]), so
 *                   mat becomes the full symmetric matrix.  Other elements of
 *                   mat (padding columns) are not touched.
 * All matrices of a call are moved by one launch (the fused pass; give
 * consecutive `packed` pointers, e.g. base + prefix sums of d(d+1)/2, to get one
 * contiguous buffer).  mat: device fp32 d x d, ld >= d, ld % 4 == 0, 16-byte
 * aligned; packed: device fp32, d(d+1)/2 elements, 4-byte aligned, not
 * overlapping mat.  n <= 4096, 1 <= d <= 65536.  Errors: KFAC_ERR_INVALID_ARG
 * before any launch.  Asynchronous on stream.                               */
typedef struct {
  float* mat;      /* device, d x d fp32 (read by pack, written by unpack)  */
  int64_t d;
  int64_t ld;      /* leading dimension of mat (elements)                   */
  float* packed;   /* device, d(d+1)/2 fp32 (written by pack, read by unpack) */
} kfac_pack_args;

int kfac_pack_upper(int n, const kfac_pack_args* args, void* stream);
int kfac_unpack_upper(int n, const kfac_pack_args* args, int mirror, void* stream);

/* ------------------------------------------------------------- index tables
 * The work units kfac_factors uses to cover the upper tiles of a d x d factor
 * on the tensor-core path (one per CTA of a CTA pair): row blocks 2s and
 * 2s + 1 both take the columns [256 s, d) cut into chunks of at most 256;
 * units 2v and 2v + 1 are the two row blocks of chunk v.  A unit stores only
 * its columns >= 128 i of an existing row block i (row block 2s + 1's first
 * chunk begins with its lower tile; with an odd number of row blocks the last
 * pair's second unit stores nothing).  Unit u is (row_block[u], col_start[u],
 * width[u]).  Writes min(count, capacity) entries and returns the total count
 * in *count.  Host only.                                                      */
int kfac_factor_tile_map(int64_t d, int64_t capacity, int32_t* row_block,
                         int64_t* col_start, int32_t* width, int64_t* count);

#ifdef __cplusplus
}
#endif

#endif /* KFAC_GB300_H */
