// CUDA-core 128 x 128 tile product used where the arithmetic must stay in
// fp32 or fp64 (fp32-input factors, the blocked Cholesky inverse and the
// preconditioning GEMMs of this version).
//
//   acc(m, n) += sum_{k < K} A(m, k) * B(n, k)
//
// A(m, k) lives at A.p[m * A.sm + k * A.sk] for m < A.mv, k < K; outside it
// reads as 0 (same for B).  256 threads; thread (ty, tx) = (tid / 16, tid % 16)
// owns rows ty*8 .. ty*8+7 and columns tx*8 .. tx*8+7 of the tile.  Operand
// slabs of KC values of k are staged in shared memory as S[k][m]; the next
// slab is fetched into registers while the current one is multiplied.
#pragma once
#include <stdint.h>

#include "common.cuh"

namespace kfac {

template <typename Tin>
struct Opnd {
  const Tin* p;
  int64_t sm, sk;  // strides of m and k (elements)
  int mv;          // valid rows (m)
};

template <typename T>
struct SimtCfg;
template <>
struct SimtCfg<float> {
  static constexpr int KC = 16;
  static constexpr int PITCH = 128 + 4;
};
template <>
struct SimtCfg<double> {
  static constexpr int KC = 8;
  static constexpr int PITCH = 128 + 2;
};

template <typename T>
constexpr int simt_smem_bytes() {
  return 2 * SimtCfg<T>::KC * SimtCfg<T>::PITCH * (int)sizeof(T);
}

template <typename T, typename Tin>
__device__ __forceinline__ T load_as(const Tin* p);
template <>
__device__ __forceinline__ float load_as<float, float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_as<float, uint16_t>(const uint16_t* p) { return bf16_to_f32(__ldg(p)); }
template <>
__device__ __forceinline__ double load_as<double, double>(const double* p) { return *p; }
template <>
__device__ __forceinline__ double load_as<double, float>(const float* p) { return (double)*p; }

// Eight consecutive shared-memory values as two or four 16-byte loads.
template <typename T>
__device__ __forceinline__ void lds8(const T* p, T (&v)[8]);
template <>
__device__ __forceinline__ void lds8<float>(const float* p, float (&v)[8]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  const float4 y = *reinterpret_cast<const float4*>(p + 4);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}
template <>
__device__ __forceinline__ void lds8<double>(const double* p, double (&v)[8]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const double2 x = *reinterpret_cast<const double2*>(p + 2 * q);
    v[2 * q] = x.x;
    v[2 * q + 1] = x.y;
  }
}

template <typename T, typename Tin>
__device__ __forceinline__ void fetch_slab(T (&reg)[(SimtCfg<T>::KC * 128) / 256], const Opnd<Tin>& o,
                                           int k0, int K) {
  constexpr int KC = SimtCfg<T>::KC;
  constexpr int EPT = (KC * 128) / 256;
  const int tid = threadIdx.x;
  if (o.sk == 1) {
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = tid + 256 * j;
      const int k = e % KC, m = e / KC;
      const int kk = k0 + k;
      reg[j] = (m < o.mv && kk < K) ? load_as<T, Tin>(o.p + (int64_t)m * o.sm + kk) : T(0);
    }
  } else {
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = tid + 256 * j;
      const int m = e % 128, k = e / 128;
      const int kk = k0 + k;
      reg[j] = (m < o.mv && kk < K) ? load_as<T, Tin>(o.p + (int64_t)m * o.sm + (int64_t)kk * o.sk) : T(0);
    }
  }
}

template <typename T, typename Tin>
__device__ __forceinline__ void store_slab(T* S, const T (&reg)[(SimtCfg<T>::KC * 128) / 256],
                                           const Opnd<Tin>& o) {
  constexpr int KC = SimtCfg<T>::KC;
  constexpr int PITCH = SimtCfg<T>::PITCH;
  constexpr int EPT = (KC * 128) / 256;
  const int tid = threadIdx.x;
  if (o.sk == 1) {
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = tid + 256 * j;
      S[(e % KC) * PITCH + e / KC] = reg[j];
    }
  } else {
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = tid + 256 * j;
      S[(e / 128) * PITCH + e % 128] = reg[j];
    }
  }
}

template <typename T>
__device__ __forceinline__ void zero_acc(T (&acc)[8][8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = T(0);
}

// smem: simt_smem_bytes<T>() bytes.  All 256 threads must call.
template <typename T, typename TinA, typename TinB>
__device__ void simt_tile(T (&acc)[8][8], const Opnd<TinA>& A, const Opnd<TinB>& B, int K, T* smem) {
  constexpr int KC = SimtCfg<T>::KC;
  constexpr int PITCH = SimtCfg<T>::PITCH;
  constexpr int EPT = (KC * 128) / 256;
  T* SA = smem;
  T* SB = smem + KC * PITCH;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  T ra[EPT], rb[EPT];
  if (K <= 0) return;
  fetch_slab<T, TinA>(ra, A, 0, K);
  fetch_slab<T, TinB>(rb, B, 0, K);
  for (int k0 = 0; k0 < K; k0 += KC) {
    __syncthreads();
    store_slab<T, TinA>(SA, ra, A);
    store_slab<T, TinB>(SB, rb, B);
    __syncthreads();
    if (k0 + KC < K) {
      fetch_slab<T, TinA>(ra, A, k0 + KC, K);
      fetch_slab<T, TinB>(rb, B, k0 + KC, K);
    }
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      T a[8], b[8];
      lds8<T>(SA + k * PITCH + ty * 8, a);
      lds8<T>(SB + k * PITCH + tx * 8, b);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
    }
  }
  __syncthreads();
}

// out = A Bᵀ for fp64 operands, in double-float arithmetic on the fp32 pipes
// (the part's fp64 rate is a small fraction of its fp32 rate).  Operands are
// staged as (hi, lo) float pairs, hi = fl32(x), lo = fl32(x - hi) (about 48
// significant bits); each multiply-add keeps the exact error of the product
// hi_a hi_b (an FMA, after Dekker's two-product) and of its addition to the
// running sum (Knuth's two-sum), and adds the cross terms hi_a lo_b + lo_a hi_b
// to the low word.  The error grows like K 2^-48 relative to the largest
// term, against K 2^-53 in fp64: ample for the inverse's fp64 pass, whose
// target is a residual of 1e-3 at condition numbers near 1e6.
// kDfThreads threads; thread (ty, tx) = (tid / 16, tid % 16) owns rows
// ty*4 .. ty*4+3 and columns tx*8 .. tx*8+7 of the tile (two words per value
// double the accumulator registers, so each thread holds half the values of
// simt_tile's and twice as many warps share an SM).
// smem: simt_smem_bytes<double>() bytes.  All kDfThreads threads must call.
constexpr int kDfThreads = 512;
constexpr int kDfEpt = (SimtCfg<double>::KC * 128) / kDfThreads;  // staged values per thread and operand

__device__ __forceinline__ float2 df_split(double x) {
  const float hi = (float)x;
  return make_float2(hi, (float)(x - (double)hi));
}

__device__ __forceinline__ void df_fetch(float2 (&reg)[kDfEpt], const Opnd<double>& o, int k0, int K) {
  constexpr int KC = SimtCfg<double>::KC;
  const int tid = threadIdx.x;
#pragma unroll
  for (int j = 0; j < kDfEpt; ++j) {
    const int e = tid + kDfThreads * j;
    const int k = o.sk == 1 ? e % KC : e / 128, m = o.sk == 1 ? e / KC : e % 128;
    const int kk = k0 + k;
    reg[j] = df_split((m < o.mv && kk < K) ? o.p[(int64_t)m * o.sm + (int64_t)kk * o.sk] : 0.0);
  }
}

__device__ __forceinline__ void df_store(float2* S, const float2 (&reg)[kDfEpt], const Opnd<double>& o) {
  constexpr int KC = SimtCfg<double>::KC;
  constexpr int PITCH = SimtCfg<double>::PITCH;
  const int tid = threadIdx.x;
#pragma unroll
  for (int j = 0; j < kDfEpt; ++j) {
    const int e = tid + kDfThreads * j;
    if (o.sk == 1)
      S[(e % KC) * PITCH + e / KC] = reg[j];
    else
      S[(e / 128) * PITCH + e % 128] = reg[j];
  }
}

template <int N>
__device__ __forceinline__ void lds_df(const float2* p, float2 (&v)[N]) {
#pragma unroll
  for (int q = 0; q < N / 2; ++q) {
    const float4 x = *reinterpret_cast<const float4*>(p + 2 * q);
    v[2 * q] = make_float2(x.x, x.y);
    v[2 * q + 1] = make_float2(x.z, x.w);
  }
}

__device__ inline void simt_tile_df(double (&out)[4][8], const Opnd<double>& A, const Opnd<double>& B, int K,
                                    double* smem) {
  constexpr int KC = SimtCfg<double>::KC;
  constexpr int PITCH = SimtCfg<double>::PITCH;
  float2* SA = reinterpret_cast<float2*>(smem);
  float2* SB = SA + KC * PITCH;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  float hi[4][8], lo[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) hi[i][j] = lo[i][j] = 0.f;
  float2 ra[kDfEpt], rb[kDfEpt];
  if (K > 0) {
    df_fetch(ra, A, 0, K);
    df_fetch(rb, B, 0, K);
  }
  for (int k0 = 0; k0 < K; k0 += KC) {
    __syncthreads();
    df_store(SA, ra, A);
    df_store(SB, rb, B);
    __syncthreads();
    if (k0 + KC < K) {
      df_fetch(ra, A, k0 + KC, K);
      df_fetch(rb, B, k0 + KC, K);
    }
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      float2 a[4], b[8];
      lds_df<4>(SA + k * PITCH + ty * 4, a);
      lds_df<8>(SB + k * PITCH + tx * 8, b);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float p = a[i].x * b[j].x;
          const float pe = fmaf(a[i].x, b[j].x, -p);  // hi_a hi_b - p, exactly
          const float s = hi[i][j] + p;
          const float bb = s - hi[i][j];
          const float e = (hi[i][j] - (s - bb)) + (p - bb);  // hi + p - s, exactly
          hi[i][j] = s;
          lo[i][j] += e + fmaf(a[i].x, b[j].y, fmaf(a[i].y, b[j].x, pe));
        }
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) out[i][j] = (double)hi[i][j] + (double)lo[i][j];
}

}  // namespace kfac
