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

}  // namespace kfac
