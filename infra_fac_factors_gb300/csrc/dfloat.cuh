// Double-float numbers: hi + lo in two fp32 words (about 48 significant
// bits), for the inverse's fp64 pass, whose fp64 rate on this part is a small
// fraction of its fp32 rate.  Built from error-free transformations: Knuth's
// two-sum for additions, Dekker's two-product through an FMA for products,
// and the fast two-sum (|s| >= |e|) to renormalise; the square root and the
// reciprocal of a pivot take one Newton step from their fp32 values.
#pragma once

namespace kfac {

struct DF {
  float hi, lo;
  DF() = default;
  __device__ DF(float h, float l) : hi(h), lo(l) {}
  __device__ DF(double x) : hi((float)x), lo((float)(x - (double)(float)x)) {}
  __device__ explicit operator double() const { return (double)hi + (double)lo; }
};

// s + e with |s| >= |e| (or s == 0), renormalised so that |lo| <= ulp(hi) / 2
__device__ __forceinline__ DF df_fast_sum(float s, float e) {
  const float h = s + e;
  return DF(h, e - (h - s));
}
__device__ __forceinline__ DF operator+(DF a, DF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb);  // a.hi + b.hi - s, exactly
  return df_fast_sum(s, e + (a.lo + b.lo));
}
__device__ __forceinline__ DF operator-(DF a) { return DF(-a.hi, -a.lo); }
__device__ __forceinline__ DF operator-(DF a, DF b) { return a + (-b); }
__device__ __forceinline__ DF operator*(DF a, DF b) {
  const float p = a.hi * b.hi;
  const float e = fmaf(a.hi, b.hi, -p);  // a.hi b.hi - p, exactly
  return df_fast_sum(p, fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e)));
}
__device__ __forceinline__ DF& operator+=(DF& a, DF b) { return a = a + b; }
__device__ __forceinline__ DF& operator-=(DF& a, DF b) { return a = a - b; }
__device__ __forceinline__ DF& operator*=(DF& a, DF b) { return a = a * b; }
__device__ __forceinline__ bool operator<(DF a, DF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ bool operator>(DF a, DF b) { return b < a; }

// ljj = sqrt(piv) and inv = 1 / ljj of a positive Cholesky pivot
__device__ __forceinline__ void pivot_scale(DF piv, DF& ljj, DF& inv) {
  const float s = sqrtf(piv.hi);
  const DF r = piv - DF(s, 0.f) * DF(s, 0.f);  // piv - s^2
  ljj = df_fast_sum(s, (r.hi + r.lo) / (2.f * s));
  const float q = 1.f / ljj.hi;
  const DF t = DF(1.f, 0.f) - ljj * DF(q, 0.f);  // 1 - ljj q
  inv = df_fast_sum(q, q * (t.hi + t.lo));
}

}  // namespace kfac
