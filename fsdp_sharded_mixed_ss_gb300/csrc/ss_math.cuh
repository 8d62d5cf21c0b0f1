// ss_math.cuh -- per-element arithmetic of the shard step (device code).
//
// The AdamW update is evaluated in "double-float" arithmetic: every value that
// feeds the final roundings is carried as an unevaluated sum hi + lo of two
// fp32 numbers, built from error-free transformations (Knuth's TwoSum, Dekker's
// Fast2Sum and the FMA-based exact product; see Muller et al., "Handbook of
// Floating-Point Arithmetic", ch. 4 and 14). The update is therefore known to
// about 2^-44 relative before it is rounded once to fp32, so the stored m, v
// and master are the correctly rounded values of the exact step except when
// the exact value lies within ~2^-44 of a rounding boundary. The kernel is
// bound by HBM bandwidth with spare issue slots; this spends them so that
// repeated steps do not accumulate fp32 rounding drift.
//
// Compile without FMA contraction (-fmad=false): every fused multiply-add here
// is written explicitly.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define SS_HD __host__ __device__ __forceinline__
#else
#define SS_HD inline
#include <cmath>
#endif

namespace ss {

struct dd {
  float hi, lo;
};

// s + e == a + b exactly (any magnitudes).
SS_HD dd two_sum(float a, float b) {
  float s = a + b;
  float bb = s - a;
  float e = (a - (s - bb)) + (b - bb);
  return {s, e};
}

// s + e == a + b exactly when |a| >= |b| (or a == 0).
SS_HD dd fast_two_sum(float a, float b) {
  float s = a + b;
  float e = b - (s - a);
  return {s, e};
}

// p + e == a * b exactly (barring underflow).
SS_HD dd two_prod(float a, float b) {
  float p = a * b;
  float e = fmaf(a, b, -p);
  return {p, e};
}

SS_HD float approx_rsqrt(float x) {
#if defined(__CUDA_ARCH__)
  return rsqrtf(x);
#else
  return 1.0f / std::sqrt(x);
#endif
}

SS_HD float approx_rcp(float x) {
#if defined(__CUDA_ARCH__)
  return __fdividef(1.0f, x);
#else
  return 1.0f / x;
#endif
}

// Step constants, prepared on the host in double and split into fp32 pairs.
// With bc1 = 1 - beta1^t and bc2 = 1 - beta2^t the AdamW step
//   p' = p (1 - lr wd) - (lr / bc1) m' / (sqrt(v' / bc2) + eps)
// is evaluated as p' = p D - A m' / (sqrt(v') + E), multiplying numerator and
// denominator by sqrt(bc2):  D = 1 - lr wd,  A = lr sqrt(bc2) / bc1,
// E = eps sqrt(bc2).
struct AdamConst {
  float b1, c1, c1_lo;  // beta1 ; 1 - beta1 as an fp32 pair (lo = 0 when beta1 >= 0.5)
  float b2, c2, c2_lo;  // beta2 ; 1 - beta2 as an fp32 pair
  float A_hi, A_lo;
  float E_hi, E_lo;
  float D_hi, D_lo;
};

// One AdamW step of one element, in place:
//   m' = b1 m + (1-b1) g ;  v' = b2 v + (1-b2) g^2 ;  p' = p D - A m' / (sqrt(v') + E)
SS_HD void adamw_elem(const AdamConst& k, float g, float& p, float& m, float& v) {
  // first moment
  dd a = two_prod(k.b1, m);
  dd b = two_prod(k.c1, g);
  b.lo = fmaf(k.c1_lo, g, b.lo);
  dd s = two_sum(a.hi, b.hi);
  dd mm = fast_two_sum(s.hi, s.lo + (a.lo + b.lo));
  // second moment
  dd g2 = two_prod(g, g);
  dd q = two_prod(k.c2, g2.hi);
  q.lo = fmaf(k.c2, g2.lo, fmaf(k.c2_lo, g2.hi, q.lo));
  dd pv = two_prod(k.b2, v);
  dd t = two_sum(pv.hi, q.hi);
  dd vv = fast_two_sum(t.hi, t.lo + (pv.lo + q.lo));
  // r = sqrt(v'): one Newton correction of an approximate root
  dd r = {0.0f, 0.0f};
  if (vv.hi > 0.0f) {
    float rs = approx_rsqrt(vv.hi);
    float r0 = vv.hi * rs;
    float res = fmaf(-r0, r0, vv.hi) + vv.lo;
    r = fast_two_sum(r0, res * (0.5f * rs));
  }
  // d = r + E
  dd de = two_sum(r.hi, k.E_hi);
  dd d = fast_two_sum(de.hi, de.lo + (r.lo + k.E_lo));
  // u1 = m' / d: approximate quotient plus one remainder correction
  float rc = approx_rcp(d.hi);
  float q0 = mm.hi * rc;
  dd qd = two_prod(q0, d.hi);
  float rem = fmaf(-q0, d.lo, ((mm.hi - qd.hi) - qd.lo) + mm.lo);
  dd qq = fast_two_sum(q0, rem * rc);
  // u = A * u1
  dd u = two_prod(k.A_hi, qq.hi);
  u.lo = fmaf(k.A_hi, qq.lo, fmaf(k.A_lo, qq.hi, u.lo));
  // p' = p D - u, rounded once
  dd pd = two_prod(p, k.D_hi);
  pd.lo = fmaf(p, k.D_lo, pd.lo);
  dd z = two_sum(pd.hi, -u.hi);
  p = z.hi + (z.lo + (pd.lo - u.lo));
  m = mm.hi;
  v = vv.hi;
}

}  // namespace ss
