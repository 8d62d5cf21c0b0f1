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
struct AdamConst {
  float b1, c1, c1_lo;  // beta1 ; 1 - beta1 as an fp32 pair (lo = 0 when beta1 >= 0.5)
  float b2, c2, c2_lo;  // beta2 ; 1 - beta2 as an fp32 pair
  float eps;
  float S_hi, S_lo;  // lr / (1 - beta1^t)
  float R_hi, R_lo;  // 1 / sqrt(1 - beta2^t)
  float L_hi, L_lo;  // lr * weight_decay
};

// One AdamW step of one element, in place:
//   m' = b1 m + (1-b1) g ;  v' = b2 v + (1-b2) g^2
//   p' = p - ( lr*wd * p + S * m' / (sqrt(v') * R + eps) )
// which is p (1 - lr wd) - lr * mhat / (sqrt(vhat) + eps) with the bias
// corrections folded into S and R.
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
  // d = r * R + eps
  dd rr = two_prod(r.hi, k.R_hi);
  rr.lo = fmaf(r.hi, k.R_lo, fmaf(r.lo, k.R_hi, rr.lo));
  rr = fast_two_sum(rr.hi, rr.lo);
  dd de = two_sum(rr.hi, k.eps);
  dd d = fast_two_sum(de.hi, de.lo + rr.lo);
  // u1 = m' / d: approximate quotient plus one remainder correction
  float rc = approx_rcp(d.hi);
  float q0 = mm.hi * rc;
  dd qd = two_prod(q0, d.hi);
  float rem = fmaf(-q0, d.lo, ((mm.hi - qd.hi) - qd.lo) + mm.lo);
  dd qq = fast_two_sum(q0, rem * rc);
  // u = S * u1 + L * p
  dd aa = two_prod(k.S_hi, qq.hi);
  aa.lo = fmaf(k.S_hi, qq.lo, fmaf(k.S_lo, qq.hi, aa.lo));
  dd w = two_prod(p, k.L_hi);
  w.lo = fmaf(p, k.L_lo, w.lo);
  dd u = two_sum(aa.hi, w.hi);
  u.lo = u.lo + (aa.lo + w.lo);
  // p' = p - u, rounded once
  dd z = two_sum(p, -u.hi);
  p = z.hi + (z.lo - u.lo);
  m = mm.hi;
  v = vv.hi;
}

}  // namespace ss
