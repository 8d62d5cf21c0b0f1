/* oracle.c -- plain, slow, obviously correct CPU oracle of the shard step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no code, header or constant table with the CUDA
 * library: it is written from the pages' description of the method.
 *
 * Sources (web pages on fully sharded data parallel training):
 *   [FSDP]  "FSDP: Fully Sharded Data Parallel Training at Scale"
 *   [ZERO]  "AI Model Sharding: FSDP, DeepSpeed ZeRO, and Tensor Parallelism"
 *   [DDL]   "Distributed Deep Learning & Model Sharding"
 *
 * Precision: the pages fix that gradients are accumulated in fp32 and that
 * the master weights and both Adam moments are stored in fp32, so those steps
 * are done (reduce) or stored (state) in fp32 here. Everything the pages leave
 * open (the Adam update's intermediate arithmetic, the clip norm) is computed
 * in double, the exact result rounded once to fp32 for storage.
 *
 * Parity pins (tests/test_oracle_*.py): layout against brute force and the
 * pages' shard rule; byte accounting against the pages' worked numbers; the
 * reduce against exact sums and a rank-order probe; AdamW against closed forms
 * (first step, zero gradient, constant gradient, gradient scale invariance);
 * the 16-bit casts exhaustively against library conversions; clipping against
 * the library's clip_grad_norm_. No function here is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "oracle.h"

#ifdef _OPENMP
#include <omp.h>
#endif

/* Thread count used by the element loops (each element is independent, so
 * the results do not depend on it). */
void ora_set_threads(int32_t n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int32_t ora_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ layout */

/* [FSDP] "How FSDP shards a layer": the unit's tensors are flattened into one
 * vector of length P and GPU k holds elements floor(kP/N) .. floor((k+1)P/N)-1.
 * offsets[t] is where tensor t starts in the flat vector (prefix sum of the
 * element counts); bounds[k] = floor(k*P/N), k = 0..N. */
int ora_flatten_layout(const int64_t* numels, int32_t n_tensors, int32_t n_ranks,
                       int64_t* offsets, int64_t* bounds) {
  if (n_tensors < 0 || n_ranks < 1 || (!numels && n_tensors) || !offsets || !bounds) return ORA_EINVAL;
  offsets[0] = 0;
  for (int32_t t = 0; t < n_tensors; ++t) {
    if (numels[t] < 0) return ORA_EINVAL;
    if (offsets[t] > INT64_MAX - numels[t]) return ORA_EOVERFLOW;
    offsets[t + 1] = offsets[t] + numels[t];
  }
  int64_t P = offsets[n_tensors];
  for (int32_t k = 0; k <= n_ranks; ++k)
    bounds[k] = (int64_t)(((__int128)k * (__int128)P) / (__int128)n_ranks);
  return ORA_OK;
}

/* The shard that owns flat element i: the k with bounds[k] <= i < bounds[k+1]
 * (searched linearly over the rule's boundaries). Returns -1 if i is outside
 * [0, P). */
int32_t ora_shard_of(int64_t P, int32_t n_ranks, int64_t i) {
  if (i < 0 || i >= P || n_ranks < 1) return -1;
  for (int32_t k = 0; k < n_ranks; ++k) {
    int64_t lo = (int64_t)(((__int128)k * P) / n_ranks);
    int64_t hi = (int64_t)(((__int128)(k + 1) * P) / n_ranks);
    if (lo <= i && i < hi) return k;
  }
  return -1;
}

/* The pieces of shard `shard` that fall in each tensor: for every tensor t
 * whose range [offsets[t], offsets[t+1]) meets [bounds[k], bounds[k+1]),
 * one segment (t, offset inside tensor, offset inside shard, length).
 * With out == NULL only the count is returned. */
int ora_shard_segments(const int64_t* offsets, int32_t n_tensors, const int64_t* bounds, int32_t shard,
                       ora_segment* out, int32_t* count) {
  if (!offsets || !bounds || !count || shard < 0 || n_tensors < 0) return ORA_EINVAL;
  int64_t lo = bounds[shard], hi = bounds[shard + 1];
  int32_t c = 0;
  for (int32_t t = 0; t < n_tensors; ++t) {
    int64_t a = offsets[t] > lo ? offsets[t] : lo;
    int64_t b = offsets[t + 1] < hi ? offsets[t + 1] : hi;
    if (b > a) {
      if (out) {
        out[c].tensor = t;
        out[c].tensor_offset = a - offsets[t];
        out[c].shard_offset = a - lo;
        out[c].length = b - a;
      }
      ++c;
    }
  }
  *count = c;
  return ORA_OK;
}

/* -------------------------------------------------------------- accounting */

/* [FSDP] "Where memory goes": fp32 training keeps 4P (params) + 4P (grads)
 * + 8P (Adam m and v) = 16P bytes; the mixed-precision bill is 2P (16-bit
 * params) + 2P (16-bit grads) + 4P (fp32 master) + 8P (fp32 moments) = 16P.
 * [FSDP] "Per-GPU memory": FULL_SHARD keeps 16P/N per GPU, plus one unit's
 * gathered parameters (4P/M with M units) at the peak. SHARD_GRAD_OP shards
 * only grads and optimizer state; NO_SHARD shards nothing.
 * [DDL] "Data parallelism only works until the replica does not fit": the
 * optimizer bill of fp32 master + m + v is 12 bytes per parameter, which
 * ZeRO-1 divides by the number of ranks. */
int ora_state_bytes(int64_t P, int32_t n_ranks, int32_t n_units, ora_bytes* out) {
  if (P < 0 || n_ranks < 1 || n_units < 1 || !out) return ORA_EINVAL;
  double p = (double)P, N = (double)n_ranks, M = (double)n_units;
  memset(out, 0, sizeof *out);
  out->fp32_params = 4 * p;
  out->fp32_grads = 4 * p;
  out->fp32_adam = 8 * p;
  out->fp32_total = out->fp32_params + out->fp32_grads + out->fp32_adam;
  out->mp_params16 = 2 * p;
  out->mp_grads16 = 2 * p;
  out->mp_master32 = 4 * p;
  out->mp_adam32 = 8 * p;
  out->mp_total = out->mp_params16 + out->mp_grads16 + out->mp_master32 + out->mp_adam32;
  out->optimizer_state = out->mp_master32 + out->mp_adam32;
  out->zero1_optimizer_per_gpu = out->optimizer_state / N;
  out->full_shard_per_gpu = out->fp32_total / N;
  out->shard_grad_op_per_gpu = out->fp32_params + (out->fp32_grads + out->fp32_adam) / N;
  out->no_shard_per_gpu = out->fp32_total;
  out->unit_gather = out->fp32_params / M;
  out->full_shard_peak = out->full_shard_per_gpu + out->unit_gather;
  out->full_shard_saving = out->no_shard_per_gpu - out->full_shard_per_gpu;
  out->shard_grad_op_saving = out->no_shard_per_gpu - out->shard_grad_op_per_gpu;
  out->mp_full_shard_per_gpu = out->mp_total / N;
  out->mp_unit_gather16 = out->mp_params16 / M;
  return ORA_OK;
}

/* ------------------------------------------------------- 16-bit formats */

/* [FSDP] "Mixed precision": bf16 keeps fp32's 8 exponent bits and 7 mantissa
 * bits; fp16 has a 5-bit exponent (largest finite value 65504) and 10
 * mantissa bits. Widening either to fp32 is exact. */
float ora_widen16(uint16_t h, int32_t dtype) {
  if (dtype == ORA_BF16) {
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return f;
  }
  int sign = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double mag;
  if (e == 0) mag = ldexp((double)m, -24);             /* subnormal: m * 2^-24 */
  else if (e == 31) mag = m ? NAN : INFINITY;
  else mag = ldexp((double)(1024 + m), e - 25);        /* (1 + m/1024) * 2^(e-15) */
  return (float)(sign ? -mag : mag);
}

/* Round-to-nearest-even of an fp32 value to bf16, from the bit layout: the
 * 16 dropped bits decide; above half rounds up, exactly half rounds to the
 * even kept pattern. A carry out of the mantissa moves into the exponent
 * (overflowing to infinity at the top). NaN stays NaN (quiet bit set). */
uint16_t ora_round_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x0040u);
  uint32_t keep = b >> 16, drop = b & 0xFFFFu;
  if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

/* Round-to-nearest-even of an fp32 value to fp16, by the definition: find
 * the fp16 spacing q at |f| (2^-24 below the smallest normal 2^-14, else
 * 2^(floor(log2|f|) - 10)), take the nearest multiple of q, ties to the even
 * multiple, and encode it. A result of 2^16 or more is beyond the largest
 * finite value 65504 and becomes infinity. */
uint16_t ora_round_fp16(float f) {
  uint16_t sign = signbit(f) ? 0x8000u : 0u;
  if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
  double a = fabs((double)f);
  if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
  if (a == 0.0) return sign;
  double q;
  if (a < ldexp(1.0, -14)) q = ldexp(1.0, -24);
  else {
    int e;
    frexp(a, &e);                 /* a = fr * 2^e, fr in [0.5, 1): floor(log2 a) = e - 1 */
    q = ldexp(1.0, (e - 1) - 10);
  }
  double k = floor(a / q);        /* exact: a and q are powers-of-two scaled integers */
  double rem = a - k * q;         /* exact */
  if (rem > 0.5 * q || (rem == 0.5 * q && fmod(k, 2.0) == 1.0)) k += 1.0;
  double r = k * q;
  if (r >= 65536.0) return (uint16_t)(sign | 0x7C00u);
  if (r < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
  int e;
  frexp(r, &e);
  int ue = e - 1;                              /* r = 1.f * 2^ue */
  double frac = r / ldexp(1.0, ue) - 1.0;      /* in [0, 1) */
  uint16_t mant = (uint16_t)(frac * 1024.0);   /* exact */
  return (uint16_t)(sign | (uint16_t)((ue + 15) << 10) | mant);
}

uint16_t ora_round16(float f, int32_t dtype) {
  return dtype == ORA_BF16 ? ora_round_bf16(f) : ora_round_fp16(f);
}

int ora_round16_array(const float* x, int64_t n, int32_t dtype, uint16_t* out) {
  if (n < 0 || (n && (!x || !out)) || (dtype != ORA_BF16 && dtype != ORA_FP16)) return ORA_EINVAL;
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = ora_round16(x[i], dtype);
  return ORA_OK;
}

int ora_widen16_array(const uint16_t* h, int64_t n, int32_t dtype, float* out) {
  if (n < 0 || (n && (!h || !out)) || (dtype != ORA_BF16 && dtype != ORA_FP16)) return ORA_EINVAL;
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = ora_widen16(h[i], dtype);
  return ORA_OK;
}

/* ------------------------------------------------------------------ reduce */

/* [FSDP] "The FSDP unit communication cycle", backward step 3: the
 * reduce-scatter sums every rank's gradient and hands GPU k the part that
 * matches its shard. [FSDP] "Mixed precision": the sum is accumulated in
 * fp32 (reduce_dtype = float32). Here the N ranks' 16-bit gradients for one
 * shard are summed element by element in rank order 0, 1, ..., N-1 in fp32,
 * starting from rank 0's value; a post_scale other than 1 (e.g. 1/N for a
 * mean, or 1/S to undo a loss scale) multiplies the fp32 sum once.
 * With accumulate != 0 the result is added to out (gradient accumulation
 * over micro-batches: out = out + scaled sum). */
int ora_grad_reduce(const uint16_t* const* ranks, int32_t n_ranks, int32_t dtype, int64_t n,
                    float post_scale, int32_t accumulate, float* out) {
  if (n < 0 || n_ranks < 1 || !ranks || (n && !out) || (dtype != ORA_BF16 && dtype != ORA_FP16))
    return ORA_EINVAL;
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float acc = ora_widen16(ranks[0][i], dtype);
    for (int32_t r = 1; r < n_ranks; ++r) acc = acc + ora_widen16(ranks[r][i], dtype);
    if (post_scale != 1.0f) acc = acc * post_scale;
    out[i] = accumulate ? out[i] + acc : acc;
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------- AdamW */

/* [FSDP] "Where memory goes": Adam keeps, per parameter, a first moment (an
 * exponential moving average of the gradient) and a second moment (an
 * exponential moving average of the squared gradient), both in fp32, next to
 * an fp32 master copy of the parameter. [FSDP] "The FSDP unit communication
 * cycle": each GPU updates its own shard from its own gradient and state
 * shards, with no communication. The pages give no update equation; this is
 * the standard Adam step with bias correction and decoupled weight decay
 * (AdamW) with the decay applied as p * (1 - lr * wd) and eps added after the
 * square root of the bias-corrected second moment:
 *   m_t = b1 m + (1 - b1) g,  v_t = b2 v + (1 - b2) g^2,
 *   p_t = p (1 - lr wd) - lr (m_t / (1 - b1^t)) / (sqrt(v_t / (1 - b2^t)) + eps).
 * The step is evaluated in double from the fp32 inputs; m_t, v_t and p_t are
 * stored rounded to fp32; the 16-bit working parameter is the nearest-even
 * 16-bit value of the stored fp32 master ([FSDP] "Mixed precision").
 * g is multiplied by grad_scale (fp32, e.g. a clip coefficient) first when
 * grad_scale != 1. p16 may be NULL. */
int ora_adamw(const ora_adamw_hp* hp, int64_t n, const float* g, float grad_scale, float* master, float* m,
              float* v, uint16_t* p16, int32_t p16_dtype) {
  if (!hp || n < 0 || hp->step < 1 || (n && (!g || !master || !m || !v))) return ORA_EINVAL;
  if (p16 && p16_dtype != ORA_BF16 && p16_dtype != ORA_FP16) return ORA_EINVAL;
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
  const double bc1 = 1.0 - pow(b1, (double)hp->step);
  const double bc2 = 1.0 - pow(b2, (double)hp->step);
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float gf = g[i];
    if (grad_scale != 1.0f) gf = gf * grad_scale;
    double gi = gf;
    double mi = b1 * (double)m[i] + (1.0 - b1) * gi;
    double vi = b2 * (double)v[i] + (1.0 - b2) * gi * gi;
    double mhat = mi / bc1, vhat = vi / bc2;
    double p = (double)master[i] * (1.0 - lr * wd) - lr * mhat / (sqrt(vhat) + eps);
    m[i] = (float)mi;
    v[i] = (float)vi;
    master[i] = (float)p;
    if (p16) p16[i] = ora_round16(master[i], p16_dtype);
  }
  return ORA_OK;
}

/* ----------------------------------------------------------- unshard copy */

/* [FSDP] "The FSDP unit communication cycle", forward step 1: the all-gather
 * gives every GPU the complete parameter vector of the unit, i.e. the
 * concatenation of the N shards in rank order; shard k lands at
 * [bounds[k], bounds[k+1]). Reshard is the reverse copy (the flat vector cut
 * back into its shards). elem_size is 2 (16-bit) or 4 (fp32) bytes. */
int ora_unshard(const void* const* shards, const int64_t* bounds, int32_t n_ranks, int32_t elem_size,
                void* flat) {
  if (!shards || !bounds || !flat || n_ranks < 1 || (elem_size != 2 && elem_size != 4)) return ORA_EINVAL;
  for (int32_t k = 0; k < n_ranks; ++k) {
    int64_t len = bounds[k + 1] - bounds[k];
    if (len < 0) return ORA_EINVAL;
    if (len) memcpy((char*)flat + bounds[k] * elem_size, shards[k], (size_t)(len * elem_size));
  }
  return ORA_OK;
}

int ora_reshard(const void* flat, const int64_t* bounds, int32_t n_ranks, int32_t elem_size,
                void* const* shards) {
  if (!shards || !bounds || !flat || n_ranks < 1 || (elem_size != 2 && elem_size != 4)) return ORA_EINVAL;
  for (int32_t k = 0; k < n_ranks; ++k) {
    int64_t len = bounds[k + 1] - bounds[k];
    if (len < 0) return ORA_EINVAL;
    if (len) memcpy(shards[k], (const char*)flat + bounds[k] * elem_size, (size_t)(len * elem_size));
  }
  return ORA_OK;
}

/* --------------------------------------------------- clipping / overflow */

/* [FSDP] "Gradient clipping": the norm that clipping uses is the norm of the
 * whole gradient, so each shard contributes its sum of squares and the
 * contributions are added across shards before the square root; a local
 * norm per shard would underestimate it. Sum of squares of an fp32 shard, in
 * double. */
double ora_sumsq(const float* g, int64_t n) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s += (double)g[i] * (double)g[i];
  return s;
}

/* The pages do not print the clip rule; this is the convention of the
 * clip_grad_norm_ call they name: coefficient = max_norm / (norm + 1e-6),
 * capped at 1, applied to every gradient element. Returned as fp32, the
 * precision in which gradients drive the update. */
float ora_clip_coef(double total_sumsq, float max_norm) {
  double norm = sqrt(total_sumsq);
  double c = (double)max_norm / (norm + 1e-6);
  return (float)(c < 1.0 ? c : 1.0);
}

/* [FSDP] "Mixed precision" and [DDL] "Memory levers that are not
 * parallelism": fp16 training scales the loss up and divides the gradients
 * back before the optimizer step. A scaled gradient that overflowed is
 * infinite or NaN; the step must then be skipped. Returns 1 when every value
 * is finite. */
int32_t ora_all_finite(const float* g, int64_t n) {
  for (int64_t i = 0; i < n; ++i)
    if (!isfinite(g[i])) return 0;
  return 1;
}
