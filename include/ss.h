/* ss.h -- C ABI of the GB300 shard-step library (libss.so).
 *
 * The library implements, on one GPU, the per-shard training-state update of
 * fully sharded data-parallel training as described on the page "FSDP: Fully
 * Sharded Data Parallel Training at Scale" (and its companions "AI Model
 * Sharding: FSDP, DeepSpeed ZeRO, and Tensor Parallelism" and "Distributed
 * Deep Learning & Model Sharding"):
 *
 *   flatten -> cut at floor(kP/N) -> sum the N ranks' 16-bit gradients in fp32
 *   -> AdamW on fp32 master/m/v -> cast to 16-bit params -> unshard copy.
 *
 * The N ranks are virtual: all their gradient buffers live in this GPU's
 * memory and nothing moves between GPUs.
 *
 * Conventions for every call:
 *   - Plain C types only. Device pointers are raw addresses of device memory
 *     (e.g. a tensor's data pointer); host pointers are marked "host".
 *   - Ownership: the caller allocates and frees every buffer. The library never
 *     allocates, frees or synchronises; GPU calls only enqueue kernels on
 *     `stream` (a cudaStream_t; NULL is the legacy default stream) and return.
 *   - Errors: every call returns an ss_status. Argument errors are detected on
 *     the host before anything is launched and leave all buffers untouched.
 *     SS_ERR_CUDA reports a failed launch; ss_last_cuda_error() names it.
 *     Errors raised later by the kernels themselves surface at the caller's
 *     next synchronisation, as for any CUDA work.
 *   - Element counts are int64; n == 0 is valid and launches nothing.
 *   - Layout: every array is dense (stride 1) in the order of the flat
 *     parameter vector. fp32 arrays must be 4-byte aligned, 16-bit arrays
 *     2-byte aligned (SS_ERR_ALIGN otherwise). The kernels use 16-byte vector
 *     accesses when all arrays of a call share one 16-byte phase; when the fp32
 *     arrays share one but 16-bit arrays do not (views at offsets that are not
 *     multiples of 8 elements), the 16-bit arrays are read as aligned 16-byte
 *     chunks and realigned in registers; with no common fp32 phase the kernels
 *     fall back to element accesses. The results are the same in every case;
 *     only the bandwidth differs.
 */
#ifndef SS_H
#define SS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SS_ABI_VERSION 2
#define SS_MAX_RANKS 1024

typedef enum ss_status {
  SS_OK = 0,
  SS_ERR_INVALID_ARG = 1, /* NULL where a buffer is required, negative size, bad hyperparameter, rank count out of range */
  SS_ERR_ALIGN = 2,       /* a pointer is not aligned to its element size */
  SS_ERR_OVERLAP = 3,     /* an output buffer overlaps another output or an input */
  SS_ERR_DTYPE = 4,       /* dtype not allowed for this argument */
  SS_ERR_OVERFLOW = 5,    /* a size or offset does not fit in int64 */
  SS_ERR_CUDA = 6         /* a CUDA runtime call or kernel launch failed */
} ss_status;

typedef enum ss_dtype { SS_BF16 = 0, SS_FP16 = 1, SS_FP32 = 2 } ss_dtype;

/* A piece of one shard that lies inside one tensor of the unit. */
typedef struct ss_segment {
  int32_t tensor;        /* index of the tensor in the unit */
  int32_t pad_;
  int64_t tensor_offset; /* first element of the piece inside that tensor */
  int64_t shard_offset;  /* first element of the piece inside the shard */
  int64_t length;        /* elements in the piece (> 0) */
} ss_segment;

/* Training-state bytes of a unit of P parameters over N ranks and M units. */
typedef struct ss_bytes {
  double fp32_params, fp32_grads, fp32_adam, fp32_total;               /* 4P, 4P, 8P, 16P */
  double mp_params16, mp_grads16, mp_master32, mp_adam32, mp_total;    /* 2P, 2P, 4P, 8P, 16P */
  double optimizer_state, zero1_optimizer_per_gpu;                     /* 12P (master+m+v), 12P/N */
  double full_shard_per_gpu, shard_grad_op_per_gpu, no_shard_per_gpu;  /* 16P/N, 4P+12P/N, 16P */
  double unit_gather, full_shard_peak;                                 /* 4P/M, 16P/N + 4P/M */
  double full_shard_saving, shard_grad_op_saving;                      /* vs NO_SHARD */
  double mp_full_shard_per_gpu, mp_unit_gather16;                      /* 16P/N, 2P/M */
} ss_bytes;

/* AdamW hyperparameters. 0 <= beta1, beta2 < 1; lr, eps, weight_decay finite
 * and >= 0; step >= 1 is the 1-based index of this update (bias correction). */
typedef struct ss_adamw_hparams {
  float lr, beta1, beta2, eps, weight_decay;
  int32_t pad_;
  int64_t step;
} ss_adamw_hparams;

/* Optional extras of ss_adam_step; pass NULL for none. All pointers device. */
typedef struct ss_step_options {
  float* g_out;                 /* [n] fp32: receives the reduced gradient (after post_scale, before dev_grad_scale) */
  int32_t* nonfinite_flag;      /* int32: set to 1 when any reduced gradient is inf or NaN; never cleared */
  const float* dev_grad_scale;  /* fp32 scalar multiplying the reduced gradient before the update (e.g. a clip coefficient) */
  const int32_t* dev_skip_flag; /* int32: when nonzero at kernel start, the call writes nothing (overflow skip) */
} ss_step_options;

/* ------------------------------------------------------------------ layout
 * "FSDP: Fully Sharded Data Parallel Training at Scale", how a layer is
 * sharded: the unit's tensors are flattened into one vector of P elements and
 * rank k owns elements [floor(kP/N), floor((k+1)P/N)).
 *
 * ss_flatten_layout: numels [n_tensors] (host, each >= 0) ->
 *   tensor_offsets [n_tensors+1] (host): exclusive prefix sum, last = P;
 *   shard_bounds   [n_ranks+1]  (host): floor(k*P/n_ranks), k = 0..n_ranks.
 * 1 <= n_ranks <= 2^30. k*P is formed in 128-bit arithmetic.
 * SS_ERR_OVERFLOW if P exceeds int64. Host only; no GPU is touched. */
ss_status ss_flatten_layout(const int64_t* numels, int32_t n_tensors, int32_t n_ranks,
                            int64_t* tensor_offsets, int64_t* shard_bounds);

/* The pieces of shard `shard` in tensor order (host only). With out == NULL,
 * only *count is written; otherwise up to `capacity` pieces are written and
 * SS_ERR_INVALID_ARG is returned if capacity is too small (*count still set). */
ss_status ss_shard_segments(const int64_t* tensor_offsets, int32_t n_tensors, const int64_t* shard_bounds,
                            int32_t n_ranks, int32_t shard, ss_segment* out, int32_t capacity, int32_t* count);

/* The shard owning flat element i, or -1 when i is outside [0, P) (host only). */
int32_t ss_shard_of(int64_t P, int32_t n_ranks, int64_t i);

/* "FSDP: Fully Sharded Data Parallel Training at Scale", where memory goes and
 * per-GPU memory: 4P/4P/8P fp32 and 2P/2P/4P/8P mixed-precision accounting,
 * divided by N under FULL_SHARD, plus one unit's gathered parameters at the
 * peak. Host only. P >= 0, n_ranks >= 1, n_units >= 1. */
ss_status ss_state_bytes(int64_t P, int32_t n_ranks, int32_t n_units, ss_bytes* out);

/* ------------------------------------------------------------------ reduce
 * "FSDP: Fully Sharded Data Parallel Training at Scale", the unit's
 * communication cycle (backward, reduce-scatter) and the mixed-precision
 * section (reduce_dtype fp32): rank k receives the sum over ranks of the
 * gradient elements of its shard, accumulated in fp32.
 *
 * rank_grads [n_ranks] (host array of device pointers, each to n elements of
 *   gdtype = SS_BF16 or SS_FP16, already offset to the shard's first element;
 *   the same pointer may appear more than once).
 * g_out [n] fp32 (device):
 *   g = ((float)G_0 + (float)G_1) + ... + (float)G_{N-1}, in rank order, then
 *   g *= post_scale when post_scale != 1 (one fp32 multiply), then
 *   g_out = accumulate ? g_out + g : g.
 * nonfinite_flag (device int32, optional): set to 1 when a written value is
 *   inf or NaN (never cleared by the library).
 * The sum is bit-exact and independent of the launch configuration.
 * g_out must not overlap any rank buffer (SS_ERR_OVERLAP). */
ss_status ss_grad_reduce(const void* const* rank_grads, int32_t n_ranks, ss_dtype gdtype, int64_t n,
                         float post_scale, int32_t accumulate, float* g_out, int32_t* nonfinite_flag,
                         void* stream);

/* ------------------------------------------------------------------- AdamW
 * "FSDP: Fully Sharded Data Parallel Training at Scale", where memory goes
 * (Adam's two fp32 moving averages and the fp32 master copy) and the local
 * optimizer step on each shard, fused with the reduce above and the 16-bit
 * cast of the mixed-precision section. One pass over the shard:
 *
 *   g  = reduce(rank_grads) (as ss_grad_reduce, post_scale applied) or g32[i]
 *   g *= *dev_grad_scale                       (when given)
 *   m  = b1 m + (1-b1) g ;  v = b2 v + (1-b2) g^2
 *   p  = p (1 - lr wd) - lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)
 *   param16 = round-to-nearest-even(p)         (when param16 != NULL)
 *
 * The update is evaluated in double-float (pairs of fp32) so the stored
 * master, m and v are the correctly rounded values of the exact step except
 * when the exact value lies within ~2^-44 relative of a rounding boundary.
 *
 * hp (host): hyperparameters; see ss_adamw_hparams.
 * n: shard length. g32 (device [n] fp32) or, when g32 == NULL, rank_grads /
 *   n_ranks / gdtype / post_scale exactly as in ss_grad_reduce.
 * master, m, v (device [n] fp32): read and updated in place.
 * param16 (device [n] of pdtype = SS_BF16/SS_FP16) or NULL. It may point into
 *   a flat full-unit buffer at the shard's offset (unshard fused into the step).
 * opts (host, optional): see ss_step_options.
 * Outputs (master, m, v, param16, g_out) must not overlap each other or the
 * inputs (SS_ERR_OVERLAP). With non-finite gradients the state becomes
 * non-finite; use nonfinite_flag in a prior ss_grad_reduce or ss_grad_sumsq pass
 * with dev_skip_flag to skip such a step. */
ss_status ss_adam_step(const ss_adamw_hparams* hp, int64_t n, const float* g32, const void* const* rank_grads,
                       int32_t n_ranks, ss_dtype gdtype, float post_scale, float* master, float* m, float* v,
                       void* param16, ss_dtype pdtype, const ss_step_options* opts, void* stream);

/* ------------------------------------------------------- global clip norm
 * "FSDP: Fully Sharded Data Parallel Training at Scale", gradient clipping:
 * the clip norm is the norm of the whole gradient, so every shard contributes
 * its sum of squares and the contributions are added across shards before the
 * square root (a per-shard norm would underestimate it).
 *
 * ss_grad_sumsq: *sumsq_out (device double) = sum of g[i]^2 over the shard,
 *   where g is the reduced gradient exactly as in ss_adam_step (rank-ordered
 *   fp32 sum of rank_grads times post_scale, or g32). Optionally writes g to
 *   g_out [n] fp32 and sets *nonfinite_flag to 1 when any g is inf/NaN.
 *   workspace: device scratch of at least ss_grad_sumsq_workspace(n) bytes,
 *   8-byte aligned, owned by the caller, overwritten (no initial contents
 *   needed). Each group of 8 squares is added in fp32, the rest in double, in
 *   an order fixed by n and the arrays' alignment (not by the launch), so the
 *   result is reproducible and within 5e-7 relative of the exact sum.
 *   Two kernel launches on `stream`; the second (the final sum over the
 *   tiles) is a programmatic dependent of the first, so its launch overlaps
 *   the first's end (it still reads nothing before the first has finished).
 * ss_grad_sumsq_workspace: the workspace size in bytes for a shard of n
 *   elements (-1 if n < 0).
 * ss_clip_coef: shard_sumsq [n_shards] (device doubles, one per shard) ->
 *   norm = sqrt(sum in shard order), *coef_out (device float) =
 *   min(1, max_norm / (norm + 1e-6)), the coefficient of the clip_grad_norm_
 *   convention; *norm_out (device double, optional) = norm. Feed coef_out to
 *   ss_adam_step as opts->dev_grad_scale. max_norm > 0 and finite. */
int64_t ss_grad_sumsq_workspace(int64_t n);
ss_status ss_grad_sumsq(int64_t n, const float* g32, const void* const* rank_grads, int32_t n_ranks,
                        ss_dtype gdtype, float post_scale, double* sumsq_out, void* workspace,
                        int64_t workspace_bytes, float* g_out, int32_t* nonfinite_flag, void* stream);
ss_status ss_clip_coef(const double* shard_sumsq, int32_t n_shards, float max_norm, float* coef_out,
                       double* norm_out, void* stream);

/* ------------------------------------------ sum of squares without allocation
 * No counterpart on the pages: an addition for callers that cannot allocate
 * device memory -- for instance plugin code running inside another framework
 * that has already reserved the GPU's memory for its own pool, or a
 * latency-critical loop where cudaMalloc's implicit device synchronisation is
 * not acceptable -- and so cannot provide ss_grad_sumsq's workspace.
 *
 * ss_grad_sumsq_noalloc computes exactly what ss_grad_sumsq computes (same
 * kernels, same bits) but keeps its scratch in a fixed array inside the
 * library: SS_NOALLOC_SUMSQ_SLOTS doubles (512 KiB), held on every GPU that
 * loads the library until the process exits. It allocates nothing and frees
 * nothing. The caller still passes the inputs and outputs, as for
 * ss_grad_sumsq.
 *   - n may be at most SS_NOALLOC_SUMSQ_MAX_N (1,073,709,056 elements);
 *     larger n returns SS_ERR_OVERFLOW and launches nothing.
 *   - The first call on a device looks up the array's device address with
 *     the runtime (no allocation) and caches it for the device's CUDA
 *     context; make that first call before any stream capture on that
 *     device. A device reset (cudaDeviceReset) ends the context and with it
 *     the array's contents and address: the next call looks the address up
 *     again, so make it, too, outside a stream capture.
 *   - All calls share the one array: calls whose kernels may overlap on the
 *     GPU (different streams without ordering) race and give wrong results.
 *     Calls ordered on one stream are safe; nothing has to be cleared between
 *     them. */
#define SS_NOALLOC_SUMSQ_SLOTS 65536
#define SS_NOALLOC_SUMSQ_MAX_N ((int64_t)(SS_NOALLOC_SUMSQ_SLOTS - 2) * 16384)
ss_status ss_grad_sumsq_noalloc(int64_t n, const float* g32, const void* const* rank_grads, int32_t n_ranks,
                                ss_dtype gdtype, float post_scale, double* sumsq_out, float* g_out,
                                int32_t* nonfinite_flag, void* stream);

/* ----------------------------------------------------------------- unshard
 * "FSDP: Fully Sharded Data Parallel Training at Scale", the unit's
 * communication cycle (forward and backward all-gather): the full flat unit is
 * the concatenation of the N shards in rank order.
 *
 * ss_unshard: shards [n_ranks] (host array of device pointers; shard k holds
 *   shard_bounds[k+1]-shard_bounds[k] elements) -> flat [P] (device), shard k
 *   written at shard_bounds[k]. shard_bounds [n_ranks+1] (host, non-decreasing,
 *   shard_bounds[0] = 0). dtype: SS_BF16, SS_FP16 or SS_FP32. One launch.
 * ss_reshard: the reverse copy, flat -> shards.
 * Bit-exact copies. Shards must not overlap the flat buffer or each other.
 * 16-byte vector stores aligned on the destination; a shard whose place in
 * the flat buffer is not at its own 16-byte phase is read as aligned 16-byte
 * chunks and shifted in registers (same results, about the same bandwidth). */
ss_status ss_unshard(const void* const* shards, const int64_t* shard_bounds, int32_t n_ranks, ss_dtype dtype,
                     void* flat, void* stream);
ss_status ss_reshard(const void* flat, const int64_t* shard_bounds, int32_t n_ranks, ss_dtype dtype,
                     void* const* shards, void* stream);

/* ------------------------------------------------------------------- misc */
const char* ss_status_string(ss_status s);      /* static string, never NULL */
const char* ss_last_cuda_error(void);           /* last CUDA error text of this thread ("" if none) */

int32_t ss_abi_version(void);                   /* SS_ABI_VERSION */

#ifdef __cplusplus
}
#endif
#endif /* SS_H */
