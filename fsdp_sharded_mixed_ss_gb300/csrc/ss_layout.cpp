// ss_layout.cpp -- host-side parts of the shard-step ABI: the flat layout and
// shard-boundary indexer, the training-state byte accounting, status strings.
//
// Layout rule ("FSDP: Fully Sharded Data Parallel Training at Scale", how a
// layer is sharded): rank k owns flat elements [floor(kP/N), floor((k+1)P/N)).
#include <cstdint>
#include <cstring>

#include "../../include/ss.h"

namespace {

// floor(k * P / N) without overflow: k <= N <= 2^30 and P < 2^63 need 93 bits.
inline int64_t bound(int64_t k, int64_t P, int64_t N) {
  return static_cast<int64_t>((static_cast<__int128>(k) * P) / N);
}

}  // namespace

extern "C" {

ss_status ss_flatten_layout(const int64_t* numels, int32_t n_tensors, int32_t n_ranks, int64_t* tensor_offsets,
                            int64_t* shard_bounds) {
  if (n_tensors < 0 || n_ranks < 1 || n_ranks > (1 << 30) || !tensor_offsets || !shard_bounds ||
      (n_tensors > 0 && !numels))
    return SS_ERR_INVALID_ARG;
  int64_t P = 0;
  for (int32_t t = 0; t < n_tensors; ++t)
    if (numels[t] < 0) return SS_ERR_INVALID_ARG;
  for (int32_t t = 0; t < n_tensors; ++t) {
    if (numels[t] > INT64_MAX - P) return SS_ERR_OVERFLOW;
    P += numels[t];
  }
  int64_t off = 0;
  tensor_offsets[0] = 0;
  for (int32_t t = 0; t < n_tensors; ++t) {
    off += numels[t];
    tensor_offsets[t + 1] = off;
  }
  for (int32_t k = 0; k <= n_ranks; ++k) shard_bounds[k] = bound(k, P, n_ranks);
  return SS_OK;
}

int32_t ss_shard_of(int64_t P, int32_t n_ranks, int64_t i) {
  if (n_ranks < 1 || P < 0 || i < 0 || i >= P) return -1;
  // i is in shard k iff floor(kP/N) <= i < floor((k+1)P/N), i.e. k*P < (i+1)*N <= (k+1)*P,
  // so k = ceil((i+1)N/P) - 1 = floor(((i+1)N - 1)/P).
  __int128 num = static_cast<__int128>(i + 1) * n_ranks - 1;
  return static_cast<int32_t>(num / P);
}

ss_status ss_shard_segments(const int64_t* tensor_offsets, int32_t n_tensors, const int64_t* shard_bounds,
                            int32_t n_ranks, int32_t shard, ss_segment* out, int32_t capacity, int32_t* count) {
  if (!tensor_offsets || !shard_bounds || !count || n_tensors < 0 || n_ranks < 1 || shard < 0 || shard >= n_ranks)
    return SS_ERR_INVALID_ARG;
  const int64_t lo = shard_bounds[shard], hi = shard_bounds[shard + 1];
  if (lo > hi) return SS_ERR_INVALID_ARG;
  // tensors are sorted by offset: find the first tensor that ends after lo (binary search)
  int32_t a = 0, b = n_tensors;
  while (a < b) {
    int32_t mid = a + (b - a) / 2;
    if (tensor_offsets[mid + 1] <= lo) a = mid + 1;
    else b = mid;
  }
  int32_t c = 0;
  bool overflow = false;
  for (int32_t t = a; t < n_tensors && tensor_offsets[t] < hi; ++t) {
    int64_t s = tensor_offsets[t] > lo ? tensor_offsets[t] : lo;
    int64_t e = tensor_offsets[t + 1] < hi ? tensor_offsets[t + 1] : hi;
    if (e <= s) continue;  // empty tensor
    if (out) {
      if (c < capacity) {
        out[c].tensor = t;
        out[c].pad_ = 0;
        out[c].tensor_offset = s - tensor_offsets[t];
        out[c].shard_offset = s - lo;
        out[c].length = e - s;
      } else {
        overflow = true;
      }
    }
    ++c;
  }
  *count = c;
  return overflow ? SS_ERR_INVALID_ARG : SS_OK;
}

ss_status ss_state_bytes(int64_t P, int32_t n_ranks, int32_t n_units, ss_bytes* out) {
  if (P < 0 || n_ranks < 1 || n_units < 1 || !out) return SS_ERR_INVALID_ARG;
  const double p = static_cast<double>(P), N = n_ranks, M = n_units;
  std::memset(out, 0, sizeof *out);
  // fp32 training: parameters, gradients, Adam's two moments
  out->fp32_params = 4.0 * p;
  out->fp32_grads = 4.0 * p;
  out->fp32_adam = 8.0 * p;
  out->fp32_total = 16.0 * p;
  // mixed precision: 16-bit params and grads, fp32 master and moments
  out->mp_params16 = 2.0 * p;
  out->mp_grads16 = 2.0 * p;
  out->mp_master32 = 4.0 * p;
  out->mp_adam32 = 8.0 * p;
  out->mp_total = 16.0 * p;
  out->optimizer_state = 12.0 * p;
  out->zero1_optimizer_per_gpu = 12.0 * p / N;
  // per-GPU steady state by strategy (fp32 accounting)
  out->full_shard_per_gpu = 16.0 * p / N;
  out->shard_grad_op_per_gpu = 4.0 * p + 12.0 * p / N;
  out->no_shard_per_gpu = 16.0 * p;
  out->unit_gather = 4.0 * p / M;
  out->full_shard_peak = out->full_shard_per_gpu + out->unit_gather;
  out->full_shard_saving = 16.0 * p - out->full_shard_per_gpu;
  out->shard_grad_op_saving = 16.0 * p - out->shard_grad_op_per_gpu;
  out->mp_full_shard_per_gpu = 16.0 * p / N;
  out->mp_unit_gather16 = 2.0 * p / M;
  return SS_OK;
}

const char* ss_status_string(ss_status s) {
  switch (s) {
    case SS_OK: return "ok";
    case SS_ERR_INVALID_ARG: return "invalid argument";
    case SS_ERR_ALIGN: return "misaligned pointer";
    case SS_ERR_OVERLAP: return "overlapping buffers";
    case SS_ERR_DTYPE: return "unsupported dtype";
    case SS_ERR_OVERFLOW: return "size overflow";
    case SS_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

int32_t ss_abi_version(void) { return SS_ABI_VERSION; }

}  // extern "C"
