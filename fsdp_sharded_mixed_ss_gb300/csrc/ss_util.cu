// ss_util.cu -- host helpers shared by the entry points: argument range and
// overlap checks, the arrays' common 16-byte phase, persistent grid sizing, and
// the per-thread CUDA error text.
#include "ss_common.cuh"

namespace ss {

thread_local char g_cuda_err[256] = "";

ss_status cuda_fail(cudaError_t e) {
  std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return SS_ERR_CUDA;
}

bool any_output_overlap(std::vector<Range>& rs) {
  rs.erase(std::remove_if(rs.begin(), rs.end(), [](const Range& r) { return r.hi <= r.lo; }), rs.end());
  std::sort(rs.begin(), rs.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
  uintptr_t max_out = 0, max_any = 0;
  for (const Range& r : rs) {
    if (r.lo < max_out) return true;
    if (r.out && r.lo < max_any) return true;
    max_any = std::max(max_any, r.hi);
    if (r.out) max_out = std::max(max_out, r.hi);
  }
  return false;
}

Range rng(const void* p, int64_t bytes, bool out) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + static_cast<uintptr_t>(bytes), out};
}

int common_phase(const std::vector<uintptr_t>& p16, const std::vector<uintptr_t>& p32) {
  for (int h = 0; h < 8; ++h) {
    bool ok = true;
    for (uintptr_t p : p16) ok = ok && ((p + 2u * h) & 15u) == 0;
    for (uintptr_t p : p32) ok = ok && ((p + 4u * h) & 15u) == 0;
    if (ok) return h;
  }
  return -1;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int blocks_per_sm(const void* fn, int threads) {
  struct Entry {
    int dev;
    const void* fn;
    int threads, blocks;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& c : cache)
    if (c.dev == dev && c.fn == fn && c.threads == threads) return c.blocks;
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, 0) != cudaSuccess || b < 1) b = 1;
  cache.push_back({dev, fn, threads, b});
  return b;
}

unsigned grid_for(const void* fn, int64_t work_items, int threads) {
  const int64_t want = std::max<int64_t>(1, (work_items + threads - 1) / threads);
  const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>(sm_count()) * blocks_per_sm(fn, threads));
  return static_cast<unsigned>(std::min(want, cap));
}

ss_status check_ranks(const void* const* rank_grads, int32_t n_ranks, ss_dtype gdtype, int64_t n,
                      std::vector<Range>& ranges, std::vector<uintptr_t>& p16) {
  if (!rank_grads || n_ranks < 1 || n_ranks > SS_MAX_RANKS) return SS_ERR_INVALID_ARG;
  if (!is16(gdtype)) return SS_ERR_DTYPE;
  for (int32_t r = 0; r < n_ranks; ++r) {
    if (!rank_grads[r]) return SS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(rank_grads[r]) & 1u) return SS_ERR_ALIGN;
    ranges.push_back(rng(rank_grads[r], 2 * n, false));
    p16.push_back(reinterpret_cast<uintptr_t>(rank_grads[r]));
  }
  return SS_OK;
}

}  // namespace ss

extern "C" const char* ss_last_cuda_error(void) { return ss::g_cuda_err; }
