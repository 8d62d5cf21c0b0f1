// ss_reduce.cu -- the standalone virtual-rank gradient reduce (ss_grad_reduce):
// the fp32 rank-ordered sum of the ranks' 16-bit gradient shards, optionally
// scaled, accumulated into the output and checked for non-finite values. Three
// forms: 16-byte vectors when the ranks and the output share a 16-byte phase,
// warp-cooperative shifted loads when the ranks share a phase that is not the
// output's, element-wise otherwise.
#include "ss_common.cuh"

namespace ss {
namespace {

// ------------------------------------------------------------------ gradient reduce

template <int GT, int MAXR>
__device__ __forceinline__ void reduce_one(const ReduceArgs<MAXR>& a, int64_t e, bool& bad) {
  float g = reduce1<GT>(a.ranks, a.n_ranks, e);
  if (a.post_scale != 1.0f) g = g * a.post_scale;
  if (a.accumulate) g = a.out[e] + g;
  bad |= !finite(g);
  a.out[e] = g;
}

// With CHUNKED (up to kReduceChunkRanks ranks) one block of 1024 threads per SM
// whose warps take chunks of 32 groups from a shared counter (ChunkMap, round
// robin); otherwise a grid-stride loop at 4 blocks of 256 threads per SM.
// Measured on GB300 at 2^26 elements, chunked against grid-stride: +3.5% at
// N = 1, +1.8% at N = 2, +8% at N = 4, +0.4% at N = 8 (+2.2% accumulating),
// -1.5% at N = 64.
constexpr int kReduceChunkThreads = 1024;
constexpr int kReduceChunkRanks = 8;

template <int GT, int MAXR, bool CHUNKED>
__global__ void __launch_bounds__(CHUNKED ? kReduceChunkThreads : kThreads) reduce_vec_kernel(
    const __grid_constant__ ReduceArgs<MAXR> a) {
  __shared__ unsigned next_chunk;
  if constexpr (CHUNKED) {
    if (threadIdx.x == 0) next_chunk = 0;
    __syncthreads();
  }
  pdl_wait();
  pdl_trigger();
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  bool bad = false;
  auto group = [&](int64_t gi) {
    const int64_t e = a.head + gi * kGroup;
    float g[8];
    reduce8<GT>(a.ranks, a.n_ranks, e, g);
    if (a.post_scale != 1.0f) {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
    }
    if (a.accumulate) {
      float o[8];
      ld8f(a.out + e, o);
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = o[j] + g[j];
    }
    if (a.nonfinite) {
#pragma unroll
      for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
    }
    st8f(a.out + e, g);
  };
  if constexpr (CHUNKED) {
    const ChunkMap<kReduceChunkThreads / 32> map(nvec);
    const int lane = threadIdx.x & 31;
    for (int64_t c = map.take<false>(&next_chunk, lane); c < map.nchunk; c = map.take<false>(&next_chunk, lane)) {
      const int64_t gi = c * 32 + lane;
      if (gi < nvec) group(gi);
    }
  } else {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t gi = tid; gi < nvec; gi += stride) group(gi);
  }
  const int64_t tail0 = a.head + nvec * kGroup;
  if (tid < a.head + (a.n - tail0)) reduce_one<GT>(a, tid < a.head ? tid : tail0 + (tid - a.head), bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

template <int GT, int MAXR>
__global__ void __launch_bounds__(kThreads) reduce_scalar_kernel(const __grid_constant__ ReduceArgs<MAXR> a) {
  pdl_wait();
  pdl_trigger();
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t e = tid; e < a.n; e += stride) reduce_one<GT>(a, e, bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

// Rank gradients all at one 16-byte phase that is not the fp32 output's (views
// at an offset that is not a multiple of 8 elements into per-rank buffers,
// with the output allocated per shard): warp-cooperative runs of kRun groups
// (ss_common.cuh), the ranks' chunks loaded in batches of 8 and summed in rank
// order before the shift, so each gradient byte is loaded once; the output
// (and its old value when accumulating) stays in aligned 16-byte vectors.
// Groups 0 and nvec - 1 and the head/tail elements go one by one.
template <int MAXR>
struct ShiftReduceArgs {
  ReduceArgs<MAXR> s;
  int32_t rphase;  // byte offset of the ranks' group starts past a 16-byte boundary (even, nonzero)
};

template <int GT, int MAXR>
__global__ void __launch_bounds__(kReduceChunkThreads) reduce_shift_kernel(const __grid_constant__ ShiftReduceArgs<MAXR> x) {
  __shared__ unsigned next_run;
  if (threadIdx.x == 0) next_run = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const ReduceArgs<MAXR>& a = x.s;
  const int64_t nvec = (a.n - a.head) / kGroup;  // >= 3 on this path
  const int64_t runs = (nvec - 2 + kRun - 1) / kRun;
  const int sh = x.rphase >> 1;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kReduceChunkThreads / 32> map(runs * 32);  // one "chunk" per run
  bool bad = false;
  for (int64_t run = map.take<false>(&next_run, lane); run < runs; run = map.take<false>(&next_run, lane)) {
    const int64_t gi = 1 + run * kRun + lane;
    const int64_t gl = gi < nvec - 1 ? gi : nvec - 1;  // past the body: a chunk inside the arrays, unused
    const int64_t el = a.head + gl * kGroup;
    float g[8];
    for (int r0 = 0; r0 < a.n_ranks; r0 += 8) {
      uint4 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (r0 + j < a.n_ranks)
          w[j] = __ldcs(reinterpret_cast<const uint4*>(
              reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[r0 + j]) + el) - x.rphase));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (r0 + j < a.n_ranks) {
          if (r0 + j == 0) widen8<GT>(w[j], g);
          else add8<GT>(w[j], g);
        }
      }
    }
    shift_down8(g, sh);
    if (lane < kRun && gi < nvec - 1) {
      const int64_t e = a.head + gi * kGroup;
      if (a.post_scale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
      }
      if (a.accumulate) {
        float o[8];
        ld8f(a.out + e, o);
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = o[j] + g[j];
      }
      if (a.nonfinite) {
#pragma unroll
        for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
      }
      st8f(a.out + e, g);
    }
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t lo_end = a.head + kGroup, hi_start = a.head + (nvec - 1) * kGroup;
  const int64_t n_edge = lo_end + (a.n - hi_start);
  if (tid < n_edge) reduce_one<GT>(a, tid < lo_end ? tid : hi_start + (tid - lo_end), bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && lane == 0) *a.nonfinite = 1;
  }
}

// The same for 7 and 8 ranks, register double-buffered: the loads of a warp's
// next run (the ranks' chunks, and the output's old values when accumulating)
// are issued before the current run is summed and stored. One 512-thread block
// per SM. Measured on GB300 at 2^26 elements with the views one element off:
// 7 ranks 6697 GB/s against 6617 single-buffered, 8 ranks 6815 against 6451;
// with fewer ranks the single-buffered form's 1024-thread blocks were faster
// (1-6 ranks 4502-6815 against 4133-6467).
template <int NR>
struct ShiftReduceGroup {
  uint4 r[NR];
  float4 o[2];  // the output's old values (accumulating only)
};

template <int GT, int MAXR, int NR>
__device__ __forceinline__ void reduce_shift_load(const ShiftReduceArgs<MAXR>& x, int64_t run, int lane, int64_t nvec,
                                                  ShiftReduceGroup<NR>& G) {
  const ReduceArgs<MAXR>& a = x.s;
  const int64_t gi = 1 + run * kRun + lane;
  const int64_t gl = gi < nvec - 1 ? gi : nvec - 1;  // past the body: a chunk inside the arrays, unused
  const int64_t el = a.head + gl * kGroup;
#pragma unroll
  for (int r = 0; r < NR; ++r)
    G.r[r] = __ldcs(reinterpret_cast<const uint4*>(
        reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[r]) + el) - x.rphase));
  if (a.accumulate && lane < kRun) {
    const int64_t gb = gi < nvec - 2 ? gi : nvec - 2;  // a body group's old values
    G.o[0] = __ldcs(reinterpret_cast<const float4*>(a.out + a.head + gb * kGroup));
    G.o[1] = __ldcs(reinterpret_cast<const float4*>(a.out + a.head + gb * kGroup) + 1);
  }
}

template <int GT, int MAXR, int NR>
__global__ void __launch_bounds__(kChunkThreads, kChunkBlocksPerSm) reduce_shift_pipe_kernel(
    const __grid_constant__ ShiftReduceArgs<MAXR> x) {
  __shared__ unsigned next_run;
  if (threadIdx.x == 0) next_run = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const ReduceArgs<MAXR>& a = x.s;
  const int64_t nvec = (a.n - a.head) / kGroup;  // >= 3 on this path
  const int64_t runs = (nvec - 2 + kRun - 1) / kRun;
  const int sh = x.rphase >> 1;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kChunkWarps> map(runs * 32);  // one "chunk" per run
  bool bad = false;
  ShiftReduceGroup<NR> cur, nxt;
  int64_t run = map.take<false>(&next_run, lane);
  if (run < runs) reduce_shift_load<GT>(x, run, lane, nvec, cur);
  while (run < runs) {  // warp-uniform
    const int64_t rn = map.take<false>(&next_run, lane);
    if (rn < runs) reduce_shift_load<GT>(x, rn, lane, nvec, nxt);
    float g[8];
    widen8<GT>(cur.r[0], g);
#pragma unroll
    for (int r = 1; r < NR; ++r) add8<GT>(cur.r[r], g);
    shift_down8(g, sh);
    const int64_t gi = 1 + run * kRun + lane;
    if (lane < kRun && gi < nvec - 1) {
      const int64_t e = a.head + gi * kGroup;
      if (a.post_scale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
      }
      if (a.accumulate) {
        const float o[8] = {cur.o[0].x, cur.o[0].y, cur.o[0].z, cur.o[0].w, cur.o[1].x, cur.o[1].y, cur.o[1].z, cur.o[1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = o[j] + g[j];
      }
      if (a.nonfinite) {
#pragma unroll
        for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
      }
      st8f(a.out + e, g);
    }
    cur = nxt;
    run = rn;
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t lo_end = a.head + kGroup, hi_start = a.head + (nvec - 1) * kGroup;
  const int64_t n_edge = lo_end + (a.n - hi_start);
  if (tid < n_edge) reduce_one<GT>(a, tid < lo_end ? tid : hi_start + (tid - lo_end), bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && lane == 0) *a.nonfinite = 1;
  }
}

template <int G, int MAXR, int NR>
ss_status launch_reduce_shift_pipe(const ShiftReduceArgs<MAXR>& x, int64_t runs, void* stream) {
  auto* fn = reduce_shift_pipe_kernel<G, MAXR, NR>;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), runs * 32, kChunkThreads), x, stream, kChunkThreads);
}


template <int MAXR>
ss_status run_reduce_shift(const ReduceArgs<MAXR>& a, int rphase, ss_dtype gt, void* stream) {
  ShiftReduceArgs<MAXR> x;
  std::memset(&x, 0, sizeof x);
  x.s = a;
  x.rphase = rphase;
  const int64_t runs = ((a.n - a.head) / kGroup - 2 + kRun - 1) / kRun;
#define SS_REDP(G, R) \
  case R: return launch_reduce_shift_pipe<G, MAXR, R>(x, runs, stream);
#define SS_REDS_CASE(G)                                                                              \
  if (gt == G) {                                                                                     \
    if constexpr (MAXR == kSmallRanks) {                                                             \
      switch (a.n_ranks) {                                                                           \
        SS_REDP(G, 7) SS_REDP(G, 8)                                                                  \
        default: break;                                                                              \
      }                                                                                              \
    }                                                                                                \
    auto* fn = reduce_shift_kernel<G, MAXR>;                                                         \
    return launch(fn, grid_for(reinterpret_cast<const void*>(fn), runs * 32, kReduceChunkThreads), x, stream, \
                  kReduceChunkThreads);                                                              \
  }
  SS_REDS_CASE(SS_BF16)
  SS_REDS_CASE(SS_FP16)
#undef SS_REDS_CASE
#undef SS_REDP
  return SS_ERR_DTYPE;
}

template <int MAXR>
ss_status run_reduce(const ReduceArgs<MAXR>& a, bool vec, ss_dtype gt, void* stream) {
#define SS_RED_CASE(G)                                                                     \
  if (gt == G) {                                                                           \
    if (vec && a.n_ranks <= kReduceChunkRanks) {                                           \
      auto* fn = reduce_vec_kernel<G, MAXR, true>;                                         \
      return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup, kReduceChunkThreads), \
                    a, stream, kReduceChunkThreads);                                       \
    }                                                                                      \
    if (vec) {                                                                             \
      auto* fn = reduce_vec_kernel<G, MAXR, false>;                                        \
      return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup), a, stream); \
    }                                                                                      \
    auto* fn = reduce_scalar_kernel<G, MAXR>;                                              \
    return launch(fn, grid_for(reinterpret_cast<const void*>(fn), a.n), a, stream);        \
  }
  SS_RED_CASE(SS_BF16)
  SS_RED_CASE(SS_FP16)
#undef SS_RED_CASE
  return SS_ERR_DTYPE;
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" {

ss_status ss_grad_reduce(const void* const* rank_grads, int32_t n_ranks, ss_dtype gdtype, int64_t n,
                         float post_scale, int32_t accumulate, float* g_out, int32_t* nonfinite_flag,
                         void* stream) {
  if (n < 0) return SS_ERR_INVALID_ARG;
  if (n > INT64_MAX / 16) return SS_ERR_OVERFLOW;
  std::vector<Range> ranges;
  std::vector<uintptr_t> p16, p32;
  ss_status st = check_ranks(rank_grads, n_ranks, gdtype, n, ranges, p16);
  if (st != SS_OK) return st;
  if (!g_out) return SS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(g_out) & 3u) return SS_ERR_ALIGN;
  if (nonfinite_flag && (reinterpret_cast<uintptr_t>(nonfinite_flag) & 3u)) return SS_ERR_ALIGN;
  ranges.push_back(rng(g_out, 4 * n, true));
  if (nonfinite_flag) ranges.push_back(rng(nonfinite_flag, 4, true));
  if (any_output_overlap(ranges)) return SS_ERR_OVERLAP;
  if (n == 0) return SS_OK;
  p32.push_back(reinterpret_cast<uintptr_t>(g_out));
  const int h = common_phase(p16, p32);
  const bool vec = h >= 0 && h < n;
  // the ranks at one phase, the output at another: groups aligned for the output, the
  // ranks read by the warp-cooperative shifted loads
  int64_t head = vec ? h : 0;
  int rphase = 0;
  if (!vec && common_phase(p16, {}) >= 0) {
    const int h32 = common_phase({}, p32);
    if (h32 >= 0 && n - h32 >= 3 * kGroup) {
      head = h32;
      rphase = static_cast<int>((reinterpret_cast<uintptr_t>(rank_grads[0]) + 2u * h32) & 15u);
    }
  }
  auto fill = [&](auto& a) {
    for (int32_t r = 0; r < n_ranks; ++r) a.ranks.p[r] = rank_grads[r];
    a.out = g_out;
    a.nonfinite = nonfinite_flag;
    a.n = n;
    a.head = head;
    a.n_ranks = n_ranks;
    a.post_scale = post_scale;
    a.accumulate = accumulate != 0;
  };
  if (n_ranks <= kSmallRanks) {
    ReduceArgs<kSmallRanks> a;
    std::memset(&a, 0, sizeof a);
    fill(a);
    return rphase ? run_reduce_shift(a, rphase, gdtype, stream) : run_reduce(a, vec, gdtype, stream);
  }
  ReduceArgs<kLargeRanks> a;
  std::memset(&a, 0, sizeof a);
  fill(a);
  return rphase ? run_reduce_shift(a, rphase, gdtype, stream) : run_reduce(a, vec, gdtype, stream);
}

}  // extern "C"
