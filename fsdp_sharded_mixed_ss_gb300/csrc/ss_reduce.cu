// ss_reduce.cu -- the standalone virtual-rank gradient reduce (ss_grad_reduce):
// the fp32 rank-ordered sum of the ranks' 16-bit gradient shards, optionally
// scaled, accumulated into the output and checked for non-finite values. Three
// forms: 16-byte vectors when the ranks and the output share a 16-byte phase,
// warp-cooperative shifted loads when the output has a phase the ranks do not
// share (at one phase or each at its own), element-wise otherwise (an output
// that is not 16-byte aligned after any whole number of elements, or fewer than
// three 8-element groups).
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

// Few ranks, warp-contiguous accesses: lane i takes elements 4i..4i+3 and
// 128+4i..128+4i+3 of its warp's 256-element chunk, so every 16-byte access of
// a warp to the fp32 output (the store, and the old values' load when
// accumulating) covers 512 contiguous bytes -- whole 32-byte sectors, where the
// 8-element groups of reduce_vec_kernel leave each instruction half of every
// sector it touches -- and every 8-byte gradient load reads 256. Measured on
// GB300 at 2^26 elements against reduce_vec_kernel: 1 rank 0.84 -> 0.87 of the
// copy peak; accumulating, 1 / 2 / 3 ranks 0.87 / 0.95 / 0.99 -> 0.93 / 1.01 /
// 1.02; without accumulating 2 and 3 ranks measured slower (0.90 / 0.93 against
// 0.95 / 1.01: the halved gradient loads), 4 ranks the same.
// Which rank counts (bit N: N ranks, 1-4) take it, not accumulating and accumulating.
#ifndef SS_RED_QUAD_MASK
#define SS_RED_QUAD_MASK (1u << 1)
#endif
#ifndef SS_RED_QUAD_ACC_MASK
#define SS_RED_QUAD_ACC_MASK ((1u << 2) | (1u << 3))
#endif
static_assert(((SS_RED_QUAD_MASK | SS_RED_QUAD_ACC_MASK) & ~0x1Eu) == 0, "quad forms exist for 1-4 ranks");
template <int GT, int MAXR, int NR, bool ACC>
__global__ void __launch_bounds__(kReduceChunkThreads) reduce_quad_kernel(const __grid_constant__ ReduceArgs<MAXR> a) {
  __shared__ unsigned next_chunk;
  if (threadIdx.x == 0) next_chunk = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kReduceChunkThreads / 32> map(nvec);
  bool bad = false;
  for (int64_t c = map.take<false>(&next_chunk, lane); c < map.nchunk; c = map.take<false>(&next_chunk, lane)) {
    uint2 w[2][NR];
    float4 o[2];
    bool ok[2];
    int64_t e[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      ok[h] = c * 32 + 16 * h + lane / 2 < nvec;  // the lane's quad h lies in group 16h + lane/2 of the chunk
      e[h] = a.head + c * 32 * kGroup + 128 * h + 4 * lane;
      if (ok[h]) {
#pragma unroll
        for (int r = 0; r < NR; ++r)
          w[h][r] = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.ranks.p[r]) + e[h]));
        if (ACC) o[h] = __ldcs(reinterpret_cast<const float4*>(a.out + e[h]));
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!ok[h]) continue;
      float2 lo = widen2<GT>(w[h][0].x), hi = widen2<GT>(w[h][0].y);
      float g[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
      for (int r = 1; r < NR; ++r) {
        lo = widen2<GT>(w[h][r].x);
        hi = widen2<GT>(w[h][r].y);
        g[0] = g[0] + lo.x; g[1] = g[1] + lo.y; g[2] = g[2] + hi.x; g[3] = g[3] + hi.y;
      }
      if (a.post_scale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 4; ++j) g[j] = g[j] * a.post_scale;
      }
      if (ACC) {
        g[0] = o[h].x + g[0]; g[1] = o[h].y + g[1]; g[2] = o[h].z + g[2]; g[3] = o[h].w + g[3];
      }
      if (a.nonfinite) {
#pragma unroll
        for (int j = 0; j < 4; ++j) bad |= !finite(g[j]);
      }
      __stcs(reinterpret_cast<float4*>(a.out + e[h]), make_float4(g[0], g[1], g[2], g[3]));
    }
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t tail0 = a.head + nvec * kGroup;
  if (tid < a.head + (a.n - tail0)) reduce_one<GT>(a, tid < a.head ? tid : tail0 + (tid - a.head), bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && lane == 0) *a.nonfinite = 1;
  }
}

template <int G, int MAXR, int NR, bool ACC>
ss_status launch_reduce_quad(const ReduceArgs<MAXR>& a, void* stream) {
  auto* fn = reduce_quad_kernel<G, MAXR, NR, ACC>;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup, kReduceChunkThreads), a,
                stream, kReduceChunkThreads);
}

// The quad form for this call, if it takes one (16-byte vectors, the small rank table).
template <int G, int MAXR>
bool reduce_quad(const ReduceArgs<MAXR>& a, ss_status& st, void* stream) {
  if constexpr (MAXR != kSmallRanks) {
    return false;
  } else {
#define SS_RED_QUAD(R)                                                                                       \
  if (a.n_ranks == R) {                                                                                      \
    if constexpr ((SS_RED_QUAD_ACC_MASK >> R) & 1u)                                                          \
      if (a.accumulate) return st = launch_reduce_quad<G, MAXR, R, true>(a, stream), true;                   \
    if constexpr ((SS_RED_QUAD_MASK >> R) & 1u)                                                              \
      if (!a.accumulate) return st = launch_reduce_quad<G, MAXR, R, false>(a, stream), true;                 \
  }
    SS_RED_QUAD(1) SS_RED_QUAD(2) SS_RED_QUAD(3) SS_RED_QUAD(4)
#undef SS_RED_QUAD
    return false;
  }
}

// The chunked form with the rank count and accumulation fixed at compile time,
// each warp's sums stored through shared memory as consecutive 16-byte vectors
// (vector f of a chunk holds elements 4f..4f+3 of its 32 groups) and, when
// accumulating, the old values loaded in that layout with the gradients. It
// keeps the 16-byte gradient loads that the quad form halves. Measured on
// GB300 at 2^26 elements against the quad and chunked forms: 2 ranks 0.95 ->
// 0.96-0.97, 1 rank accumulating 0.93 -> 0.99-1.00; 2-3 ranks accumulating
// 0.97 / 1.02 against the quad form's 1.01 / 1.03; 3-8 ranks within 1%.
#ifndef SS_RED_VEC_TX_MASK
#define SS_RED_VEC_TX_MASK (1u << 2)  // bit N: N ranks (1-8), not accumulating
#endif
#ifndef SS_RED_VEC_TX_ACC_MASK
#define SS_RED_VEC_TX_ACC_MASK (1u << 1)  // the same, accumulating
#endif
template <int GT, int MAXR, int NR, bool ACC>
__global__ void __launch_bounds__(kReduceChunkThreads) reduce_vec_tx_kernel(const __grid_constant__ ReduceArgs<MAXR> a) {
  __shared__ unsigned next_chunk;
  __shared__ float4 tx[kReduceChunkThreads / 32][64];
  if (threadIdx.x == 0) next_chunk = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int lane = threadIdx.x & 31;
  float4* t = tx[threadIdx.x >> 5];
  const ChunkMap<kReduceChunkThreads / 32> map(nvec);
  bool bad = false;
  for (int64_t c = map.take<false>(&next_chunk, lane); c < map.nchunk; c = map.take<false>(&next_chunk, lane)) {
    const int64_t gi = c * 32 + lane;
    const int64_t cb = a.head + c * 32 * kGroup;  // the chunk's first element
    uint4 w[NR];
    float4 ot[2];
    if (gi < nvec) {
#pragma unroll
      for (int r = 0; r < NR; ++r)
        w[r] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.ranks.p[r]) + cb + lane * kGroup));
    }
    if (ACC) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = lane + 32 * k;
        if (c * 32 + f / 2 < nvec) ot[k] = __ldcs(reinterpret_cast<const float4*>(a.out + cb + 4 * f));
      }
    }
    float g[8];
    widen8<GT>(w[0], g);
#pragma unroll
    for (int r = 1; r < NR; ++r) add8<GT>(w[r], g);
    t[2 * lane] = make_float4(g[0], g[1], g[2], g[3]);
    t[2 * lane + 1] = make_float4(g[4], g[5], g[6], g[7]);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int f = lane + 32 * k;
      if (c * 32 + f / 2 < nvec) {
        float4 v = t[f];
        if (a.post_scale != 1.0f) {
          v.x = v.x * a.post_scale; v.y = v.y * a.post_scale; v.z = v.z * a.post_scale; v.w = v.w * a.post_scale;
        }
        if (ACC) {
          v.x = ot[k].x + v.x; v.y = ot[k].y + v.y; v.z = ot[k].z + v.z; v.w = ot[k].w + v.w;
        }
        if (a.nonfinite) bad |= !finite(v.x) || !finite(v.y) || !finite(v.z) || !finite(v.w);
        __stcs(reinterpret_cast<float4*>(a.out + cb + 4 * f), v);
      }
    }
    __syncwarp();
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t tail0 = a.head + nvec * kGroup;
  if (tid < a.head + (a.n - tail0)) reduce_one<GT>(a, tid < a.head ? tid : tail0 + (tid - a.head), bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && lane == 0) *a.nonfinite = 1;
  }
}

template <int G, int MAXR>
bool reduce_vec_tx(const ReduceArgs<MAXR>& a, ss_status& st, void* stream) {
  if constexpr (MAXR != kSmallRanks || (SS_RED_VEC_TX_MASK | SS_RED_VEC_TX_ACC_MASK) == 0) {
    return false;
  } else {
    auto go = [&](auto* fn) {
      st = launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup, kReduceChunkThreads), a,
                  stream, kReduceChunkThreads);
      return true;
    };
#define SS_RED_TX(R)                                                                                          \
  if (a.n_ranks == R) {                                                                                       \
    if constexpr ((SS_RED_VEC_TX_ACC_MASK >> R) & 1u)                                                         \
      if (a.accumulate) return go(reduce_vec_tx_kernel<G, MAXR, R, true>);                                    \
    if constexpr ((SS_RED_VEC_TX_MASK >> R) & 1u)                                                             \
      if (!a.accumulate) return go(reduce_vec_tx_kernel<G, MAXR, R, false>);                                  \
  }
    SS_RED_TX(1) SS_RED_TX(2) SS_RED_TX(3) SS_RED_TX(4) SS_RED_TX(5) SS_RED_TX(6) SS_RED_TX(7) SS_RED_TX(8)
#undef SS_RED_TX
    return false;
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

// Rank gradients off the fp32 output's 16-byte phase (views at an offset that
// is not a multiple of 8 elements into per-rank buffers, with the output
// allocated per shard): warp-cooperative runs of kRun groups (ss_common.cuh).
// Ranks at one phase: their chunks are summed in rank order, then shifted once;
// ranks at mixed phases: each rank's packed chunk is moved into place by its
// own phase before it is added -- the same fp32 additions in the same order
// either way. Each gradient byte is loaded once; the output (and its old value
// when accumulating) stays in aligned 16-byte vectors. Groups 0 and nvec - 1
// and the head/tail elements go one by one.
//
// The forms differ in how they keep enough bytes in flight:
//  * 1-2 ranks: a warp takes U adjacent runs at a time and issues all their
//    loads before the first is summed (one 1024-thread block per SM), and
//    stores the sums through shared memory as warp-contiguous vectors
//    (tx_store_run). With one run at a time the loads in flight per SM were too
//    few: measured on GB300 at 2^26 elements, one element off, 1 rank 0.67 of
//    the copy peak -> 0.81 with U = 4 (0.76 with U = 8: fewer, larger batches
//    end less evenly) -> 0.88-0.89 with the contiguous stores, 2 ranks 0.80 ->
//    0.88 with U = 2 (0.83 with U = 4) -> 0.94; accumulating 0.87-0.88 ->
//    0.92-0.93. 3-4 ranks measured slower this way (0.93 against 0.94-0.99; the
//    contiguous stores in the any-rank form cost 3-5% there) and take the
//    any-rank form, except 3 ranks at mixed phases not accumulating.
//  * 7-8 ranks at one phase: register double-buffered (the next run's loads
//    issued before the current run is summed and stored), one 512-thread block
//    per SM. At mixed phases 8 ranks measured 0.87 there, so they take the
//    any-rank form.
//  * otherwise: batches of rank chunks, all loads of a batch before its adds,
//    the old output values requested with the first batch; one 1024-thread
//    block per SM.
template <int MAXR>
struct ShiftReduceArgs {
  ReduceArgs<MAXR> s;
  uint8_t rphase[MAXR];  // byte offset of each rank's group starts past a 16-byte boundary (even)
};

// Scale, old value (accumulating), finiteness check and store of one body group's sums.
template <int MAXR>
__device__ __forceinline__ void reduce_store8(const ReduceArgs<MAXR>& a, int64_t e, float (&g)[8],
                                              const float4 (&o)[2], bool acc, bool& bad) {
  if (a.post_scale != 1.0f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
  }
  if (acc) {
    const float ov[8] = {o[0].x, o[0].y, o[0].z, o[0].w, o[1].x, o[1].y, o[1].z, o[1].w};
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = ov[j] + g[j];
  }
  if (a.nonfinite) {
#pragma unroll
    for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
  }
  st8f(a.out + e, g);
}

// The groups outside the body [1, nvec - 1) and the head/tail elements, one per
// thread, then the block's non-finite flag (all threads call it).
template <int GT, int MAXR>
__device__ __forceinline__ void reduce_shift_edges(const ReduceArgs<MAXR>& a, int64_t nvec, int lane, bool bad) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t lo_end = a.head + kGroup, hi_start = a.head + (nvec - 1) * kGroup;
  const int64_t n_edge = lo_end + (a.n - hi_start);
  if (tid < n_edge) reduce_one<GT>(a, tid < lo_end ? tid : hi_start + (tid - lo_end), bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && lane == 0) *a.nonfinite = 1;
  }
}

// One run's loads of one lane: the ranks' aligned 16-byte chunks and, when
// accumulating, its group's old output values.
template <int NR>
struct ShiftReduceGroup {
  uint4 r[NR];
  float4 o[2];
};

template <int GT, int MAXR, int NR, bool MIXED>
__device__ __forceinline__ void reduce_shift_load(const ShiftReduceArgs<MAXR>& x, int64_t run, int lane, int64_t nvec,
                                                  bool acc, ShiftReduceGroup<NR>& G) {
  const ReduceArgs<MAXR>& a = x.s;
  const int64_t gi = 1 + run * kRun + lane;
  const int64_t gl = gi < nvec - 1 ? gi : nvec - 1;  // past the body: a chunk inside the arrays, unused
  const int64_t el = a.head + gl * kGroup;
#pragma unroll
  for (int r = 0; r < NR; ++r)
    G.r[r] = __ldcs(reinterpret_cast<const uint4*>(
        reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[r]) + el) - x.rphase[MIXED ? r : 0]));
  if (acc && lane < kRun) {
    const int64_t gb = gi < nvec - 2 ? gi : nvec - 2;  // a body group's old values
    G.o[0] = __ldcs(reinterpret_cast<const float4*>(a.out + a.head + gb * kGroup));
    G.o[1] = __ldcs(reinterpret_cast<const float4*>(a.out + a.head + gb * kGroup) + 1);
  }
}

// Sums one run's chunks in rank order, moves the sums into place and stores the lane's body group.
template <int GT, int MAXR, int NR, bool MIXED>
__device__ __forceinline__ void reduce_shift_group(const ShiftReduceArgs<MAXR>& x, const ShiftReduceGroup<NR>& G,
                                                   int64_t run, int lane, int64_t nvec, bool acc, bool& bad) {
  float g[8];
  if constexpr (MIXED) {
    widen8<GT>(shift_chunk(G.r[0], x.rphase[0] >> 1), g);
#pragma unroll
    for (int r = 1; r < NR; ++r) add8<GT>(shift_chunk(G.r[r], x.rphase[r] >> 1), g);
  } else {
    widen8<GT>(G.r[0], g);
#pragma unroll
    for (int r = 1; r < NR; ++r) add8<GT>(G.r[r], g);
    shift_down8(g, x.rphase[0] >> 1);
  }
  const int64_t gi = 1 + run * kRun + lane;
  if (lane < kRun && gi < nvec - 1) reduce_store8(x.s, x.s.head + gi * kGroup, g, G.o, acc, bad);
}

// Stores through shared memory: a run's sums pass through the warp's 64
// float4 slots so that the warp stores (and, accumulating, loads) the output as
// consecutive 16-byte vectors -- vector f of a run (f < 62) holds elements
// 4f..4f+3 of its 31 groups, and each instruction covers 512 contiguous bytes,
// where each lane storing its own group leaves every instruction half of each
// 32-byte sector it touches. tx_load_old: the run's old output values in that
// layout (accumulating); tx_store_run: scale, old value, check and store.
template <int MAXR>
__device__ __forceinline__ void tx_load_old(const ReduceArgs<MAXR>& a, int64_t run, int lane, int64_t nvec,
                                            float4 (&ot)[2]) {
  const int64_t e0 = a.head + (1 + run * kRun) * kGroup;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int f = lane + 32 * k;
    if (f < 2 * kRun && 1 + run * kRun + f / 2 < nvec - 1) ot[k] = __ldcs(reinterpret_cast<const float4*>(a.out + e0 + 4 * f));
  }
}

template <int MAXR>
__device__ __forceinline__ void tx_store_run(const ReduceArgs<MAXR>& a, float4* t, const float (&g)[8], int64_t run,
                                             int lane, int64_t nvec, bool acc, const float4 (&ot)[2], bool& bad) {
  t[2 * lane] = make_float4(g[0], g[1], g[2], g[3]);
  t[2 * lane + 1] = make_float4(g[4], g[5], g[6], g[7]);
  __syncwarp();
  const int64_t e0 = a.head + (1 + run * kRun) * kGroup;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int f = lane + 32 * k;
    if (f < 2 * kRun && 1 + run * kRun + f / 2 < nvec - 1) {
      float4 v = t[f];
      if (a.post_scale != 1.0f) {
        v.x = v.x * a.post_scale; v.y = v.y * a.post_scale; v.z = v.z * a.post_scale; v.w = v.w * a.post_scale;
      }
      if (acc) {
        v.x = ot[k].x + v.x; v.y = ot[k].y + v.y; v.z = ot[k].z + v.z; v.w = ot[k].w + v.w;
      }
      if (a.nonfinite) bad |= !finite(v.x) || !finite(v.y) || !finite(v.z) || !finite(v.w);
      __stcs(reinterpret_cast<float4*>(a.out + e0 + 4 * f), v);
    }
  }
  __syncwarp();  // the slots are free for the warp's next run
}

// The rank-ordered sum of one run's chunks, moved into place (all lanes).
template <int GT, int MAXR, int NR, bool MIXED>
__device__ __forceinline__ void shift_sum(const ShiftReduceArgs<MAXR>& x, const uint4 (&r)[NR], float (&g)[8]) {
  if constexpr (MIXED) {
    widen8<GT>(shift_chunk(r[0], x.rphase[0] >> 1), g);
#pragma unroll
    for (int k = 1; k < NR; ++k) add8<GT>(shift_chunk(r[k], x.rphase[k] >> 1), g);
  } else {
    widen8<GT>(r[0], g);
#pragma unroll
    for (int k = 1; k < NR; ++k) add8<GT>(r[k], g);
    shift_down8(g, x.rphase[0] >> 1);
  }
}

// Runs a warp takes at a time in the 1-4-rank form: enough loads in flight per
// SM without spilling in a 1024-thread block (64 registers a thread).
#ifndef SS_RED_BATCH_MAX_RANKS
#define SS_RED_BATCH_MAX_RANKS 2
#endif
#ifndef SS_RED_BATCH_RUNS_1
#define SS_RED_BATCH_RUNS_1 4
#endif
#ifndef SS_RED_BATCH_RUNS
#define SS_RED_BATCH_RUNS 2
#endif
__host__ __device__ constexpr int reduce_batch_runs(int nr, bool acc) {
  return acc ? (nr <= 2 ? 2 : 1) : (nr == 1 ? SS_RED_BATCH_RUNS_1 : SS_RED_BATCH_RUNS);
}

template <int GT, int MAXR, int NR, bool ACC, bool MIXED>
__global__ void __launch_bounds__(kReduceChunkThreads) reduce_shift_batch_kernel(
    const __grid_constant__ ShiftReduceArgs<MAXR> x) {
  constexpr int U = reduce_batch_runs(NR, ACC);
  __shared__ unsigned next_batch;
  __shared__ float4 tx[kReduceChunkThreads / 32][64];  // each warp's run of sums, for tx_store_run
  if (threadIdx.x == 0) next_batch = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int64_t nvec = (x.s.n - x.s.head) / kGroup;  // >= 3 on this path
  const int64_t runs = (nvec - 2 + kRun - 1) / kRun;
  const int64_t batches = (runs + U - 1) / U;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kReduceChunkThreads / 32> map(batches * 32);  // one "chunk" per U adjacent runs
  float4* t = tx[threadIdx.x >> 5];
  bool bad = false;
  for (int64_t b = map.take<false>(&next_batch, lane); b < batches; b = map.take<false>(&next_batch, lane)) {
    ShiftReduceGroup<NR> G[U];
    float4 ot[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      reduce_shift_load<GT, MAXR, NR, MIXED>(x, b * U + u, lane, nvec, false, G[u]);
      if (ACC) tx_load_old(x.s, b * U + u, lane, nvec, ot[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float g[8];
      shift_sum<GT, MAXR, NR, MIXED>(x, G[u].r, g);
      tx_store_run(x.s, t, g, b * U + u, lane, nvec, ACC, ot[u], bad);
    }
  }
  reduce_shift_edges<GT>(x.s, nvec, lane, bad);
}

// 7 and 8 ranks. Measured on GB300 at 2^26 elements with the views one element
// off: 7 ranks 6697 GB/s against 6617 in the any-rank form below, 8 ranks 6815
// against 6451; with 5-6 ranks the any-rank form's 1024-thread blocks were faster.
template <int GT, int MAXR, int NR, bool MIXED>
__global__ void __launch_bounds__(kChunkThreads, kChunkBlocksPerSm) reduce_shift_pipe_kernel(
    const __grid_constant__ ShiftReduceArgs<MAXR> x) {
  __shared__ unsigned next_run;
  if (threadIdx.x == 0) next_run = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int64_t nvec = (x.s.n - x.s.head) / kGroup;  // >= 3 on this path
  const int64_t runs = (nvec - 2 + kRun - 1) / kRun;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kChunkWarps> map(runs * 32);  // one "chunk" per run
  const bool acc = x.s.accumulate;
  bool bad = false;
  ShiftReduceGroup<NR> cur, nxt;
  int64_t run = map.take<false>(&next_run, lane);
  if (run < runs) reduce_shift_load<GT, MAXR, NR, MIXED>(x, run, lane, nvec, acc, cur);
  while (run < runs) {  // warp-uniform
    const int64_t rn = map.take<false>(&next_run, lane);
    if (rn < runs) reduce_shift_load<GT, MAXR, NR, MIXED>(x, rn, lane, nvec, acc, nxt);
    reduce_shift_group<GT, MAXR, NR, MIXED>(x, cur, run, lane, nvec, acc, bad);
    cur = nxt;
    run = rn;
  }
  reduce_shift_edges<GT>(x.s, nvec, lane, bad);
}

// Any rank count. Accumulating, the old values' registers leave room for
// batches of 6 rank chunks (8 spilled).
#ifndef SS_RED_ACC_BATCH
#define SS_RED_ACC_BATCH 6
#endif
template <int GT, int MAXR, bool ACC, bool MIXED>
__global__ void __launch_bounds__(kReduceChunkThreads) reduce_shift_kernel(const __grid_constant__ ShiftReduceArgs<MAXR> x) {
  constexpr int B = ACC ? SS_RED_ACC_BATCH : 8;
  __shared__ unsigned next_run;
  if (threadIdx.x == 0) next_run = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const ReduceArgs<MAXR>& a = x.s;
  const int64_t nvec = (a.n - a.head) / kGroup;  // >= 3 on this path
  const int64_t runs = (nvec - 2 + kRun - 1) / kRun;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kReduceChunkThreads / 32> map(runs * 32);  // one "chunk" per run
  bool bad = false;
  for (int64_t run = map.take<false>(&next_run, lane); run < runs; run = map.take<false>(&next_run, lane)) {
    const int64_t gi = 1 + run * kRun + lane;
    const int64_t gl = gi < nvec - 1 ? gi : nvec - 1;  // past the body: a chunk inside the arrays, unused
    const int64_t el = a.head + gl * kGroup;
    const bool body = lane < kRun && gi < nvec - 1;
    float g[8];
    float4 o[2];
    for (int r0 = 0; r0 < a.n_ranks; r0 += B) {
      uint4 w[B];
#pragma unroll
      for (int j = 0; j < B; ++j)
        if (r0 + j < a.n_ranks)
          w[j] = __ldcs(reinterpret_cast<const uint4*>(
              reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[r0 + j]) + el) -
              x.rphase[MIXED ? r0 + j : 0]));
      if (ACC && r0 == 0 && body) {
        o[0] = __ldcs(reinterpret_cast<const float4*>(a.out + a.head + gi * kGroup));
        o[1] = __ldcs(reinterpret_cast<const float4*>(a.out + a.head + gi * kGroup) + 1);
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
        if (r0 + j < a.n_ranks) {
          const uint4 c = MIXED ? shift_chunk(w[j], x.rphase[r0 + j] >> 1) : w[j];
          if (r0 + j == 0) widen8<GT>(c, g);
          else add8<GT>(c, g);
        }
      }
    }
    if constexpr (!MIXED) shift_down8(g, x.rphase[0] >> 1);
    if (body) reduce_store8(a, a.head + gi * kGroup, g, o, ACC, bad);
  }
  reduce_shift_edges<GT>(a, nvec, lane, bad);
}

template <int G, int MAXR, int NR, bool MIXED>
ss_status launch_reduce_shift_batch(const ShiftReduceArgs<MAXR>& x, int64_t runs, void* stream) {
  auto go = [&](auto* fn, int u) {
    const int64_t batches = (runs + u - 1) / u;
    return launch(fn, grid_for(reinterpret_cast<const void*>(fn), batches * 32, kReduceChunkThreads), x, stream,
                  kReduceChunkThreads);
  };
  if (x.s.accumulate) return go(reduce_shift_batch_kernel<G, MAXR, NR, true, MIXED>, reduce_batch_runs(NR, true));
  return go(reduce_shift_batch_kernel<G, MAXR, NR, false, MIXED>, reduce_batch_runs(NR, false));
}

template <int G, int MAXR, int NR, bool MIXED>
ss_status launch_reduce_shift_pipe(const ShiftReduceArgs<MAXR>& x, int64_t runs, void* stream) {
  auto* fn = reduce_shift_pipe_kernel<G, MAXR, NR, MIXED>;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), runs * 32, kChunkThreads), x, stream, kChunkThreads);
}

template <int G, int MAXR, bool MIXED>
ss_status launch_reduce_shift(const ShiftReduceArgs<MAXR>& x, void* stream) {
  const ReduceArgs<MAXR>& a = x.s;
  const int64_t runs = ((a.n - a.head) / kGroup - 2 + kRun - 1) / kRun;
  if constexpr (MAXR == kSmallRanks) {
    switch (a.n_ranks) {
      case 1: return launch_reduce_shift_batch<G, MAXR, 1, MIXED>(x, runs, stream);
      case 2:
        if constexpr (SS_RED_BATCH_MAX_RANKS >= 2) return launch_reduce_shift_batch<G, MAXR, 2, MIXED>(x, runs, stream);
        break;
      case 3:
        if constexpr (SS_RED_BATCH_MAX_RANKS >= 3) {
          return launch_reduce_shift_batch<G, MAXR, 3, MIXED>(x, runs, stream);
        } else if constexpr (MIXED) {
          // 3 ranks at mixed phases, not accumulating: the batched form (0.94-0.95 of the copy
          // peak against 0.89 in the any-rank form; one phase and accumulating it measured slower)
          if (!a.accumulate) {
            auto* fn = reduce_shift_batch_kernel<G, MAXR, 3, false, true>;
            const int64_t u = reduce_batch_runs(3, false);
            return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (runs + u - 1) / u * 32, kReduceChunkThreads),
                          x, stream, kReduceChunkThreads);
          }
        }
        break;
      case 4:
        if constexpr (SS_RED_BATCH_MAX_RANKS >= 4) return launch_reduce_shift_batch<G, MAXR, 4, MIXED>(x, runs, stream);
        break;
      case 7: if (!MIXED) return launch_reduce_shift_pipe<G, MAXR, 7, false>(x, runs, stream); break;
      case 8: if (!MIXED) return launch_reduce_shift_pipe<G, MAXR, 8, false>(x, runs, stream); break;
      default: break;
    }
  }
  auto go = [&](auto* fn) {
    return launch(fn, grid_for(reinterpret_cast<const void*>(fn), runs * 32, kReduceChunkThreads), x, stream,
                  kReduceChunkThreads);
  };
  return a.accumulate ? go(reduce_shift_kernel<G, MAXR, true, MIXED>) : go(reduce_shift_kernel<G, MAXR, false, MIXED>);
}

#ifndef SS_RED_ONE_PHASE_SHIFT_EACH_ABOVE
#define SS_RED_ONE_PHASE_SHIFT_EACH_ABOVE 16
#endif
// rphase: each rank's byte phase at the output's group starts (even; not all zero).
template <int MAXR>
ss_status run_reduce_shift(const ReduceArgs<MAXR>& a, const uint8_t* rphase, ss_dtype gt, void* stream) {
  ShiftReduceArgs<MAXR> x;
  std::memset(&x, 0, sizeof x);
  x.s = a;
  bool mixed = false;
  for (int32_t r = 0; r < a.n_ranks; ++r) {
    x.rphase[r] = rphase[r];
    mixed = mixed || rphase[r] != rphase[0];
  }
  // more than 16 ranks at one phase take the per-rank-shift form too (the same fp32 adds in
  // the same order): measured on GB300 at 2^26 elements, 64 ranks one element off 0.91 -> 0.96
  // of the copy peak; 9 ranks 1.00 -> 0.98 and 16 ranks unchanged, so not there
  mixed = mixed || a.n_ranks > SS_RED_ONE_PHASE_SHIFT_EACH_ABOVE;
  if (gt == SS_BF16) return mixed ? launch_reduce_shift<SS_BF16, MAXR, true>(x, stream)
                                  : launch_reduce_shift<SS_BF16, MAXR, false>(x, stream);
  if (gt == SS_FP16) return mixed ? launch_reduce_shift<SS_FP16, MAXR, true>(x, stream)
                                  : launch_reduce_shift<SS_FP16, MAXR, false>(x, stream);
  return SS_ERR_DTYPE;
}

template <int MAXR>
ss_status run_reduce(const ReduceArgs<MAXR>& a, bool vec, ss_dtype gt, void* stream) {
#define SS_RED_CASE(G)                                                                     \
  if (gt == G) {                                                                           \
    ss_status st = SS_OK;                                                                  \
    if (vec && reduce_quad<G>(a, st, stream)) return st;                                   \
    if (vec && reduce_vec_tx<G>(a, st, stream)) return st;                                 \
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
  bool shifted = false;
  std::vector<uint8_t> rphase;
  if (!vec) {
    const int h32 = common_phase({}, p32);
    if (h32 >= 0 && n - h32 >= 3 * kGroup) {
      // every rank's byte phase at the output's group starts (not all zero: else vec)
      shifted = true;
      head = h32;
      rphase.resize(n_ranks);
      for (int32_t r = 0; r < n_ranks; ++r)
        rphase[r] = static_cast<uint8_t>((reinterpret_cast<uintptr_t>(rank_grads[r]) + 2u * h32) & 15u);
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
    return shifted ? run_reduce_shift(a, rphase.data(), gdtype, stream) : run_reduce(a, vec, gdtype, stream);
  }
  ReduceArgs<kLargeRanks> a;
  std::memset(&a, 0, sizeof a);
  fill(a);
  return shifted ? run_reduce_shift(a, rphase.data(), gdtype, stream) : run_reduce(a, vec, gdtype, stream);
}

}  // extern "C"
