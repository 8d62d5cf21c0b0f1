// ss_norm.cu -- the global gradient-norm clip: the per-shard sum of squares of
// the reduced gradient (ss_grad_sumsq, and ss_grad_sumsq_noalloc with its slots
// in a fixed device array) and the clip coefficient from all shards' sums
// (ss_clip_coef).
#include <cuda.h>

#include "ss_common.cuh"

namespace ss {
namespace {

// ------------------------------------------------------------------ gradient sum of squares (global clip norm)
//
// Deterministic per-shard sum of squares of the reduced gradient. The shard is
// cut into tiles of kThreads x kSumsqGroups groups of 8 elements (after the
// 0..7-element head that aligns the vectors); thread j of a tile owns groups
// j, j + kThreads, ..., loads them (for up to 8 ranks pipelined across the
// block's tiles), adds each group's 8 squares in fp32 (a fixed FMA chain) and
// the group sums in group order as an fp32 pair (TwoSum); the block combines
// its threads' pairs through a fixed shuffle tree and the warps in order, and
// writes ONE double per tile into the caller's workspace (GB300's fp64 rate is
// low, so fp64 is kept to one value per tile). The head/tail elements (< 16)
// get a slot of their own. A second one-block kernel adds the slots in a fixed
// order. The partition depends only on n and the arrays' 16-byte phases, never
// on the grid size, so the result is bit-reproducible.
//
// Error: each 8-element fp32 chain of non-negative terms is within 8 * 2^-24
// relative of its exact value; the fp32-pair and double sums add < 2^-40 (the
// pairs lose at most 2^-48 per addition of non-negative terms); so the result
// is within ~5e-7 relative of the exact sum of squares of the fp32 gradients.

template <int MAXR>
struct SumsqArgs {
  RankTable<MAXR> ranks;
  const float* g32;
  float* g_out;
  int32_t* nonfinite;
  double* partials;  // [ntiles + 1]
  int64_t n;
  int64_t head;
  int64_t ntiles;
  int32_t n_ranks;
  float post_scale;
};

constexpr int kSumsqGroups = 8;                          // groups per thread per tile
constexpr int kSumsqTile = kThreads * kGroup * kSumsqGroups;  // elements per tile

// Block-wide sum of per-thread values carried as fp32 pairs (hi + lo, summed
// with TwoSum through a fixed shuffle tree, then over the warps in order by
// thread 0); fp64 only for the block's result, meaningful in thread 0. `red`
// holds two sets of per-warp slots used on alternate calls (`it` = the
// block's call count), so one barrier per call suffices: a warp can only
// write a set again after the next call's barrier, which thread 0 reaches
// after reading it.
__device__ __forceinline__ double block_sum(dd x, float2* red, int it) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float h = __shfl_xor_sync(0xFFFFFFFFu, x.hi, off);
    const float l = __shfl_xor_sync(0xFFFFFFFFu, x.lo, off);
    const dd t = two_sum(x.hi, h);
    x = {t.hi, t.lo + (x.lo + l)};
  }
  float2* set = red + (it & 1) * (kThreads / 32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) set[warp] = make_float2(x.hi, x.lo);
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0) {
    dd acc = {set[0].x, set[0].y};
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) {
      const dd t = two_sum(acc.hi, set[w].x);
      acc = {t.hi, t.lo + (acc.lo + set[w].y)};
    }
    s = static_cast<double>(acc.hi) + static_cast<double>(acc.lo);
  }
  return s;
}

template <int GT, bool FROM_G32, bool VEC, int MAXR>
__device__ __forceinline__ float reduced1(const SumsqArgs<MAXR>& a, int64_t e) {
  if constexpr (FROM_G32) return a.g32[e];
  float g = reduce1<GT>(a.ranks, a.n_ranks, e);
  if (a.post_scale != 1.0f) g = g * a.post_scale;
  return g;
}

// g (this lane's group at element e) stored to g_out when g_out is K floats past
// a 16-byte boundary at the group's start: the lane writes the two aligned
// float4 vectors that start inside its group -- elements 4-K..7-K, and 8-K..7
// followed by the next lane's first 4-K, taken by shuffle -- so the lanes of a
// warp, which hold consecutive groups, cover their elements with aligned
// stores; lane 0 writes its first 4-K elements one by one, and a lane whose
// next lane has no group (lane 31, or the shard's last group) its last K.
// All lanes call it (the shuffles); `valid` says the lane holds a group.
template <int K>
__device__ __forceinline__ void store_g_out_shifted(float* out, const float (&g)[8], bool valid, bool next_valid) {
  static_assert(K >= 1 && K <= 3, "an fp32 array is 1-3 floats off a 16-byte boundary");
  const int lane = threadIdx.x & 31;
  float nx[4 - K];
#pragma unroll
  for (int j = 0; j < 4 - K; ++j) nx[j] = __shfl_down_sync(0xFFFFFFFFu, g[j], 1);
  if (!valid) return;
  __stcs(reinterpret_cast<float4*>(out + 4 - K), make_float4(g[4 - K], g[5 - K], g[6 - K], g[7 - K]));
  if (lane < 31 && next_valid) {
    float w[4];
#pragma unroll
    for (int j = 0; j < K; ++j) w[j] = g[8 - K + j];
#pragma unroll
    for (int j = 0; j < 4 - K; ++j) w[K + j] = nx[j];
    __stcs(reinterpret_cast<float4*>(out + 8 - K), make_float4(w[0], w[1], w[2], w[3]));
  } else {
#pragma unroll
    for (int j = 0; j < K; ++j) out[8 - K + j] = g[8 - K + j];
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < 4 - K; ++j) out[j] = g[j];
  }
}

// The same vectors staged through the warp's 64 float4 slots: lane l's two
// vectors are the warp's consecutive aligned vectors 2l and 2l + 1 (counted from
// lane 0's first), so after the exchange each store instruction covers 512
// contiguous bytes. `wv`: the number of the warp's groups in the shard; a vector
// is stored when the groups it covers are (the others' elements go one by one).
template <int K>
__device__ __forceinline__ void store_g_out_shifted_staged(float* out, const float (&g)[8], bool valid,
                                                           float4* t, int wv) {
  static_assert(K >= 1 && K <= 3, "an fp32 array is 1-3 floats off a 16-byte boundary");
  const int lane = threadIdx.x & 31;
  float nx[4 - K];
#pragma unroll
  for (int j = 0; j < 4 - K; ++j) nx[j] = __shfl_down_sync(0xFFFFFFFFu, g[j], 1);
  float w[4];
#pragma unroll
  for (int j = 0; j < K; ++j) w[j] = g[8 - K + j];
#pragma unroll
  for (int j = 0; j < 4 - K; ++j) w[K + j] = nx[j];
  t[2 * lane] = make_float4(g[4 - K], g[5 - K], g[6 - K], g[7 - K]);
  t[2 * lane + 1] = make_float4(w[0], w[1], w[2], w[3]);
  __syncwarp();
  float4* base = reinterpret_cast<float4*>(out - kGroup * lane + 4 - K);  // lane 0's first vector
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int f = lane + 32 * k;
    const int l = f >> 1;
    if ((f & 1) ? l + 1 < wv : l < wv) __stcs(base + f, t[f]);
  }
  __syncwarp();
  if (valid && !(lane + 1 < wv)) {
#pragma unroll
    for (int j = 0; j < K; ++j) out[8 - K + j] = g[8 - K + j];
  }
  if (valid && lane == 0) {
#pragma unroll
    for (int j = 0; j < 4 - K; ++j) out[j] = g[j];
  }
}

// How g_out is written: as 16-byte vectors at the inputs' phase, realigned
// between lanes by store_g_out_shifted (g_out 1-3 floats off that phase),
// element by element, or staged: the warp's 32 consecutive groups pass through
// 1 KB of shared memory and are stored as consecutive 16-byte vectors, each
// instruction covering 512 bytes (where each lane storing its own group leaves
// every instruction half of each 32-byte sector it touches).
enum GoutStore : int { kGoutVec = 0, kGoutShuffle = 1, kGoutElem = 2, kGoutStaged = 3, kGoutShuffleStaged = 4 };

// One reduced group of 8 values at element e: optionally stored to g_out, its
// squares added in fp32 (a fixed FMA chain), and the sum added to the thread's
// fp32 pair. The finiteness test runs per element only when the group's sum is
// not finite (a non-finite value, or squares past the fp32 range). With
// kGoutShuffle and kGoutStaged all lanes of the warp call it, `valid` telling
// which hold a group (kGoutStaged: `stage` is the warp's 64 float4 slots and
// `warp_valid` the number of the warp's groups in the shard); otherwise only
// lanes holding a group call it.
template <bool VEC, int GOUT, int MAXR>
__device__ __forceinline__ void sumsq_group(const SumsqArgs<MAXR>& a, int64_t e, const float (&g)[8], dd& s,
                                            bool& bad, bool valid = true, bool next_valid = true,
                                            float4* stage = nullptr, int warp_valid = 0) {
  if (a.g_out) {
    if constexpr (GOUT == kGoutStaged) {
      const int lane = threadIdx.x & 31;
      stage[2 * lane] = make_float4(g[0], g[1], g[2], g[3]);
      stage[2 * lane + 1] = make_float4(g[4], g[5], g[6], g[7]);
      __syncwarp();
      float* ew = a.g_out + e - kGroup * lane;  // the warp's first group (consecutive groups)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = lane + 32 * k;
        if (f / 2 < warp_valid) __stcs(reinterpret_cast<float4*>(ew) + f, stage[f]);
      }
      __syncwarp();
    } else if constexpr (GOUT == kGoutShuffleStaged) {
      switch ((reinterpret_cast<uintptr_t>(a.g_out + e) & 15u) >> 2) {  // the same for every group
        case 1: store_g_out_shifted_staged<1>(a.g_out + e, g, valid, stage, warp_valid); break;
        case 2: store_g_out_shifted_staged<2>(a.g_out + e, g, valid, stage, warp_valid); break;
        default: store_g_out_shifted_staged<3>(a.g_out + e, g, valid, stage, warp_valid); break;
      }
    } else if constexpr (GOUT == kGoutShuffle) {
      switch ((reinterpret_cast<uintptr_t>(a.g_out + e) & 15u) >> 2) {  // the same for every group
        case 1: store_g_out_shifted<1>(a.g_out + e, g, valid, next_valid); break;
        case 2: store_g_out_shifted<2>(a.g_out + e, g, valid, next_valid); break;
        default: store_g_out_shifted<3>(a.g_out + e, g, valid, next_valid); break;
      }
    } else if constexpr (VEC && GOUT == kGoutVec) {
      st8f(a.g_out + e, g);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) a.g_out[e + j] = g[j];
    }
  }
  if constexpr (GOUT == kGoutShuffle || GOUT == kGoutStaged || GOUT == kGoutShuffleStaged) {
    if (!valid) return;
  }
  float c = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) c = fmaf(g[j], g[j], c);
  if (!finite(c)) {
#pragma unroll
    for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
  }
  const dd t = two_sum(s.hi, c);
  s = {t.hi, s.lo + t.lo};
}

// Minimum resident blocks per SM asked of the compiler: none (0), which leaves
// the register count to ptxas, except for the unstaged realigned-g_out instances
// (rank counts outside SS_SUMSQ_SHUFFLE_STAGED) of the rank counts in
// SS_SUMSQ_SHUFFLE_TWO_BLOCKS (bit N: N ranks), which ask for 2.
// An explicit 1 is not the same as none: with __launch_bounds__(256, 1) ptxas
// gave the general tiles 147 registers (one block per SM; measured on GB300 at
// 2^26 elements, 64 ranks, 0.76 of the copy peak) where plain
// __launch_bounds__(256) gives 124 (two blocks; 1.00). Two blocks measured, for
// g_out one element off the inputs' phase: 1 rank 0.70 -> 0.75, 3 ranks 0.81 ->
// 0.88, 4 ranks 0.90 -> 0.85, 2 and 5-8 ranks within 1%.
#ifndef SS_SUMSQ_SHUFFLE_TWO_BLOCKS
#define SS_SUMSQ_SHUFFLE_TWO_BLOCKS ((1u << 1) | (1u << 3))
#endif
// The general tiles (any rank count) write an off-phase g_out element by element
// (measured against realigned stores there: 9 / 16 / 64 ranks 0.53 / 0.73 / 0.85
// of the copy peak against 0.50 / 0.68 / 0.73).
constexpr int sumsq_min_blocks(int nr, int gout) {
  return gout == kGoutShuffle && nr > 0 && ((SS_SUMSQ_SHUFFLE_TWO_BLOCKS >> nr) & 1u) ? 2 : 0;
}

// Tiles of the compile-time rank count NR (1..8), 16-byte vectors: a block's
// tiles form one stream of load batches (kB groups x NR ranks per batch),
// double-buffered in registers -- the loads of batch i+1 are in flight while
// batch i is converted and squared, and the first batch of the block's next
// tile is in flight across the tile's block reduction. Batches past the end
// (of the shard or of the block's tiles) read group 0 instead, always in
// range, and are dropped, so no branch stands between the loads.
template <int GT, int MAXR, int NR, int GOUT>
__device__ __forceinline__ void sumsq_ranked_tiles(const SumsqArgs<MAXR>& a, float2* red, bool& bad,
                                                   float4* stage) {
  constexpr int kB = NR == 2 ? 4 : (NR <= 4 ? 2 : 1);  // groups per batch (measured best on GB300)
  static_assert(kSumsqGroups % (2 * kB) == 0, "two batches per pipeline round");
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t stride = static_cast<int64_t>(gridDim.x);
  auto load = [&](uint4 (&w)[kB][NR], int64_t tile, int q0) {
    const int64_t g0 = tile * kSumsqGroups * kThreads + threadIdx.x;
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int64_t gq = g0 + (q0 + b) * kThreads;
      const int64_t e = a.head + (gq < nvec ? gq : 0) * kGroup;
#pragma unroll
      for (int r = 0; r < NR; ++r)
        w[b][r] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.ranks.p[r]) + e));
    }
  };
  auto consume = [&](const uint4 (&w)[kB][NR], int64_t tile, int q0, dd& s) {
    const int64_t g0 = tile * kSumsqGroups * kThreads + threadIdx.x;
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      float g[8];
      widen8<GT>(w[b][0], g);
#pragma unroll
      for (int r = 1; r < NR; ++r) add8<GT>(w[b][r], g);
      if (a.post_scale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
      }
      const int64_t gq = g0 + (q0 + b) * kThreads;
      if constexpr (GOUT == kGoutShuffle) {
        sumsq_group<true, GOUT>(a, a.head + gq * kGroup, g, s, bad, gq < nvec, gq + 1 < nvec);
      } else if constexpr (GOUT == kGoutStaged || GOUT == kGoutShuffleStaged) {
        const int64_t left = nvec - (gq - (threadIdx.x & 31));  // groups of the warp's 32 in the shard
        sumsq_group<true, GOUT>(a, a.head + gq * kGroup, g, s, bad, gq < nvec, true, stage,
                                static_cast<int>(left < 0 ? 0 : (left > 32 ? 32 : left)));
      } else if (gq < nvec) {
        sumsq_group<true, GOUT>(a, a.head + gq * kGroup, g, s, bad);
      }
    }
  };
  int64_t tile = blockIdx.x;
  if (tile >= a.ntiles) return;
  uint4 wa[kB][NR], wb[kB][NR];
  load(wa, tile, 0);
  for (int it = 0;; ++it) {
    const int64_t next = tile + stride < a.ntiles ? tile + stride : tile;
    dd s = {0.0f, 0.0f};
#pragma unroll
    for (int q0 = 0; q0 < kSumsqGroups; q0 += 2 * kB) {
      load(wb, tile, q0 + kB);
      consume(wa, tile, q0, s);
      if (q0 + 2 * kB < kSumsqGroups) load(wa, tile, q0 + 2 * kB);
      else load(wa, next, 0);
      consume(wb, tile, q0 + kB, s);
    }
    const double t = block_sum(s, red, it);
    if (threadIdx.x == 0) a.partials[tile] = t;
    if (next == tile) break;
    tile = next;
  }
}

// NR > 0 (16-bit ranks, 16-byte vectors): the rank count as a compile-time
// constant (N <= 8), pipelined as above; NR == 0: any rank count, an fp32
// gradient, or element-wise access -- each thread issues its tile's loads
// group by group, then squares and sums them.
template <int GT, bool FROM_G32, bool VEC, int MAXR, int NR, int GOUT = kGoutVec>
__global__ void __launch_bounds__(kThreads, sumsq_min_blocks(NR, GOUT))
    sumsq_tiles_kernel(const __grid_constant__ SumsqArgs<MAXR> a) {
  __shared__ float2 red[2 * (kThreads / 32)];
  __shared__ float4 stage[GOUT == kGoutStaged || GOUT == kGoutShuffleStaged ? (kThreads / 32) * 64 : 1];
  pdl_wait();
  pdl_trigger();  // the slot sum may be scheduled now; it waits for this grid to finish
  const int64_t nvec = (a.n - a.head) / kGroup;
  bool bad = false;
  if constexpr (VEC && !FROM_G32 && NR > 0) {
    sumsq_ranked_tiles<GT, MAXR, NR, GOUT>(
        a, red, bad, stage + (GOUT == kGoutStaged || GOUT == kGoutShuffleStaged ? (threadIdx.x >> 5) * 64 : 0));
  } else {
    int it = 0;
    for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++it) {
      // Loads of all groups first, unconditionally: a group past the end reads
      // group 0 of the shard instead (always in range: ntiles > 0 implies
      // nvec > 0) and is dropped below, so no branch stands between the loads.
      float g[kSumsqGroups][8];
      const int64_t g0 = tile * kSumsqGroups * kThreads + threadIdx.x;
#pragma unroll
      for (int q = 0; q < kSumsqGroups; ++q) {
        const int64_t gq = g0 + q * kThreads;
        const int64_t e = a.head + (gq < nvec ? gq : 0) * kGroup;
        if constexpr (VEC) {
          if constexpr (FROM_G32) {
            ld8f(a.g32 + e, g[q]);
          } else {
            reduce8<GT>(a.ranks, a.n_ranks, e, g[q]);
            if (a.post_scale != 1.0f) {
#pragma unroll
              for (int j = 0; j < 8; ++j) g[q][j] = g[q][j] * a.post_scale;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) g[q][j] = reduced1<GT, FROM_G32, VEC>(a, e + j);
        }
      }
      dd s = {0.0f, 0.0f};  // the thread's group sums, accumulated exactly enough as an fp32 pair
#pragma unroll
      for (int q = 0; q < kSumsqGroups; ++q) {
        const int64_t gi = g0 + q * kThreads;
        if constexpr (GOUT == kGoutShuffle)
          sumsq_group<VEC, GOUT>(a, a.head + gi * kGroup, g[q], s, bad, gi < nvec, gi + 1 < nvec);
        else if (gi < nvec) sumsq_group<VEC, GOUT>(a, a.head + gi * kGroup, g[q], s, bad);
      }
      const double t = block_sum(s, red, it);
      if (threadIdx.x == 0) a.partials[tile] = t;
    }
  }
  // Head and tail (< 16 elements) in slot ntiles: lane i of the last block's
  // first warp takes the i-th of them (head first), lane 0 adds the squares
  // in that order. The last block has the fewest tiles.
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x < 32) {
    const int64_t tail0 = a.head + nvec * kGroup;
    const int cnt = static_cast<int>(a.head + (a.n - tail0));
    const int i = static_cast<int>(threadIdx.x);
    double x = 0.0;
    if (i < cnt) {
      const int64_t e = i < a.head ? i : tail0 + (i - a.head);
      const float g = reduced1<GT, FROM_G32, VEC>(a, e);
      if (a.g_out) a.g_out[e] = g;
      bad |= !finite(g);
      x = static_cast<double>(fmaf(g, g, 0.0f));
    }
    double s = 0.0;
    for (int j = 0; j < cnt; ++j) s += __shfl_sync(0xFFFFFFFFu, x, j);
    if (i == 0) a.partials[a.ntiles] = s;
  }
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

// out = sum of partials[0..count) in a fixed order, by one block: thread t
// adds slots t, t + kSlotThreads, ... in that order (eight loads in flight),
// then a fixed shuffle tree and the warps in order. Launched as a programmatic
// dependent of the tiles kernel, so its launch overlaps that kernel's end.
constexpr int kSlotThreads = 256;

__global__ void __launch_bounds__(kSlotThreads) sum_slots_kernel(const double* partials, int64_t count, double* out) {
  __shared__ double red[kSlotThreads / 32];
  pdl_wait();
  pdl_trigger();
  constexpr int kU = 8;
  double s = 0.0;
  for (int64_t base = threadIdx.x; base < count; base += kU * kSlotThreads) {
    double v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + u * kSlotThreads;
      v[u] = partials[i < count ? i : 0];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (base + u * kSlotThreads < count) s += v[u];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kSlotThreads / 32; ++w) t += red[w];
    *out = t;
  }
}

// Global clip coefficient from the shards' sums of squares, added in rank order.
__global__ void clip_coef_kernel(const double* shard_sumsq, int32_t n_shards, float max_norm, float* coef,
                                 double* norm_out) {
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double total = 0.0;
  for (int32_t k = 0; k < n_shards; ++k) total += shard_sumsq[k];
  const double norm = sqrt(total);
  const double c = static_cast<double>(max_norm) / (norm + 1e-6);
  *coef = static_cast<float>(c < 1.0 ? c : 1.0);
  if (norm_out) *norm_out = norm;
}

// SH: g_out 1-3 floats off the inputs' phase (vector forms only): the per-rank-count
// tiles realign it between lanes (measured on GB300 at 2^26 elements with the gradients
// one element off: 2 ranks 0.82 of the copy peak against 0.29 element by element, 8 ranks
// 0.91 against 0.72), the general tiles write it element by element (64 ranks: 0.87,
// against 0.72 realigned).
// The per-rank-count tiles writing g_out at the inputs' phase stage it (bit N: N
// ranks). Measured on GB300 at 2^26 elements against per-lane 16-byte stores, one
// box: 1 / 2 / 3 ranks 0.75 / 0.83 / 0.84 -> 0.84 / 0.86 / 0.90 of the copy peak,
// 4-8 ranks 0.90-0.97 -> 0.94-0.98; the results are the same bits. Without g_out
// the unstaged instances run (the staged ones hold more registers).
#ifndef SS_SUMSQ_STAGED
#define SS_SUMSQ_STAGED 0x1FEu
#endif
// Likewise with g_out 1-3 floats off the inputs' phase: the realigned vectors
// pass through the same slots (store_g_out_shifted_staged). Measured on GB300 at
// 2^26 elements, gradients one element off g_out's phase, against per-lane
// realigned stores: 1 / 2 / 3 ranks 0.77 / 0.82 / 0.88 -> 0.87 / 0.87 / 0.90 of
// the copy peak, 4-5 ranks 0.88-0.90 -> 0.91, 6-8 ranks the same (0.91-0.92).
#ifndef SS_SUMSQ_SHUFFLE_STAGED
#define SS_SUMSQ_SHUFFLE_STAGED 0x1FEu
#endif
template <int MAXR, bool SH>
ss_status run_sumsq_t(const SumsqArgs<MAXR>& a, bool vec, bool from_g32, ss_dtype gt, double* out, void* stream) {
  // One wave: no more blocks than fit on the GPU at once (the kernel's own
  // occupancy), so every block takes the same number of tiles within one and
  // none waits for a free slot while the others finish.
  ss_status launched = SS_ERR_DTYPE;
  auto go = [&](auto* fn) {
    const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(fn));
    const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(a.ntiles, cap)));
    launched = launch(fn, grid, a, stream);
  };
  const int nr = (vec && !from_g32 && a.n_ranks <= 8) ? a.n_ranks : 0;
  constexpr int kRanked = SH ? kGoutShuffle : kGoutVec;
  constexpr int kGeneral = SH ? kGoutElem : kGoutVec;
  // g_out given, for the rank counts in SS_SUMSQ_STAGED (g_out at the inputs' phase) or
  // SS_SUMSQ_SHUFFLE_STAGED (off it): staged stores
  constexpr unsigned kStagedMask = SH ? SS_SUMSQ_SHUFFLE_STAGED : SS_SUMSQ_STAGED;
  constexpr int kStaged = SH ? kGoutShuffleStaged : kGoutStaged;
  const bool staged = a.g_out != nullptr && ((kStagedMask >> nr) & 1u);  // SH: g_out is given
#define SS_SUMSQ_NR(G, R)                                                                 \
  case R:                                                                                 \
    if constexpr (SH && ((kStagedMask >> R) & 1u)) {                                      \
      go(sumsq_tiles_kernel<G, false, true, MAXR, R, kStaged>);                           \
    } else {                                                                              \
      if constexpr ((kStagedMask >> R) & 1u) {                                            \
        if (staged) {                                                                     \
          go(sumsq_tiles_kernel<G, false, true, MAXR, R, kStaged>);                       \
          break;                                                                          \
        }                                                                                 \
      }                                                                                   \
      go(sumsq_tiles_kernel<G, false, true, MAXR, R, kRanked>);                           \
    }                                                                                     \
    break;
// The per-rank-count forms exist for the small rank table only (at most 8 ranks),
// and an fp32 gradient always travels with the small table.
#define SS_SUMSQ_RANKED(G)                                                                              \
  if constexpr (MAXR == kSmallRanks) {                                                                  \
    switch (nr) {                                                                                       \
      SS_SUMSQ_NR(G, 1) SS_SUMSQ_NR(G, 2) SS_SUMSQ_NR(G, 3) SS_SUMSQ_NR(G, 4)                           \
      SS_SUMSQ_NR(G, 5) SS_SUMSQ_NR(G, 6) SS_SUMSQ_NR(G, 7) SS_SUMSQ_NR(G, 8)                           \
      default: go(sumsq_tiles_kernel<G, false, true, MAXR, 0, kGeneral>);                               \
    }                                                                                                   \
  } else {                                                                                              \
    go(sumsq_tiles_kernel<G, false, true, MAXR, 0, kGeneral>);                                          \
  }
  if (from_g32) {
    if constexpr (MAXR != kSmallRanks) return SS_ERR_INVALID_ARG;
    else if (vec) go(sumsq_tiles_kernel<SS_BF16, true, true, MAXR, 0, kGeneral>);
    else go(sumsq_tiles_kernel<SS_BF16, true, false, MAXR, 0>);
  } else if (vec && gt == SS_BF16) {
    SS_SUMSQ_RANKED(SS_BF16)
  } else if (vec && gt == SS_FP16) {
    SS_SUMSQ_RANKED(SS_FP16)
  } else if (gt == SS_BF16) {
    go(sumsq_tiles_kernel<SS_BF16, false, false, MAXR, 0>);
  } else if (gt == SS_FP16) {
    go(sumsq_tiles_kernel<SS_FP16, false, false, MAXR, 0>);
  } else {
    return SS_ERR_DTYPE;
  }
#undef SS_SUMSQ_RANKED
#undef SS_SUMSQ_NR
  if (launched != SS_OK) return launched;
  return launch_dependent(sum_slots_kernel, dim3(1), dim3(kSlotThreads), 0, stream, a.partials, a.ntiles + 1, out);
}

template <int MAXR>
ss_status run_sumsq(const SumsqArgs<MAXR>& a, bool vec, bool shift_gout, bool from_g32, ss_dtype gt, double* out,
                    void* stream) {
  return shift_gout ? run_sumsq_t<MAXR, true>(a, vec, from_g32, gt, out, stream)
                    : run_sumsq_t<MAXR, false>(a, vec, from_g32, gt, out, stream);
}

// Shared by ss_grad_sumsq and any entry point that supplies its own slots.
ss_status grad_sumsq_impl(int64_t n, const float* g32, const void* const* rank_grads, int32_t n_ranks,
                          ss_dtype gdtype, float post_scale, double* sumsq_out, double* slots, int64_t slots_bytes,
                          float* g_out, int32_t* nonfinite_flag, void* stream) {
  if (n < 0 || !sumsq_out || !slots) return SS_ERR_INVALID_ARG;
  if (n > INT64_MAX / 16) return SS_ERR_OVERFLOW;
  if (slots_bytes < ss_grad_sumsq_workspace(n)) return SS_ERR_INVALID_ARG;
  std::vector<Range> ranges;
  std::vector<uintptr_t> p16, p32;
  const bool from_g32 = g32 != nullptr;
  if (from_g32) {
    if (reinterpret_cast<uintptr_t>(g32) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(g32, 4 * n, false));
    p32.push_back(reinterpret_cast<uintptr_t>(g32));
  } else {
    ss_status st = check_ranks(rank_grads, n_ranks, gdtype, n, ranges, p16);
    if (st != SS_OK) return st;
  }
  if ((reinterpret_cast<uintptr_t>(sumsq_out) & 7u) || (reinterpret_cast<uintptr_t>(slots) & 7u)) return SS_ERR_ALIGN;
  ranges.push_back(rng(sumsq_out, 8, true));
  ranges.push_back(rng(slots, ss_grad_sumsq_workspace(n), true));
  if (g_out) {
    if (reinterpret_cast<uintptr_t>(g_out) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(g_out, 4 * n, true));
    p32.push_back(reinterpret_cast<uintptr_t>(g_out));
  }
  if (nonfinite_flag) {
    if (reinterpret_cast<uintptr_t>(nonfinite_flag) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(nonfinite_flag, 4, true));
  }
  if (any_output_overlap(ranges)) return SS_ERR_OVERLAP;
  int h = common_phase(p16, p32);
  bool vec = h >= 0 && h < n;
  bool shift_gout = false;
  if (!vec && g_out) {
    // the inputs at one phase and g_out at another: the groups follow the inputs (16-byte
    // loads) and g_out's values are realigned between lanes (it was the last array listed)
    const std::vector<uintptr_t> in32(p32.begin(), p32.end() - 1);
    const int hin = common_phase(p16, in32);
    if (hin >= 0 && hin < n) {
      h = hin;
      vec = true;
      shift_gout = true;
    }
  }
  const int64_t head = vec ? h : 0;
  const int64_t nvec = (n - head) / kGroup;
  const int64_t ntiles = (nvec + kThreads * kSumsqGroups - 1) / (kThreads * kSumsqGroups);
  auto fill = [&](auto& a) {
    if (!from_g32)
      for (int32_t r = 0; r < n_ranks; ++r) a.ranks.p[r] = rank_grads[r];
    a.g32 = g32;
    a.g_out = g_out;
    a.nonfinite = nonfinite_flag;
    a.partials = slots;
    a.n = n;
    a.head = head;
    a.ntiles = ntiles;
    a.n_ranks = from_g32 ? 0 : n_ranks;
    a.post_scale = post_scale;
  };
  const ss_dtype gt = from_g32 ? SS_BF16 : gdtype;
  if (from_g32 || n_ranks <= kSmallRanks) {
    SumsqArgs<kSmallRanks> a;
    std::memset(&a, 0, sizeof a);
    fill(a);
    return run_sumsq(a, vec, shift_gout, from_g32, gt, sumsq_out, stream);
  }
  SumsqArgs<kLargeRanks> a;
  std::memset(&a, 0, sizeof a);
  fill(a);
  return run_sumsq(a, vec, shift_gout, from_g32, gt, sumsq_out, stream);
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" {

int64_t ss_grad_sumsq_workspace(int64_t n) {
  if (n < 0) return -1;
  return static_cast<int64_t>(sizeof(double)) * ((n + kSumsqTile - 1) / kSumsqTile + 2);
}

ss_status ss_grad_sumsq(int64_t n, const float* g32, const void* const* rank_grads, int32_t n_ranks,
                        ss_dtype gdtype, float post_scale, double* sumsq_out, void* workspace,
                        int64_t workspace_bytes, float* g_out, int32_t* nonfinite_flag, void* stream) {
  return grad_sumsq_impl(n, g32, rank_grads, n_ranks, gdtype, post_scale, sumsq_out,
                         static_cast<double*>(workspace), workspace_bytes, g_out, nonfinite_flag, stream);
}

}  // extern "C"

// ---------------------------------------------------------------- sum of squares without allocation
//
// ss_grad_sumsq_noalloc keeps its tile slots in this fixed array instead of a
// caller workspace, for callers that cannot allocate device memory. Every GPU
// that loads the library holds the array (SS_NOALLOC_SUMSQ_SLOTS doubles =
// 512 KiB) until the process exits. All calls share it: each call overwrites
// every slot it reads before reading it, so nothing needs clearing, but two
// calls whose kernels overlap on the GPU race on the slots.
static __device__ __align__(256) double g_noalloc_sumsq_slots[SS_NOALLOC_SUMSQ_SLOTS];

namespace {

// The driver's context queries, reached through the runtime (the library does
// not link the driver library itself): the identity of the current context
// decides whether a cached address of the slot array is still valid.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// A unique id of the calling thread's current context (ids are never reused
// within a process), or 0 when there is none or the driver cannot say.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the slot array in the current context. The name of the
// array is only a host-side stand-in; the address comes from the runtime, with
// the device current, the first time a context calls (the array lives in the
// context's copy of the library's device code, so a device reset, which makes
// a new context, gets a new lookup). Without a context id the lookup runs on
// every call.
ss_status noalloc_slots(double** out) {
  constexpr int kCached = 64;
  static std::mutex mu;
  static unsigned long long ids[kCached] = {};
  static double* addrs[kCached] = {};
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = current_context_id();
  if (id != 0) {
    for (int i = 0; i < kCached; ++i) {
      if (ids[i] == id) {
        *out = addrs[i];
        return SS_OK;
      }
    }
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_sumsq_slots);
  if (e != cudaSuccess) return cuda_fail(e);
  // the lookup above makes the device's context current if nothing was, so ask again
  const unsigned long long now = id != 0 ? id : current_context_id();
  if (now != 0) {
    ids[next] = now;
    addrs[next] = static_cast<double*>(p);
    next = (next + 1) % kCached;
  }
  *out = static_cast<double*>(p);
  return SS_OK;
}

}  // namespace

extern "C" {

ss_status ss_grad_sumsq_noalloc(int64_t n, const float* g32, const void* const* rank_grads, int32_t n_ranks,
                                ss_dtype gdtype, float post_scale, double* sumsq_out, float* g_out,
                                int32_t* nonfinite_flag, void* stream) {
  if (n < 0) return SS_ERR_INVALID_ARG;
  if (n > SS_NOALLOC_SUMSQ_MAX_N) return SS_ERR_OVERFLOW;
  double* slots = nullptr;
  const ss_status st = noalloc_slots(&slots);
  if (st != SS_OK) return st;
  return grad_sumsq_impl(n, g32, rank_grads, n_ranks, gdtype, post_scale, sumsq_out, slots,
                         static_cast<int64_t>(sizeof(double)) * SS_NOALLOC_SUMSQ_SLOTS, g_out, nonfinite_flag,
                         stream);
}

ss_status ss_clip_coef(const double* shard_sumsq, int32_t n_shards, float max_norm, float* coef_out,
                       double* norm_out, void* stream) {
  if (!shard_sumsq || !coef_out || n_shards < 1 || !(max_norm > 0.0f) || !std::isfinite(max_norm))
    return SS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(shard_sumsq) & 7u) || (reinterpret_cast<uintptr_t>(coef_out) & 3u) ||
      (norm_out && (reinterpret_cast<uintptr_t>(norm_out) & 7u)))
    return SS_ERR_ALIGN;
  std::vector<Range> ranges = {rng(shard_sumsq, 8 * static_cast<int64_t>(n_shards), false), rng(coef_out, 4, true)};
  if (norm_out) ranges.push_back(rng(norm_out, 8, true));
  if (any_output_overlap(ranges)) return SS_ERR_OVERLAP;
  return launch_dependent(clip_coef_kernel, dim3(1), dim3(32), 0, stream, shard_sumsq, n_shards, max_norm, coef_out,
                          norm_out);
}

}  // extern "C"
