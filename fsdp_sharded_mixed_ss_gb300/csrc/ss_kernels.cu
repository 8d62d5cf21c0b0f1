// ss_kernels.cu -- device side of the shard-step ABI: the virtual-rank gradient
// reduce, the fused reduce + AdamW + 16-bit cast step, and the unshard /
// reshard gather copies, with their host-side argument checks and launches.
//
// Method ("FSDP: Fully Sharded Data Parallel Training at Scale"): the unit's
// flat parameter vector is cut into N contiguous shards; in backward the
// reduce-scatter gives rank k the fp32 sum over ranks of its shard's
// gradients; the optimizer step then updates the shard's fp32 master, m and v
// locally; the all-gather concatenates the 16-bit shards into the full unit.
//
// Every kernel here is a streaming, HBM-bound pass: no contraction, so no
// tensor cores. Design for GB300 (sm_103a):
//   * one thread owns a group of 8 consecutive elements: one 16-byte load per
//     rank gradient (8 x 16-bit), two 16-byte loads per fp32 state array;
//     every access is a full 16-byte vector, so each warp moves 512 bytes of
//     each array per instruction, fully coalesced;
//   * persistent grid (SM count x resident blocks), grid-stride loop;
//   * rank gradients are summed in rank order in batches of 8 loads issued
//     before the adds (8 x 16 B in flight per thread for any N);
//   * streaming cache hints (evict-first) on read-once and write-once data;
//   * rank pointer tables travel in the kernel's parameter space
//     (__grid_constant__), so indexing them costs a constant-bank load;
//   * odd-length shards and arbitrary views: the first 0..7 elements up to
//     the common 16-byte phase and the last 0..7 elements are done one by one
//     by the first threads of the grid; if the arrays do not share a phase the
//     whole call takes the element-wise kernel (same results).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/ss.h"
#include "ss_math.cuh"

namespace ss {
namespace {

constexpr int kThreads = 256;
// Block shape of the fused step kernel (the register-heavy one): threads per
// block and the minimum resident blocks per SM asked of the compiler.
#ifndef SS_STEP_THREADS
#define SS_STEP_THREADS 256
#endif
#ifndef SS_STEP_MIN_BLOCKS
#define SS_STEP_MIN_BLOCKS 1
#endif
constexpr int kStepThreads = SS_STEP_THREADS;
constexpr int kGroup = 8;         // elements per thread per iteration
constexpr int kSmallRanks = 64;   // pointer table size of the common kernels
constexpr int kLargeRanks = SS_MAX_RANKS;

thread_local char g_cuda_err[256] = "";

ss_status cuda_fail(cudaError_t e) {
  std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return SS_ERR_CUDA;
}

// ------------------------------------------------------------------ device helpers

template <int DT>
__device__ __forceinline__ float widen1(uint16_t h) {
  if constexpr (DT == SS_BF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  else return __half2float(__ushort_as_half(h));
}

template <int DT>
__device__ __forceinline__ uint16_t narrow1(float x) {
  if constexpr (DT == SS_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

// Two packed 16-bit values (element 0 in the low half) -> two floats.
template <int DT>
__device__ __forceinline__ float2 widen2(uint32_t w) {
  if constexpr (DT == SS_BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  else {
    __half2 h;
    std::memcpy(&h, &w, 4);
    return __half22float2(h);
  }
}

template <int DT>
__device__ __forceinline__ uint32_t narrow2(float a, float b) {
  uint32_t w;
  if constexpr (DT == SS_BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    std::memcpy(&w, &h, 4);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    std::memcpy(&w, &h, 4);
  }
  return w;
}

template <int DT>
__device__ __forceinline__ void widen8(const uint4& w, float (&f)[8]) {
  float2 a = widen2<DT>(w.x), b = widen2<DT>(w.y), c = widen2<DT>(w.z), d = widen2<DT>(w.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <int DT>
__device__ __forceinline__ void add8(const uint4& w, float (&f)[8]) {
  float t[8];
  widen8<DT>(w, t);
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = f[j] + t[j];
}

template <int DT>
__device__ __forceinline__ uint4 narrow8(const float (&f)[8]) {
  return make_uint4(narrow2<DT>(f[0], f[1]), narrow2<DT>(f[2], f[3]), narrow2<DT>(f[4], f[5]),
                    narrow2<DT>(f[6], f[7]));
}

__device__ __forceinline__ void ld8f(const float* p, float (&f)[8]) {
  float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void st8f(float* p, const float (&f)[8]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(f[0], f[1], f[2], f[3]));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(f[4], f[5], f[6], f[7]));
}

__device__ __forceinline__ bool finite(float x) { return fabsf(x) <= 3.402823466e38f; }

// ------------------------------------------------------------------ argument blocks

template <int MAXR>
struct RankTable {
  const void* p[MAXR];
};

template <int MAXR>
struct StepArgs {
  RankTable<MAXR> ranks;
  const float* g32;
  float* master;
  float* m;
  float* v;
  void* p16;
  float* g_out;
  int32_t* nonfinite;
  const float* dev_scale;
  const int32_t* dev_skip;
  int64_t n;
  int64_t head;  // elements before the first 16-byte-aligned group (vector kernel only)
  int32_t n_ranks;
  float post_scale;
  AdamConst k;
};

template <int MAXR>
struct ReduceArgs {
  RankTable<MAXR> ranks;
  float* out;
  int32_t* nonfinite;
  int64_t n;
  int64_t head;
  int32_t n_ranks;
  float post_scale;
  int32_t accumulate;
};

// Sum of the ranks' 8 elements starting at e, in rank order, fp32.
template <int GT, int MAXR>
__device__ __forceinline__ void reduce8(const RankTable<MAXR>& t, int n_ranks, int64_t e, float (&g)[8]) {
  for (int r0 = 0; r0 < n_ranks; r0 += 8) {
    uint4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (r0 + j < n_ranks) w[j] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(t.p[r0 + j]) + e));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (r0 + j < n_ranks) {
        if (r0 + j == 0) widen8<GT>(w[j], g);
        else add8<GT>(w[j], g);
      }
    }
  }
}

template <int GT, int MAXR>
__device__ __forceinline__ float reduce1(const RankTable<MAXR>& t, int n_ranks, int64_t e) {
  float acc = widen1<GT>(static_cast<const uint16_t*>(t.p[0])[e]);
  for (int r = 1; r < n_ranks; ++r) acc = acc + widen1<GT>(static_cast<const uint16_t*>(t.p[r])[e]);
  return acc;
}

// ------------------------------------------------------------------ fused AdamW step

template <int GT, int PT, bool FROM_G32, bool WRITE_P16, int MAXR>
__device__ __forceinline__ void step1(const StepArgs<MAXR>& a, int64_t e, float gs, bool& bad) {
  float g;
  if constexpr (FROM_G32) {
    g = a.g32[e];
  } else {
    g = reduce1<GT>(a.ranks, a.n_ranks, e);
    if (a.post_scale != 1.0f) g = g * a.post_scale;
  }
  bad |= !finite(g);
  if (a.g_out) a.g_out[e] = g;
  if (a.dev_scale) g = g * gs;
  float p = a.master[e], m = a.m[e], v = a.v[e];
  adamw_elem(a.k, g, p, m, v);
  a.master[e] = p;
  a.m[e] = m;
  a.v[e] = v;
  if constexpr (WRITE_P16) static_cast<uint16_t*>(a.p16)[e] = narrow1<PT>(p);
}

template <int GT, int PT, bool FROM_G32, bool WRITE_P16, int MAXR>
__global__ void __launch_bounds__(kStepThreads, SS_STEP_MIN_BLOCKS) adam_vec_kernel(const __grid_constant__ StepArgs<MAXR> a) {
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t gi = tid; gi < nvec; gi += stride) {
    const int64_t e = a.head + gi * kGroup;
    float g[8];
    if constexpr (FROM_G32) {
      ld8f(a.g32 + e, g);
    } else {
      reduce8<GT>(a.ranks, a.n_ranks, e, g);
      if (a.post_scale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
      }
    }
    if (a.nonfinite) {
#pragma unroll
      for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
    }
    if (a.g_out) st8f(a.g_out + e, g);
    if (a.dev_scale) {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = g[j] * gs;
    }
    float p[8], m[8], v[8];
    ld8f(a.master + e, p);
    ld8f(a.m + e, m);
    ld8f(a.v + e, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) adamw_elem(a.k, g[j], p[j], m[j], v[j]);
    st8f(a.master + e, p);
    st8f(a.m + e, m);
    st8f(a.v + e, v);
    if constexpr (WRITE_P16) __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.p16) + e), narrow8<PT>(p));
  }
  // the (< 8) elements before the aligned body and the (< 8) after it
  const int64_t tail0 = a.head + nvec * kGroup;
  if (tid < a.head + (a.n - tail0)) {
    const int64_t e = tid < a.head ? tid : tail0 + (tid - a.head);
    step1<GT, PT, FROM_G32, WRITE_P16>(a, e, gs, bad);
  }
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

// Register double-buffered form for small rank counts: the loads of a
// thread's next group are issued before the update of its current group, so
// each thread keeps two groups of bytes in flight (for N <= SS_PIPE_MAX_RANKS,
// where one group alone is too few bytes to cover HBM latency at the
// residency the update's registers allow). NR is the rank count; with F the
// gradient is the fp32 array g32, held as NR = 2 raw 16-byte chunks.
#ifndef SS_PIPE_MAX_RANKS
#define SS_PIPE_MAX_RANKS 8
#endif
template <int NR>
struct PipeGroup {
  uint4 r[NR];
  float4 s[6];  // master, m, v: two float4 each
};

template <int GT, int NR, bool F, int MAXR>
__device__ __forceinline__ void pipe_load(const StepArgs<MAXR>& a, int64_t gi, PipeGroup<NR>& G) {
  const int64_t e = a.head + gi * kGroup;
  if constexpr (F) {
    static_assert(NR == 2, "the fp32 gradient occupies two chunks");
    G.r[0] = __ldcs(reinterpret_cast<const uint4*>(a.g32 + e));
    G.r[1] = __ldcs(reinterpret_cast<const uint4*>(a.g32 + e) + 1);
  } else {
#pragma unroll
    for (int r = 0; r < NR; ++r) G.r[r] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.ranks.p[r]) + e));
  }
  G.s[0] = __ldcs(reinterpret_cast<const float4*>(a.master + e));
  G.s[1] = __ldcs(reinterpret_cast<const float4*>(a.master + e) + 1);
  G.s[2] = __ldcs(reinterpret_cast<const float4*>(a.m + e));
  G.s[3] = __ldcs(reinterpret_cast<const float4*>(a.m + e) + 1);
  G.s[4] = __ldcs(reinterpret_cast<const float4*>(a.v + e));
  G.s[5] = __ldcs(reinterpret_cast<const float4*>(a.v + e) + 1);
}

template <int GT, int PT, bool F, bool WRITE_P16, int MAXR, int NR>
__global__ void __launch_bounds__(kThreads, 2) adam_pipe_kernel(const __grid_constant__ StepArgs<MAXR> a) {
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  PipeGroup<NR> cur, nxt;
  if (tid < nvec) pipe_load<GT, NR, F>(a, tid, cur);
  for (int64_t gi = tid; gi < nvec; gi += stride) {
    if (gi + stride < nvec) pipe_load<GT, NR, F>(a, gi + stride, nxt);
    const int64_t e = a.head + gi * kGroup;
    float g[8];
    if constexpr (F) {
      const uint4 x = cur.r[0], y = cur.r[1];
      g[0] = __uint_as_float(x.x); g[1] = __uint_as_float(x.y); g[2] = __uint_as_float(x.z); g[3] = __uint_as_float(x.w);
      g[4] = __uint_as_float(y.x); g[5] = __uint_as_float(y.y); g[6] = __uint_as_float(y.z); g[7] = __uint_as_float(y.w);
    } else {
      widen8<GT>(cur.r[0], g);
#pragma unroll
      for (int r = 1; r < NR; ++r) add8<GT>(cur.r[r], g);
      if (a.post_scale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
      }
    }
    if (a.nonfinite) {
#pragma unroll
      for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
    }
    if (a.g_out) st8f(a.g_out + e, g);
    if (a.dev_scale) {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = g[j] * gs;
    }
    float p[8] = {cur.s[0].x, cur.s[0].y, cur.s[0].z, cur.s[0].w, cur.s[1].x, cur.s[1].y, cur.s[1].z, cur.s[1].w};
    float m[8] = {cur.s[2].x, cur.s[2].y, cur.s[2].z, cur.s[2].w, cur.s[3].x, cur.s[3].y, cur.s[3].z, cur.s[3].w};
    float v[8] = {cur.s[4].x, cur.s[4].y, cur.s[4].z, cur.s[4].w, cur.s[5].x, cur.s[5].y, cur.s[5].z, cur.s[5].w};
#pragma unroll
    for (int j = 0; j < 8; ++j) adamw_elem(a.k, g[j], p[j], m[j], v[j]);
    st8f(a.master + e, p);
    st8f(a.m + e, m);
    st8f(a.v + e, v);
    if constexpr (WRITE_P16) __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.p16) + e), narrow8<PT>(p));
    cur = nxt;
  }
  // the (< 8) elements before the aligned body and the (< 8) after it
  const int64_t tail0 = a.head + nvec * kGroup;
  if (tid < a.head + (a.n - tail0)) {
    const int64_t e = tid < a.head ? tid : tail0 + (tid - a.head);
    step1<GT, PT, F, WRITE_P16>(a, e, gs, bad);
  }
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

template <int GT, int PT, bool FROM_G32, bool WRITE_P16, int MAXR>
__global__ void __launch_bounds__(kThreads) adam_scalar_kernel(const __grid_constant__ StepArgs<MAXR> a) {
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t e = tid; e < a.n; e += stride) step1<GT, PT, FROM_G32, WRITE_P16>(a, e, gs, bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

// ------------------------------------------------------------------ gradient reduce

template <int GT, int MAXR>
__device__ __forceinline__ void reduce_one(const ReduceArgs<MAXR>& a, int64_t e, bool& bad) {
  float g = reduce1<GT>(a.ranks, a.n_ranks, e);
  if (a.post_scale != 1.0f) g = g * a.post_scale;
  if (a.accumulate) g = a.out[e] + g;
  bad |= !finite(g);
  a.out[e] = g;
}

template <int GT, int MAXR>
__global__ void __launch_bounds__(kThreads) reduce_vec_kernel(const __grid_constant__ ReduceArgs<MAXR> a) {
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t gi = tid; gi < nvec; gi += stride) {
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
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t e = tid; e < a.n; e += stride) reduce_one<GT>(a, e, bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

// ------------------------------------------------------------------ gradient sum of squares (global clip norm)
//
// Deterministic per-shard sum of squares of the reduced gradient. The shard is
// cut into tiles of kThreads x kSumsqGroups groups of 8 elements (after the
// 0..7-element head that aligns the vectors); thread j of a tile owns groups
// j, j + kThreads, ..., issues all their loads first, adds each group's 8
// squares in fp32 (a fixed FMA chain) and the group sums in double in group
// order as fp32 pairs (TwoSum); the block combines its threads' pairs through
// a fixed shuffle tree and writes ONE double per tile into the caller's
// workspace (GB300's fp64 rate is low, so fp64 is kept to one value per tile). The
// head/tail elements (< 16) get a slot of their own. A second one-block
// kernel adds the slots in index order. The partition depends only on n and
// the arrays' 16-byte phase, never on the grid size, so the result is
// bit-reproducible.
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
// with TwoSum through a fixed shuffle tree and a fixed warp order); fp64 only
// for the block's result. Meaningful in thread 0.
__device__ __forceinline__ double block_sum(dd x, float2* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float h = __shfl_xor_sync(0xFFFFFFFFu, x.hi, off);
    const float l = __shfl_xor_sync(0xFFFFFFFFu, x.lo, off);
    const dd t = two_sum(x.hi, h);
    x = {t.hi, t.lo + (x.lo + l)};
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = make_float2(x.hi, x.lo);
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kThreads / 32; ++w) s += static_cast<double>(red[w].x) + static_cast<double>(red[w].y);
  __syncthreads();
  return s;
}

template <int GT, bool FROM_G32, bool VEC, int MAXR>
__device__ __forceinline__ float reduced1(const SumsqArgs<MAXR>& a, int64_t e) {
  if constexpr (FROM_G32) return a.g32[e];
  float g = reduce1<GT>(a.ranks, a.n_ranks, e);
  if (a.post_scale != 1.0f) g = g * a.post_scale;
  return g;
}

// NR > 0: the rank count as a compile-time constant (N <= 8), which lets the
// loads of several groups be issued together (batches of ~16 loads per
// thread); NR == 0: any rank count, one group's ranks at a time.
template <int GT, bool FROM_G32, bool VEC, int MAXR, int NR>
__global__ void __launch_bounds__(kThreads) sumsq_tiles_kernel(const __grid_constant__ SumsqArgs<MAXR> a) {
  __shared__ float2 red[kThreads / 32];
  const int64_t nvec = (a.n - a.head) / kGroup;
  bool bad = false;
  for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    // Loads of all groups first, unconditionally: a group past the end reads
    // group 0 of the shard instead (always in range: ntiles > 0 implies
    // nvec > 0) and is dropped below, so no branch stands between the loads.
    float g[kSumsqGroups][8];
    const int64_t g0 = tile * kSumsqGroups * kThreads + threadIdx.x;
    if constexpr (VEC && !FROM_G32 && NR > 0) {
      constexpr int kBatch = NR <= 2 ? 8 : (NR <= 4 ? 4 : 2);  // groups whose loads are issued together
#pragma unroll
      for (int q0 = 0; q0 < kSumsqGroups; q0 += kBatch) {
        uint4 w[kBatch][NR];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int64_t gq = g0 + (q0 + b) * kThreads;
          const int64_t e = a.head + (gq < nvec ? gq : 0) * kGroup;
#pragma unroll
          for (int r = 0; r < NR; ++r)
            w[b][r] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.ranks.p[r]) + e));
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          widen8<GT>(w[b][0], g[q0 + b]);
#pragma unroll
          for (int r = 1; r < NR; ++r) add8<GT>(w[b][r], g[q0 + b]);
          if (a.post_scale != 1.0f) {
#pragma unroll
            for (int j = 0; j < 8; ++j) g[q0 + b][j] = g[q0 + b][j] * a.post_scale;
          }
        }
      }
    } else {
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
    }
    dd s = {0.0f, 0.0f};  // the thread's group sums, accumulated exactly enough as an fp32 pair
#pragma unroll
    for (int q = 0; q < kSumsqGroups; ++q) {
      const int64_t gi = g0 + q * kThreads;
      if (gi < nvec) {
        const int64_t e = a.head + gi * kGroup;
        if (a.g_out) {
          if constexpr (VEC) {
            st8f(a.g_out + e, g[q]);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) a.g_out[e + j] = g[q][j];
          }
        }
        float c = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          bad |= !finite(g[q][j]);
          c = fmaf(g[q][j], g[q][j], c);
        }
        const dd t = two_sum(s.hi, c);
        s = {t.hi, s.lo + t.lo};
      }
    }
    const double t = block_sum(s, red);
    if (threadIdx.x == 0) a.partials[tile] = t;
  }
  // head and tail (< 16 elements) in slot ntiles, summed in element order by one thread
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int64_t tail0 = a.head + nvec * kGroup;
    double s = 0.0;
    for (int64_t i = 0; i < a.head + (a.n - tail0); ++i) {
      const int64_t e = i < a.head ? i : tail0 + (i - a.head);
      const float g = reduced1<GT, FROM_G32, VEC>(a, e);
      if (a.g_out) a.g_out[e] = g;
      bad |= !finite(g);
      s += static_cast<double>(fmaf(g, g, 0.0f));
    }
    a.partials[a.ntiles] = s;
  }
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

// out = sum of partials[0..count) in a fixed order (one block).
__global__ void __launch_bounds__(1024) sum_slots_kernel(const double* partials, int64_t count, double* out) {
  __shared__ double red[32];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < count; i += blockDim.x) s += partials[i];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
    *out = t;
  }
}

// Global clip coefficient from the shards' sums of squares, added in rank order.
__global__ void clip_coef_kernel(const double* shard_sumsq, int32_t n_shards, float max_norm, float* coef,
                                 double* norm_out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double total = 0.0;
  for (int32_t k = 0; k < n_shards; ++k) total += shard_sumsq[k];
  const double norm = sqrt(total);
  const double c = static_cast<double>(max_norm) / (norm + 1e-6);
  *coef = static_cast<float>(c < 1.0 ? c : 1.0);
  if (norm_out) *norm_out = norm;
}

// ------------------------------------------------------------------ unshard / reshard copies

template <int MAXR>
struct CopyArgs {
  const void* src[MAXR];
  void* dst[MAXR];
  int64_t bytes[MAXR];
  int32_t n_seg;
  int32_t esize;
};

// 16 bytes starting SOFF bytes into the 32-byte window (c0, c1).
template <int SOFF>
__device__ __forceinline__ uint4 window16(const uint4& c0, const uint4& c1) {
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  constexpr int q = SOFF / 4;
  constexpr int r = SOFF % 4;
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (r == 0) o[i] = w[q + i];
    else o[i] = __funnelshift_r(w[q + i], w[q + i + 1], 8 * r);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Body of one segment: destination-aligned 16-byte vectors. The source of
// vector j starts SOFF bytes past a 16-byte boundary; misaligned sources are
// read as the two aligned 16-byte chunks that hold it, and only when both
// chunks lie inside the source range -- otherwise element by element.
template <int SOFF>
__device__ __forceinline__ uint4 copy_src16(const char* s, int64_t off, int64_t bytes, int esize, bool& direct) {
  if constexpr (SOFF == 0) {
    direct = true;
    return __ldcs(reinterpret_cast<const uint4*>(s + off));
  } else {
    const char* c0 = s + off - SOFF;
    direct = c0 >= s && (off - SOFF) + 32 <= bytes;
    if (!direct) return make_uint4(0u, 0u, 0u, 0u);
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(c0));
    const uint4 b = __ldcs(reinterpret_cast<const uint4*>(c0 + 16));
    return window16<SOFF>(a, b);
  }
}

// Body of one segment: destination-aligned 16-byte vectors, kCopyUnroll per
// thread per iteration with their loads issued first. The source of vector j
// starts SOFF bytes past a 16-byte boundary; misaligned sources are read as
// the two aligned 16-byte chunks that hold it, and only when both chunks lie
// inside the source range -- otherwise element by element.
constexpr int kCopyUnroll = 4;

template <int SOFF>
__device__ __forceinline__ void copy_body(const char* s, char* d, int64_t h, int64_t nvec, int64_t bytes, int esize,
                                          int64_t tid, int64_t stride) {
  for (int64_t j0 = tid; j0 < nvec; j0 += stride * kCopyUnroll) {
    // all loads first; a vector past the end re-reads vector j0 (in range) and is not stored
    uint4 v[kCopyUnroll];
    bool direct[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t j = j0 + u * stride;
      v[u] = copy_src16<SOFF>(s, h + 16 * (j < nvec ? j : j0), bytes, esize, direct[u]);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t j = j0 + u * stride;
      if (j >= nvec) break;
      const int64_t off = h + 16 * j;
      if (direct[u]) {
        __stcs(reinterpret_cast<uint4*>(d + off), v[u]);
      } else {
        for (int i = 0; i < 16; i += esize) {
          if (esize == 2) *reinterpret_cast<uint16_t*>(d + off + i) = *reinterpret_cast<const uint16_t*>(s + off + i);
          else *reinterpret_cast<uint32_t*>(d + off + i) = *reinterpret_cast<const uint32_t*>(s + off + i);
        }
      }
    }
  }
}

template <int MAXR>
__global__ void __launch_bounds__(kThreads) copy_segments_kernel(const __grid_constant__ CopyArgs<MAXR> a) {
  const int k = blockIdx.y;
  const int64_t bytes = a.bytes[k];
  if (bytes == 0) return;
  const char* s = static_cast<const char*>(a.src[k]);
  char* d = static_cast<char*>(a.dst[k]);
  int64_t h = static_cast<int64_t>((16u - (reinterpret_cast<uintptr_t>(d) & 15u)) & 15u);
  if (h > bytes) h = bytes;
  const int64_t nvec = (bytes - h) >> 4;
  const int64_t t0 = h + (nvec << 4);
  const int soff = static_cast<int>(reinterpret_cast<uintptr_t>(s + h) & 15u);
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  switch (soff) {
    case 0: copy_body<0>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
    case 2: copy_body<2>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
    case 4: copy_body<4>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
    case 6: copy_body<6>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
    case 8: copy_body<8>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
    case 10: copy_body<10>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
    case 12: copy_body<12>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
    default: copy_body<14>(s, d, h, nvec, bytes, a.esize, tid, stride); break;
  }
  // head (h bytes) and tail (bytes - t0) element by element
  const int64_t nh = h / a.esize, nt = (bytes - t0) / a.esize;
  if (tid < nh + nt) {
    const int64_t off = tid < nh ? tid * a.esize : t0 + (tid - nh) * a.esize;
    if (a.esize == 2) *reinterpret_cast<uint16_t*>(d + off) = *reinterpret_cast<const uint16_t*>(s + off);
    else *reinterpret_cast<uint32_t*>(d + off) = *reinterpret_cast<const uint32_t*>(s + off);
  }
}

// ------------------------------------------------------------------ unshard / reshard with the bulk-copy engine
//
// When every segment's source and destination share a 16-byte phase, the copy
// is handed to the TMA engine: a one-warp block streams its chunks of a
// segment global -> shared -> global with cp.async.bulk, kTmaSlots chunks of
// kTmaChunk bytes in flight (loads completed on an mbarrier, stores tracked as
// bulk groups). The threads only issue copies, so a few blocks per SM keep
// ~200 KB moving. The 0..14 bytes before the first 16-byte boundary and the
// 0..14 after the last are copied element by element.
//
// Each mbarrier wait is bounded (about one second of %globaltimer); on expiry
// the block records bit 0 in the library's device error word
// (ss_device_error), lets its copies in flight land (bounded again) and
// returns instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
#ifndef SS_TMA_CHUNK
#define SS_TMA_CHUNK 16384
#endif
#ifndef SS_TMA_SLOTS
#define SS_TMA_SLOTS 4
#endif
constexpr int kTmaChunk = SS_TMA_CHUNK;
constexpr int kTmaSlots = SS_TMA_SLOTS;
enum : uint32_t { SS_DEVERR_TIMEOUT = 1u };

__device__ uint32_t g_device_error = 0;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Wait for the phase of the given parity to complete, for at most ~1 s.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_device_error, SS_DEVERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Global -> shared; bytes and both addresses multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Shared -> global; bytes and both addresses multiples of 16.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int MAXR>
__global__ void __launch_bounds__(32) copy_tma_kernel(const __grid_constant__ CopyArgs<MAXR> a) {
  extern __shared__ __align__(128) unsigned char buf[];  // [kTmaSlots][kTmaChunk]
  __shared__ __align__(8) uint64_t bars[kTmaSlots];
  const int k = blockIdx.y;
  const int64_t bytes = a.bytes[k];
  if (bytes == 0) return;
  const char* s = static_cast<const char*>(a.src[k]);
  char* d = static_cast<char*>(a.dst[k]);
  int64_t h = static_cast<int64_t>((16u - (reinterpret_cast<uintptr_t>(d) & 15u)) & 15u);
  if (h > bytes) h = bytes;
  const int64_t body = ((bytes - h) / 16) * 16;
  const int lane = threadIdx.x;
  // head and tail (< 16 bytes each), element by element, in block 0 of the segment
  if (blockIdx.x == 0) {
    const int64_t nh = h / a.esize, nt = (bytes - h - body) / a.esize;
    if (lane < nh + nt) {
      const int64_t off = lane < nh ? lane * a.esize : h + body + (lane - nh) * a.esize;
      if (a.esize == 2) *reinterpret_cast<uint16_t*>(d + off) = *reinterpret_cast<const uint16_t*>(s + off);
      else *reinterpret_cast<uint32_t*>(d + off) = *reinterpret_cast<const uint32_t*>(s + off);
    }
  }
  if (lane != 0) return;
  const uint32_t bar0 = smem_addr(bars), buf0 = smem_addr(buf);
  for (int i = 0; i < kTmaSlots; ++i) mbar_init(bar0 + 8u * i, 1u);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const int64_t nch = (body + kTmaChunk - 1) / kTmaChunk;
  const int64_t bx = blockIdx.x, gx = gridDim.x;
  const int64_t cnt = nch > bx ? (nch - bx + gx - 1) / gx : 0;  // chunks bx, bx + gx, ...
  auto chunk_bytes = [&](int64_t i) {
    const int64_t left = body - (bx + i * gx) * kTmaChunk;
    return static_cast<uint32_t>(left < kTmaChunk ? left : kTmaChunk);
  };
  auto issue = [&](int64_t i) {
    const uint32_t slot = static_cast<uint32_t>(i % kTmaSlots);
    const uint32_t nb = chunk_bytes(i);
    mbar_expect_tx(bar0 + 8u * slot, nb);
    bulk_load(buf0 + slot * kTmaChunk, s + h + (bx + i * gx) * kTmaChunk, nb, bar0 + 8u * slot);
  };
  const int64_t first = cnt < kTmaSlots ? cnt : kTmaSlots;
  for (int64_t i = 0; i < first; ++i) issue(i);
  int64_t issued = first, i = 0;
  for (; i < cnt; ++i) {
    const uint32_t slot = static_cast<uint32_t>(i % kTmaSlots);
    if (!mbar_wait(bar0 + 8u * slot, static_cast<uint32_t>((i / kTmaSlots) & 1))) break;
    bulk_store(d + h + (bx + i * gx) * kTmaChunk, buf0 + slot * kTmaChunk, chunk_bytes(i));
    bulk_commit();
    if (issued < cnt) {
      bulk_wait_read_all();  // the store just issued has read its slot: the slot may be refilled
      issue(issued++);
    }
  }
  bulk_wait_all();
  // after a timed-out wait: let the loads already issued land before the block exits
  for (int64_t j = i + 1; j < issued; ++j)
    mbar_wait(bar0 + 8u * static_cast<uint32_t>(j % kTmaSlots), static_cast<uint32_t>((j / kTmaSlots) & 1));
}

// ------------------------------------------------------------------ fused AdamW step, 16-bit arrays off the state's phase
//
// When the fp32 arrays share a 16-byte phase but some 16-bit arrays (rank
// gradients, param16) do not -- shard views at boundaries that are not
// multiples of 8 elements, or param16 inside a flat buffer at such a
// boundary -- groups still start where the fp32 arrays are 16-byte aligned.
// Every 16-bit gradient array is read as the two aligned 16-byte chunks that
// hold the group (all loads issued first) and funnel-shifted to its phase;
// param16 is stored in 4- or 2-byte pieces when it is off phase. The body is groups 1 .. nvec-2, so every chunk read lies inside its
// array; the first and last groups and the head/tail elements are done one by
// one.
template <int MAXR>
struct ShiftArgs {
  StepArgs<MAXR> s;
  uint8_t rphase[MAXR];  // byte offset of each rank's group starts past a 16-byte boundary (even)
  uint8_t pphase;        // the same for param16
};

// The 16 bytes that start `phase` bytes into the 32-byte window (a, b).
__device__ __forceinline__ uint4 window_at(const uint4& a, const uint4& b, int phase) {
  switch (phase) {
    case 0: return a;
    case 2: return window16<2>(a, b);
    case 4: return window16<4>(a, b);
    case 6: return window16<6>(a, b);
    case 8: return window16<8>(a, b);
    case 10: return window16<10>(a, b);
    case 12: return window16<12>(a, b);
    default: return window16<14>(a, b);
  }
}

__device__ __forceinline__ void st16_at_phase(void* p, const uint4& v, int phase) {
  if (phase == 0) {
    __stcs(reinterpret_cast<uint4*>(p), v);
  } else if ((phase & 3) == 0) {
    uint32_t* q = static_cast<uint32_t*>(p);
    q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
  } else {
    uint16_t* q = static_cast<uint16_t*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      q[2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
      q[2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
    }
  }
}

template <int GT, int PT, bool FROM_G32, bool WRITE_P16, int MAXR>
__global__ void __launch_bounds__(kThreads) adam_shift_kernel(const __grid_constant__ ShiftArgs<MAXR> x) {
  const StepArgs<MAXR>& a = x.s;
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t g_lo = nvec >= 3 ? 1 : 0, g_hi = nvec >= 3 ? nvec - 1 : 0;  // vector body [g_lo, g_hi)
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t gi = g_lo + tid; gi < g_hi; gi += stride) {
    const int64_t e = a.head + gi * kGroup;
    float g[8];
    if constexpr (FROM_G32) {
      ld8f(a.g32 + e, g);
    } else {
      for (int r0 = 0; r0 < a.n_ranks; r0 += 8) {
        // both aligned chunks around every rank's group, all loads issued before any use
        // (in the body the second chunk is always inside the array, even at phase 0)
        uint4 c0[8], c1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (r0 + j < a.n_ranks) {
            const uint4* c = reinterpret_cast<const uint4*>(
                reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[r0 + j]) + e) - x.rphase[r0 + j]);
            c0[j] = __ldcs(c);
            c1[j] = __ldcs(c + 1);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (r0 + j < a.n_ranks) {
            const uint4 w = window_at(c0[j], c1[j], x.rphase[r0 + j]);
            if (r0 + j == 0) widen8<GT>(w, g);
            else add8<GT>(w, g);
          }
        }
      }
      if (a.post_scale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
      }
    }
    if (a.nonfinite) {
#pragma unroll
      for (int j = 0; j < 8; ++j) bad |= !finite(g[j]);
    }
    if (a.g_out) st8f(a.g_out + e, g);
    if (a.dev_scale) {
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = g[j] * gs;
    }
    float p[8], m[8], v[8];
    ld8f(a.master + e, p);
    ld8f(a.m + e, m);
    ld8f(a.v + e, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) adamw_elem(a.k, g[j], p[j], m[j], v[j]);
    st8f(a.master + e, p);
    st8f(a.m + e, m);
    st8f(a.v + e, v);
    if constexpr (WRITE_P16) st16_at_phase(static_cast<uint16_t*>(a.p16) + e, narrow8<PT>(p), x.pphase);
  }
  // everything outside the vector body, one element per thread (< 31 elements)
  const int64_t lo_end = a.head + g_lo * kGroup, hi_start = a.head + g_hi * kGroup;
  const int64_t n_edge = lo_end + (a.n - hi_start);
  if (tid < n_edge) step1<GT, PT, FROM_G32, WRITE_P16>(a, tid < lo_end ? tid : hi_start + (tid - lo_end), gs, bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && (threadIdx.x & 31) == 0) *a.nonfinite = 1;
  }
}

// ------------------------------------------------------------------ host helpers

struct Range {
  uintptr_t lo, hi;
  bool out;
};

// True when some output byte range overlaps any other range (inputs may overlap inputs).
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

// Smallest h in [0, 8) with every 16-bit pointer at a 16-byte boundary after h
// elements and every fp32 pointer likewise; -1 when none exists.
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

// Resident blocks per SM of a kernel launched with `threads` per block (cached per kernel).
int blocks_per_sm(const void* fn, int threads = kThreads) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& c : cache)
    if (c.first == fn) return c.second;
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, 0) != cudaSuccess || b < 1) b = 1;
  cache.emplace_back(fn, b);
  return b;
}

unsigned grid_for(const void* fn, int64_t work_items, int threads = kThreads) {
  const int64_t want = std::max<int64_t>(1, (work_items + threads - 1) / threads);
  const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>(sm_count()) * blocks_per_sm(fn, threads));
  return static_cast<unsigned>(std::min(want, cap));
}

template <typename Args, typename Fn>
ss_status launch(Fn* fn, unsigned grid, const Args& args, void* stream, int threads = kThreads) {
  fn<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(args);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SS_OK : cuda_fail(e);
}

bool is16(ss_dtype d) { return d == SS_BF16 || d == SS_FP16; }

// Splits a double into an fp32 pair hi + lo (hi = nearest float, lo = nearest float to the rest).
void split(double x, float& hi, float& lo) {
  hi = static_cast<float>(x);
  lo = static_cast<float>(x - static_cast<double>(hi));
}

AdamConst make_const(const ss_adamw_hparams& hp) {
  const double b1 = hp.beta1, b2 = hp.beta2;
  const double bc1 = 1.0 - std::pow(b1, static_cast<double>(hp.step));
  const double bc2 = 1.0 - std::pow(b2, static_cast<double>(hp.step));
  const double sq = std::sqrt(bc2);
  AdamConst k;
  k.b1 = hp.beta1;
  split(1.0 - b1, k.c1, k.c1_lo);
  k.b2 = hp.beta2;
  split(1.0 - b2, k.c2, k.c2_lo);
  split(static_cast<double>(hp.lr) * sq / bc1, k.A_hi, k.A_lo);
  split(static_cast<double>(hp.eps) * sq, k.E_hi, k.E_lo);
  split(1.0 - static_cast<double>(hp.lr) * static_cast<double>(hp.weight_decay), k.D_hi, k.D_lo);
  return k;
}

bool valid_hp(const ss_adamw_hparams* hp) {
  if (!hp || hp->step < 1) return false;
  const float f[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
  for (float x : f)
    if (!std::isfinite(x) || x < 0.0f) return false;
  return hp->beta1 < 1.0f && hp->beta2 < 1.0f;
}

// ---- dispatch tables (template instantiation by runtime dtype / options)

enum class Path { kScalar, kVector, kPipe, kShift };

template <int G, int P, bool F, bool W, int MAXR>
ss_status launch_shift(const StepArgs<MAXR>& a, const uint8_t* rphase, uint8_t pphase, void* stream) {
  ShiftArgs<MAXR> x;
  std::memset(&x, 0, sizeof x);
  x.s = a;
  for (int32_t r = 0; r < a.n_ranks; ++r) x.rphase[r] = rphase[r];
  x.pphase = pphase;
  auto* fn = adam_shift_kernel<G, P, F, W, MAXR>;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup), x, stream);
}

template <int G, int P, bool W, int MAXR, int NR, bool F = false>
ss_status launch_pipe_n(const StepArgs<MAXR>& a, void* stream) {
  auto* fn = adam_pipe_kernel<G, P, F, W, MAXR, NR>;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup), a, stream);
}

template <int G, int P, bool W, int MAXR>
ss_status launch_pipe(const StepArgs<MAXR>& a, void* stream) {
  switch (a.n_ranks) {
    case 1: return launch_pipe_n<G, P, W, MAXR, 1>(a, stream);
    case 2: return launch_pipe_n<G, P, W, MAXR, 2>(a, stream);
#if SS_PIPE_MAX_RANKS >= 3
    case 3: return launch_pipe_n<G, P, W, MAXR, 3>(a, stream);
#endif
#if SS_PIPE_MAX_RANKS >= 4
    case 4: return launch_pipe_n<G, P, W, MAXR, 4>(a, stream);
#endif
#if SS_PIPE_MAX_RANKS >= 8
    case 5: return launch_pipe_n<G, P, W, MAXR, 5>(a, stream);
    case 6: return launch_pipe_n<G, P, W, MAXR, 6>(a, stream);
    case 7: return launch_pipe_n<G, P, W, MAXR, 7>(a, stream);
    case 8: return launch_pipe_n<G, P, W, MAXR, 8>(a, stream);
#endif
    default: return SS_ERR_INVALID_ARG;
  }
}

template <int MAXR>
ss_status run_adam(const StepArgs<MAXR>& a, Path path, bool from_g32, bool p16, ss_dtype gt, ss_dtype pt,
                   const uint8_t* rphase, uint8_t pphase, void* stream) {
#define SS_ADAM_CASE(G, P, F, W)                                                          \
  if (gt == G && pt == P && from_g32 == F && p16 == W) {                                  \
    if (path == Path::kShift) return launch_shift<G, P, F, W, MAXR>(a, rphase, pphase, stream); \
    if (path == Path::kPipe) {                                                            \
      if constexpr (F) return launch_pipe_n<G, P, W, MAXR, 2, true>(a, stream);           \
      else return launch_pipe<G, P, W, MAXR>(a, stream);                                  \
    }                                                                                     \
    if (path == Path::kVector) {                                                          \
      auto* fn = adam_vec_kernel<G, P, F, W, MAXR>;                                       \
      return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup, kStepThreads), a, \
                    stream, kStepThreads);                                                \
    }                                                                                     \
    auto* fn = adam_scalar_kernel<G, P, F, W, MAXR>;                                      \
    return launch(fn, grid_for(reinterpret_cast<const void*>(fn), a.n), a, stream);       \
  }
#define SS_ADAM_P(G, P) SS_ADAM_CASE(G, P, false, true) SS_ADAM_CASE(G, P, false, false) \
                        SS_ADAM_CASE(G, P, true, true) SS_ADAM_CASE(G, P, true, false)
  SS_ADAM_P(SS_BF16, SS_BF16)
  SS_ADAM_P(SS_BF16, SS_FP16)
  SS_ADAM_P(SS_FP16, SS_BF16)
  SS_ADAM_P(SS_FP16, SS_FP16)
#undef SS_ADAM_P
#undef SS_ADAM_CASE
  return SS_ERR_DTYPE;
}

template <int MAXR>
ss_status run_reduce(const ReduceArgs<MAXR>& a, bool vec, ss_dtype gt, void* stream) {
#define SS_RED_CASE(G)                                                                     \
  if (gt == G) {                                                                           \
    if (vec) {                                                                             \
      auto* fn = reduce_vec_kernel<G, MAXR>;                                               \
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

// Raise a kernel's dynamic shared memory limit once (cached per kernel).
bool allow_smem(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, size_t>> done;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& d : done)
    if (d.first == fn && d.second >= bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess)
    return false;
  done.emplace_back(fn, bytes);
  return true;
}

template <int MAXR>
ss_status run_copy(const void* const* src, void* const* dst, const int64_t* bytes, int32_t n_seg, int32_t esize,
                   int64_t total_bytes, void* stream) {
  CopyArgs<MAXR> a;
  std::memset(&a, 0, sizeof a);
  bool same_phase = true;
  for (int32_t k = 0; k < n_seg; ++k) {
    a.src[k] = src[k];
    a.dst[k] = dst[k];
    a.bytes[k] = bytes[k];
    if (bytes[k] > 0 && ((reinterpret_cast<uintptr_t>(src[k]) - reinterpret_cast<uintptr_t>(dst[k])) & 15u) != 0)
      same_phase = false;
  }
  a.n_seg = n_seg;
  a.esize = esize;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (same_phase && total_bytes >= (int64_t{1} << 20)) {
    // bulk-copy engine: one-warp blocks, kTmaSlots chunks in flight each
    auto* fn = copy_tma_kernel<MAXR>;
    const size_t smem = static_cast<size_t>(kTmaSlots) * kTmaChunk;
    const void* f = reinterpret_cast<const void*>(fn);
    if (!allow_smem(f, smem)) return cuda_fail(cudaGetLastError());
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, 32, smem) != cudaSuccess || per_sm < 1) per_sm = 1;
    const int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
    const int64_t chunks = (total_bytes / std::max(1, n_seg)) / kTmaChunk + 1;
    const int64_t gx = std::max<int64_t>(1, std::min<int64_t>((cap + n_seg - 1) / n_seg, chunks));
    fn<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(n_seg)), 32, smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SS_OK : cuda_fail(e);
  }
  auto* fn = copy_segments_kernel<MAXR>;
  const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(fn)));
  const int64_t per_seg_work = (total_bytes / std::max(1, n_seg)) / 16 + 1;
  int64_t gx = std::min<int64_t>((cap + n_seg - 1) / n_seg, (per_seg_work + kThreads - 1) / kThreads);
  gx = std::max<int64_t>(gx, 1);
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(n_seg));
  fn<<<grid, kThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SS_OK : cuda_fail(e);
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

}  // namespace
}  // namespace ss

namespace ss {
namespace {

template <int MAXR>
ss_status run_sumsq(const SumsqArgs<MAXR>& a, bool vec, bool from_g32, ss_dtype gt, double* out, void* stream) {
  const unsigned grid = static_cast<unsigned>(
      std::max<int64_t>(1, std::min<int64_t>(a.ntiles, static_cast<int64_t>(sm_count()) * 4)));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nr = (vec && !from_g32 && a.n_ranks <= 8) ? a.n_ranks : 0;
#define SS_SUMSQ_NR(G, R) \
  case R: sumsq_tiles_kernel<G, false, true, MAXR, R><<<grid, kThreads, 0, st>>>(a); break;
#define SS_SUMSQ_RANKED(G)                                                                              \
  switch (nr) {                                                                                         \
    SS_SUMSQ_NR(G, 1) SS_SUMSQ_NR(G, 2) SS_SUMSQ_NR(G, 3) SS_SUMSQ_NR(G, 4)                             \
    SS_SUMSQ_NR(G, 5) SS_SUMSQ_NR(G, 6) SS_SUMSQ_NR(G, 7) SS_SUMSQ_NR(G, 8)                             \
    default: sumsq_tiles_kernel<G, false, true, MAXR, 0><<<grid, kThreads, 0, st>>>(a);                 \
  }
  if (!from_g32 && vec && gt == SS_BF16) {
    SS_SUMSQ_RANKED(SS_BF16)
  } else if (!from_g32 && vec && gt == SS_FP16) {
    SS_SUMSQ_RANKED(SS_FP16)
  } else if (!from_g32 && gt == SS_BF16) {
    sumsq_tiles_kernel<SS_BF16, false, false, MAXR, 0><<<grid, kThreads, 0, st>>>(a);
  } else if (!from_g32 && gt == SS_FP16) {
    sumsq_tiles_kernel<SS_FP16, false, false, MAXR, 0><<<grid, kThreads, 0, st>>>(a);
  } else if (from_g32 && vec) {
    sumsq_tiles_kernel<SS_BF16, true, true, MAXR, 0><<<grid, kThreads, 0, st>>>(a);
  } else if (from_g32) {
    sumsq_tiles_kernel<SS_BF16, true, false, MAXR, 0><<<grid, kThreads, 0, st>>>(a);
  } else {
    return SS_ERR_DTYPE;
  }
#undef SS_SUMSQ_RANKED
#undef SS_SUMSQ_NR
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  sum_slots_kernel<<<1, 1024, 0, st>>>(a.partials, a.ntiles + 1, out);
  e = cudaGetLastError();
  return e == cudaSuccess ? SS_OK : cuda_fail(e);
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
  const int h = common_phase(p16, p32);
  const bool vec = h >= 0 && h < n;
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
    return run_sumsq(a, vec, from_g32, gt, sumsq_out, stream);
  }
  SumsqArgs<kLargeRanks> a;
  std::memset(&a, 0, sizeof a);
  fill(a);
  return run_sumsq(a, vec, from_g32, gt, sumsq_out, stream);
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" {

const char* ss_last_cuda_error(void) { return g_cuda_err; }

ss_status ss_device_error(uint32_t* out, int32_t clear) {
  if (!out) return SS_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(e);
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return SS_OK;
}

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
  auto fill = [&](auto& a) {
    for (int32_t r = 0; r < n_ranks; ++r) a.ranks.p[r] = rank_grads[r];
    a.out = g_out;
    a.nonfinite = nonfinite_flag;
    a.n = n;
    a.head = vec ? h : 0;
    a.n_ranks = n_ranks;
    a.post_scale = post_scale;
    a.accumulate = accumulate != 0;
  };
  if (n_ranks <= kSmallRanks) {
    ReduceArgs<kSmallRanks> a;
    std::memset(&a, 0, sizeof a);
    fill(a);
    return run_reduce(a, vec, gdtype, stream);
  }
  ReduceArgs<kLargeRanks> a;
  std::memset(&a, 0, sizeof a);
  fill(a);
  return run_reduce(a, vec, gdtype, stream);
}

ss_status ss_adam_step(const ss_adamw_hparams* hp, int64_t n, const float* g32, const void* const* rank_grads,
                       int32_t n_ranks, ss_dtype gdtype, float post_scale, float* master, float* m, float* v,
                       void* param16, ss_dtype pdtype, const ss_step_options* opts, void* stream) {
  if (!valid_hp(hp) || n < 0) return SS_ERR_INVALID_ARG;
  if (n > INT64_MAX / 16) return SS_ERR_OVERFLOW;
  if (!master || !m || !v) return SS_ERR_INVALID_ARG;
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
  for (const float* p : {static_cast<const float*>(master), static_cast<const float*>(m), static_cast<const float*>(v)}) {
    if (reinterpret_cast<uintptr_t>(p) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(p, 4 * n, true));
    p32.push_back(reinterpret_cast<uintptr_t>(p));
  }
  if (param16) {
    if (!is16(pdtype)) return SS_ERR_DTYPE;
    if (reinterpret_cast<uintptr_t>(param16) & 1u) return SS_ERR_ALIGN;
    ranges.push_back(rng(param16, 2 * n, true));
    p16.push_back(reinterpret_cast<uintptr_t>(param16));
  }
  ss_step_options o{};
  if (opts) o = *opts;
  if (o.g_out) {
    if (reinterpret_cast<uintptr_t>(o.g_out) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(o.g_out, 4 * n, true));
    p32.push_back(reinterpret_cast<uintptr_t>(o.g_out));
  }
  if (o.nonfinite_flag) {
    if (reinterpret_cast<uintptr_t>(o.nonfinite_flag) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(o.nonfinite_flag, 4, true));
  }
  if (o.dev_grad_scale) {
    if (reinterpret_cast<uintptr_t>(o.dev_grad_scale) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(o.dev_grad_scale, 4, false));
  }
  if (o.dev_skip_flag) {
    if (reinterpret_cast<uintptr_t>(o.dev_skip_flag) & 3u) return SS_ERR_ALIGN;
    ranges.push_back(rng(o.dev_skip_flag, 4, false));
  }
  if (any_output_overlap(ranges)) return SS_ERR_OVERLAP;
  if (n == 0) return SS_OK;
  int h = common_phase(p16, p32);
  const bool vec = h >= 0 && h < n;
  Path path = !vec ? Path::kScalar : ((from_g32 || n_ranks <= SS_PIPE_MAX_RANKS) ? Path::kPipe : Path::kVector);
  // 16-bit arrays off the fp32 arrays' phase: per-array byte phases at the fp32 group starts
  std::vector<uint8_t> rphase(from_g32 ? 0 : n_ranks, 0);
  uint8_t pphase = 0;
  if (!vec) {
    const int h32 = common_phase({}, p32);
    if (h32 >= 0 && n - h32 >= 3 * kGroup) {
      h = h32;
      path = Path::kShift;
      if (!from_g32)
        for (int32_t r = 0; r < n_ranks; ++r)
          rphase[r] = static_cast<uint8_t>((reinterpret_cast<uintptr_t>(rank_grads[r]) + 2u * h) & 15u);
      if (param16) pphase = static_cast<uint8_t>((reinterpret_cast<uintptr_t>(param16) + 2u * h) & 15u);
    }
  }
  const AdamConst k = make_const(*hp);
  auto fill = [&](auto& a) {
    if (!from_g32)
      for (int32_t r = 0; r < n_ranks; ++r) a.ranks.p[r] = rank_grads[r];
    a.g32 = g32;
    a.master = master;
    a.m = m;
    a.v = v;
    a.p16 = param16;
    a.g_out = o.g_out;
    a.nonfinite = o.nonfinite_flag;
    a.dev_scale = o.dev_grad_scale;
    a.dev_skip = o.dev_skip_flag;
    a.n = n;
    a.head = path == Path::kScalar ? 0 : h;
    a.n_ranks = from_g32 ? 0 : n_ranks;
    a.post_scale = post_scale;
    a.k = k;
  };
  const ss_dtype gt = from_g32 ? SS_BF16 : gdtype;
  const ss_dtype pt = param16 ? pdtype : SS_BF16;
  if (from_g32 || n_ranks <= kSmallRanks) {
    StepArgs<kSmallRanks> a;
    std::memset(&a, 0, sizeof a);
    fill(a);
    return run_adam(a, path, from_g32, param16 != nullptr, gt, pt, rphase.data(), pphase, stream);
  }
  StepArgs<kLargeRanks> a;
  std::memset(&a, 0, sizeof a);
  fill(a);
  return run_adam(a, path, from_g32, param16 != nullptr, gt, pt, rphase.data(), pphase, stream);
}

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

// Device address of the slot array on the current device. The name of the
// array is only a host-side stand-in; the address comes from the runtime, once
// per device, with that device current.
ss_status noalloc_slots(double** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static double* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return SS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_sumsq_slots);
    if (e != cudaSuccess) return cuda_fail(e);
    addr[dev] = static_cast<double*>(p);
  }
  *out = addr[dev];
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
  clip_coef_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(shard_sumsq, n_shards, max_norm, coef_out, norm_out);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SS_OK : cuda_fail(e);
}

static ss_status copy_common(const void* const* src, void* const* dst, const int64_t* shard_bounds, int32_t n_ranks,
                             ss_dtype dtype, bool unshard, void* stream) {
  if (!shard_bounds || n_ranks < 1 || n_ranks > SS_MAX_RANKS) return SS_ERR_INVALID_ARG;
  if (dtype != SS_BF16 && dtype != SS_FP16 && dtype != SS_FP32) return SS_ERR_DTYPE;
  const int32_t es = dtype == SS_FP32 ? 4 : 2;
  if (shard_bounds[0] != 0) return SS_ERR_INVALID_ARG;
  for (int32_t k = 0; k < n_ranks; ++k)
    if (shard_bounds[k + 1] < shard_bounds[k]) return SS_ERR_INVALID_ARG;
  const int64_t P = shard_bounds[n_ranks];
  if (P > INT64_MAX / 8) return SS_ERR_OVERFLOW;
  std::vector<const void*> s(n_ranks);
  std::vector<void*> d(n_ranks);
  std::vector<int64_t> b(n_ranks);
  std::vector<Range> ranges;
  const void* flat = unshard ? static_cast<const void*>(dst[0]) : src[0];
  if (!flat && P > 0) return SS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(flat) % es) return SS_ERR_ALIGN;
  ranges.push_back(rng(flat, es * P, unshard));
  for (int32_t k = 0; k < n_ranks; ++k) {
    const int64_t len = shard_bounds[k + 1] - shard_bounds[k];
    const void* shard = unshard ? src[k + 1] : static_cast<const void*>(dst[k + 1]);
    if (len > 0 && !shard) return SS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(shard) % es) return SS_ERR_ALIGN;
    ranges.push_back(rng(shard, es * len, !unshard));
    char* fk = static_cast<char*>(const_cast<void*>(flat)) + es * shard_bounds[k];
    s[k] = unshard ? shard : fk;
    d[k] = unshard ? static_cast<void*>(fk) : const_cast<void*>(shard);
    b[k] = es * len;
  }
  if (any_output_overlap(ranges)) return SS_ERR_OVERLAP;
  if (P == 0) return SS_OK;
  if (n_ranks <= kSmallRanks) return run_copy<kSmallRanks>(s.data(), d.data(), b.data(), n_ranks, es, es * P, stream);
  return run_copy<kLargeRanks>(s.data(), d.data(), b.data(), n_ranks, es, es * P, stream);
}

ss_status ss_unshard(const void* const* shards, const int64_t* shard_bounds, int32_t n_ranks, ss_dtype dtype,
                     void* flat, void* stream) {
  if (!shards || n_ranks < 1 || n_ranks > SS_MAX_RANKS) return SS_ERR_INVALID_ARG;
  std::vector<const void*> src(n_ranks + 1);
  std::vector<void*> dst(n_ranks + 1);
  dst[0] = flat;
  for (int32_t k = 0; k < n_ranks; ++k) src[k + 1] = shards[k];
  return copy_common(src.data(), dst.data(), shard_bounds, n_ranks, dtype, true, stream);
}

ss_status ss_reshard(const void* flat, const int64_t* shard_bounds, int32_t n_ranks, ss_dtype dtype,
                     void* const* shards, void* stream) {
  if (!shards || n_ranks < 1 || n_ranks > SS_MAX_RANKS) return SS_ERR_INVALID_ARG;
  std::vector<const void*> src(n_ranks + 1);
  std::vector<void*> dst(n_ranks + 1);
  src[0] = flat;
  for (int32_t k = 0; k < n_ranks; ++k) dst[k + 1] = shards[k];
  return copy_common(src.data(), dst.data(), shard_bounds, n_ranks, dtype, false, stream);
}

}  // extern "C"
