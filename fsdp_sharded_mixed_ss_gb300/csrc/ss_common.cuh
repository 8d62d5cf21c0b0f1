// ss_common.cuh -- pieces shared by the CUDA sources of the shard-step library:
// launch constants, 16-bit <-> fp32 vector helpers, the kernels' argument
// blocks, the rank-ordered gradient sum, and the host-side argument checks.
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
//   * persistent grid, one wave (SM count x resident blocks); the fused step
//     and the reduce of up to 8 ranks run one block per SM whose warps take
//     chunks of 32 groups from a shared-memory counter (work division below),
//     the other kernels a grid-stride loop;
//   * rank gradients are summed in rank order in batches of 8 loads issued
//     before the adds (8 x 16 B in flight per thread for any N);
//   * streaming cache hints (evict-first) on read-once and write-once data;
//   * rank pointer tables travel in the kernel's parameter space
//     (__grid_constant__), so indexing them costs a constant-bank load;
//   * odd-length shards and arbitrary views: the first 0..7 elements up to
//     the common 16-byte phase and the last 0..7 elements are done one by one
//     by the first threads of the grid; 16-bit arrays off the fp32 arrays'
//     phase are read as aligned chunk pairs and shifted into place; arrays
//     with no usable phase at all take the element-wise kernel (same results).
#pragma once

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

constexpr int kThreads = 256;
// Block shape of the fused step kernels whose warps take chunks of work from a
// counter in shared memory (the register-heavy ones): 512 threads, one block
// per SM at 128 registers a thread, so all 16 warps of an SM share one counter.
#ifndef SS_CHUNK_THREADS
#define SS_CHUNK_THREADS 512
#endif
constexpr int kChunkThreads = SS_CHUNK_THREADS;
constexpr int kChunkWarps = kChunkThreads / 32;
constexpr int kChunkBlocksPerSm = 512 / kChunkThreads;
constexpr int kGroup = 8;         // elements per thread per iteration
constexpr int kSmallRanks = 64;   // pointer table size of the common kernels
constexpr int kLargeRanks = SS_MAX_RANKS;

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

// Hint to the L2: fetch `bytes` bytes at p from DRAM now (one bulk prefetch;
// p 16-byte aligned, bytes a multiple of 16, the range inside one array).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

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

// ------------------------------------------------------------------ warp-cooperative shifted loads
//
// A 16-bit array whose 8-element groups do not start on 16-byte boundaries
// (a view at an offset that is not a multiple of 8 elements) is read by whole
// warps: a warp takes runs of kRun consecutive groups; lane j loads the aligned
// 16-byte chunk under the start of group j of the run (lane 31 the one under
// the group after the run), the lanes combine their chunks element by element
// as the caller needs (e.g. the ranks' fp32 sum), and each lane then moves its
// group's 8 values into place, taking the ones past its own chunk from the
// next lane by shuffle. Each byte is loaded once.
constexpr int kRun = 31;  // groups per warp run

// c <- elements SH .. SH + 7 of the 16 values (this lane's c, the next lane's c),
// in place: only the SH values that come from the next lane are shuffled, and
// they are taken before c is moved down (all lanes of the warp call it with
// the same SH).
template <int SH>
__device__ __forceinline__ void shift_down8(float (&c)[8]) {
  float d[SH > 0 ? SH : 1];
#pragma unroll
  for (int j = 0; j < SH; ++j) d[j] = __shfl_down_sync(0xFFFFFFFFu, c[j], 1);
#pragma unroll
  for (int i = 0; i + SH < 8; ++i) c[i] = c[i + SH];
#pragma unroll
  for (int j = 0; j < SH; ++j) c[8 - SH + j] = d[j];
}

__device__ __forceinline__ void shift_down8(float (&g)[8], int sh) {
  switch (sh) {  // warp-uniform
    case 0: break;
    case 1: shift_down8<1>(g); break;
    case 2: shift_down8<2>(g); break;
    case 3: shift_down8<3>(g); break;
    case 4: shift_down8<4>(g); break;
    case 5: shift_down8<5>(g); break;
    case 6: shift_down8<6>(g); break;
    default: shift_down8<7>(g); break;
  }
}

// The 16-bit values SH .. SH + 7 of the 16 in (this lane's chunk c, the next
// lane's chunk), still packed: only the ceil(SH / 2) words that hold values
// from the next lane are shuffled, then funnel-shifted into place (all lanes of
// the warp call it with the same SH). Shifting before widening moves half the
// words a shift of the eight fp32 values would.
template <int SH>
__device__ __forceinline__ uint4 shift_chunk(const uint4& c) {
  constexpr int nw = (SH + 1) / 2;
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t d[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < nw; ++j) d[j] = __shfl_down_sync(0xFFFFFFFFu, w[j], 1);
  return window16<2 * SH>(c, make_uint4(d[0], d[1], d[2], d[3]));
}

__device__ __forceinline__ uint4 shift_chunk(const uint4& c, int sh) {
  switch (sh) {  // warp-uniform
    case 0: return c;
    case 1: return shift_chunk<1>(c);
    case 2: return shift_chunk<2>(c);
    case 3: return shift_chunk<3>(c);
    case 4: return shift_chunk<4>(c);
    case 5: return shift_chunk<5>(c);
    case 6: return shift_chunk<6>(c);
    default: return shift_chunk<7>(c);
  }
}

// ------------------------------------------------------------------ work division
//
// The step and reduce kernels run one wave of blocks, one per SM. A chunk is 32
// consecutive 8-element groups, one per lane of a warp; each block owns a fixed
// set of chunks and its warps take them in order from a counter in shared
// memory, so a warp whose loads come back sooner takes more of them and the
// warps of an SM finish together. Measured on GB300 (fused step, GPT-2 shard,
// N = 8, per-warp timer stamps in a probe build): with one fixed chunk per warp
// and pass over the grid the warps of an SM finished up to ~9 us apart in a
// ~100 us launch, with the counter within ~3 us.
//
// Which chunks block b of B owns: round robin, chunks b, b + B, b + 2B, ...
// (the blocks' counts differ by at most one); or ADJACENT: W adjacent chunks
// (W = warps per block) of every full pass of the grid over W * B chunks, and
// round robin over the final partial pass. Either way the grid as a whole
// moves through the arrays front to back. The L2-prefetching forms of the
// double-buffered step kernel (fp32 gradient, N <= 6) measured 1-2% faster
// with adjacent chunks; every other form 1-4% faster round robin.
template <int W>
struct ChunkMap {
  int64_t nchunk, pass, full;
  __device__ explicit ChunkMap(int64_t nvec)
      : nchunk((nvec + 31) / 32), pass(static_cast<int64_t>(gridDim.x) * W), full(nchunk / pass) {}
  // The block's j-th chunk; increasing in j, so once a value reaches nchunk
  // every later one does too.
  template <bool ADJACENT>
  __device__ __forceinline__ int64_t chunk(unsigned j) const {
    if constexpr (ADJACENT) {
      const int64_t s = j / W;
      if (s < full) return s * pass + static_cast<int64_t>(blockIdx.x) * W + j % W;
      return full * pass + (static_cast<int64_t>(j) - full * W) * gridDim.x + blockIdx.x;
    } else {
      return static_cast<int64_t>(j) * gridDim.x + blockIdx.x;
    }
  }
  // The calling warp's next chunk from the block's counter (all lanes call;
  // >= nchunk once the block's chunks are all taken).
  template <bool ADJACENT>
  __device__ __forceinline__ int64_t take(unsigned* counter, int lane) const {
    unsigned j = 0;
    if (lane == 0) j = atomicAdd(counter, 1u);
    return chunk<ADJACENT>(__shfl_sync(0xFFFFFFFFu, j, 0));
  }
};

// Programmatic dependent launch (sm_90 and later). A kernel launched with the
// programmatic stream serialization attribute (launch_dependent below) may be
// scheduled before the kernel ahead of it in the stream has finished, once
// every block of that kernel has called pdl_trigger() or exited. pdl_wait()
// then holds it until that kernel's grid has completed and its writes are
// visible -- the hardware's kernel boundary, moved into the kernel; without
// the attribute it returns at once. Only the launch latency is overlapped:
// nothing before pdl_wait() may touch memory the previous kernel writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host helpers shared by the entry points (defined in ss_util.cu).

// Byte range of one argument array; `out` marks arrays the call writes.
struct Range {
  uintptr_t lo, hi;
  bool out;
};

// Text of the last CUDA error seen by this thread (ss_last_cuda_error).
extern thread_local char g_cuda_err[256];
// Records `e` as the thread's last CUDA error and returns SS_ERR_CUDA.
ss_status cuda_fail(cudaError_t e);
// True when some output byte range overlaps any other range (inputs may overlap inputs).
bool any_output_overlap(std::vector<Range>& rs);
Range rng(const void* p, int64_t bytes, bool out);
// Smallest h in [0, 8) with every 16-bit pointer at a 16-byte boundary after h
// elements and every fp32 pointer likewise; -1 when none exists.
int common_phase(const std::vector<uintptr_t>& p16, const std::vector<uintptr_t>& p32);
int sm_count();
// Resident blocks per SM of a kernel launched with `threads` per block (cached per device,
// kernel and block size).
int blocks_per_sm(const void* fn, int threads = kThreads);
// Persistent grid for `work_items` thread-items: at most SM count x resident blocks.
unsigned grid_for(const void* fn, int64_t work_items, int threads = kThreads);
// Checks the rank gradient pointers (non-null, 2-byte aligned, 16-bit dtype) and
// appends their byte ranges and addresses.
ss_status check_ranks(const void* const* rank_grads, int32_t n_ranks, ss_dtype gdtype, int64_t n,
                      std::vector<Range>& ranges, std::vector<uintptr_t>& p16);

inline bool is16(ss_dtype d) { return d == SS_BF16 || d == SS_FP16; }


// Launches fn<<<grid, block, smem, stream>>>(args...) as a programmatic
// dependent of the previous kernel in the stream (see pdl_wait). Every kernel
// of the library starts with pdl_wait() and pdl_trigger(). The next kernel can
// launch only once every block of this grid has triggered, i.e. has started,
// so its waiting blocks never hold resources this grid's blocks still need;
// grids are sized to one wave (all but a copy of more shards than resident
// blocks), which lets the next launch overlap this grid's last blocks.
template <typename... Params, typename... Args>
ss_status launch_dependent(void (*fn)(Params...), dim3 grid, dim3 block, size_t smem, void* stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
#ifdef SS_NO_PDL
  cfg.numAttrs = 0;
#else
  cfg.numAttrs = 1;
#endif
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, static_cast<Params>(args)...);
  return e == cudaSuccess ? SS_OK : cuda_fail(e);
}

template <typename Args, typename Fn>
ss_status launch(Fn* fn, unsigned grid, const Args& args, void* stream, int threads = kThreads) {
  return launch_dependent(fn, dim3(grid), dim3(static_cast<unsigned>(threads)), 0, stream, args);
}

}  // namespace ss
