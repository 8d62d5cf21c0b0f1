// ss_step_shift.cu -- the fused shard step (ss_adam_step) when 16-bit arrays are
// off the fp32 state's 16-byte phase: gradient views at boundaries that are not
// multiples of 8 elements, or param16 inside a flat buffer at such a boundary
// (and, at phase 0, aligned gradients of 4, 5 and 9-16 ranks, where the
// double-buffered form here measured fastest). Three kernel forms share the
// per-element arithmetic of ss_math.cuh: a warp-cooperative double-buffered one
// for up to 16 ranks at one phase, or up to 12 with each rank shifted by its own
// phase; a warp-cooperative single-buffered one for more ranks at one phase; and
// a per-thread one for more ranks at mixed phases (or an fp32 gradient with
// param16 off phase). Each gradient byte is loaded once in the
// warp-cooperative forms.
#include "ss_step.cuh"

namespace ss {
namespace {

// ------------------------------------------------------------------ fused AdamW step, 16-bit arrays off the state's phase
//
// When the fp32 arrays share a 16-byte phase but some 16-bit arrays (rank
// gradients, param16) do not -- shard views at boundaries that are not
// multiples of 8 elements, or param16 inside a flat buffer at such a
// boundary -- groups still start where the fp32 arrays are 16-byte aligned.
// Every 16-bit gradient array is read as the two aligned 16-byte chunks that
// hold the group (all loads issued first) and funnel-shifted to its phase;
// param16 is stored in 4- or 2-byte pieces when it is off phase. The body is
// groups 1 .. nvec-2, so every chunk read lies inside its array; the first
// and last groups and the head/tail elements are done one by one.


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

// The per-thread form: at least 2 blocks of 256 threads per SM (128 registers). With the
// state requested before the gradients it needs 138 and the occupancy halves: measured on
// GB300 at 2^26 elements, 9-64 ranks at mixed phases 0.46-0.52 of the copy peak at one block
// per SM against 0.74-0.82 at two.
#ifndef SS_SHIFT_THREAD_BLOCKS
#define SS_SHIFT_THREAD_BLOCKS 2
#endif
template <int GT, int PT, bool FROM_G32, bool WRITE_P16, int MAXR>
__global__ void __launch_bounds__(kThreads, SS_SHIFT_THREAD_BLOCKS) adam_shift_kernel(const __grid_constant__ ShiftArgs<MAXR> x) {
  pdl_wait();
  pdl_trigger();
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
    // the group's state is requested first, so it arrives with the gradients (no output
    // overlaps an input, so nothing stored below changes it)
    float p[8], m[8], v[8];
    ld8f(a.master + e, p);
    ld8f(a.m + e, m);
    ld8f(a.v + e, v);
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

// Warp-cooperative forms of the shifted-load step for 16-bit rank gradients
// that all sit at the same 16-byte phase (views at one offset into
// identically allocated buffers, the usual case). A warp takes runs of 31
// consecutive groups of the vector body: lane j loads, per rank, the aligned
// 16-byte chunk under the start of group j of the run (lane 31 the chunk under
// the start of the group after the run) and sums the ranks' chunks element by
// element in rank order -- the same fp32 sum each element gets anywhere else,
// only held in a neighbouring register -- then each lane moves its group's
// sums into place, taking the ones past its own chunk from the upper lane by
// shuffle. Each gradient byte is loaded once; lanes 0..30 load and update
// their group's state. Every chunk lies under a group in [1, nvec - 1], so
// inside its array; the groups outside the body [1, nvec - 1) and the
// head/tail elements are done one by one. Runs are taken from a per-block
// counter in shared memory and owned round robin, as the aligned kernels take
// their chunks.
//
// Up to 8 ranks: register double-buffered (the loads of the warp's next run
// are issued before the current run's update). The double-float update and
// two runs' loads need more than 128 registers from 4 ranks on, so the block
// shape depends on the rank count: up to 3 ranks one 512-thread block per SM
// (128 registers) with an L2 prefetch of the run after next, from 4 ranks one
// 384-thread block per SM (up to 170 registers) without it. Measured on GB300
// at 2^26 elements with the gradients one element off phase: 8 ranks 0.82 of
// the copy peak in the 128-register form (it spilled), 0.96 in this one;
// 1-8 ranks 0.92-1.01. The prefetch gained 1-3% at 2-3 ranks and cost 3-6%
// at 4-6.
// More ranks: single-buffered, each run's state requested with the first
// batch of 8 rank chunks, all loads of a batch before its adds (16 and 32
// ranks 0.99 of the copy peak; 9-12 ranks only 0.77-0.82 -- one batch of 8
// and a short second one, where the update's issue time is no longer hidden
// behind memory).

#ifndef SS_SHIFT_NARROW_RANKS
#define SS_SHIFT_NARROW_RANKS 3  // up to this many ranks: one 512-thread block per SM (128 registers)
#endif
#ifndef SS_SHIFT_WIDE_THREADS
#define SS_SHIFT_WIDE_THREADS 384  // above: one 384-thread block per SM (up to 170 registers)
#endif
#ifndef SS_SHIFT_WIDE_BLOCKS
#define SS_SHIFT_WIDE_BLOCKS 1
#endif
// Rank counts up to which the warp-cooperative kernels also prefetch a later
// run's bytes into L2 (as the aligned kernels do for few ranks).
#ifndef SS_SHIFT_PF_RANKS
#define SS_SHIFT_PF_RANKS 3
#endif
#ifndef SS_SHIFT_VEC_PF_RANKS
#define SS_SHIFT_VEC_PF_RANKS 13
#endif
// Above 8 ranks (one phase) two runs' chunks need up to ~215 registers: one 256-thread
// block per SM (up to 255 registers). Measured on GB300 at 2^26 elements, 9-16 ranks one
// element off phase: 0.99-1.05 of the copy peak, against 0.75-0.98 single-buffered.
#ifndef SS_SHIFT_PIPE_MAX_RANKS
#define SS_SHIFT_PIPE_MAX_RANKS 16
#endif
// Up to this many ranks at mixed phases take the double-buffered warp-cooperative kernel,
// each rank's packed chunk shifted by its own phase. Measured on GB300 at 2^26 elements, rank
// r's view (r % 7) + 1 elements off: 9-11 ranks 0.85-0.86 of the copy peak against 0.74-0.75
// per-thread, 12 ranks 0.78 against 0.77, 13-16 ranks 0.66-0.78 against 0.78-0.81.
#ifndef SS_SHIFT_MIXED_MAX_RANKS
#define SS_SHIFT_MIXED_MAX_RANKS 12
#endif
#ifndef SS_SHIFT_MIXED_VEC
#define SS_SHIFT_MIXED_VEC 0
#endif
template <int NR>
struct ShiftShape {
  static constexpr bool kNarrow = NR <= SS_SHIFT_NARROW_RANKS;
  static constexpr bool kMany = NR > 8;
  static constexpr int kThreadsPerBlock = kNarrow ? kChunkThreads : (kMany ? 256 : SS_SHIFT_WIDE_THREADS);
  static constexpr int kBlocksPerSm = kNarrow ? kChunkBlocksPerSm : (kMany ? 1 : SS_SHIFT_WIDE_BLOCKS);
};

// One run's loads of one lane: the ranks' aligned 16-byte gradient chunks and
// its group's master, m and v (two float4 each).
template <int NR>
struct ShiftGroup {
  uint4 r[NR];
  float4 s[6];
};

template <int GT, int NR, bool MIXED, int MAXR>
__device__ __forceinline__ void shift_pipe_load(const ShiftArgs<MAXR>& x, int64_t run, int lane, int64_t nvec,
                                                ShiftGroup<NR>& G) {
  const StepArgs<MAXR>& a = x.s;
  int64_t gi = 1 + run * kRun + lane;  // the group whose start this lane's chunks cover
  gi = gi < nvec - 1 ? gi : nvec - 1;  // past the body: a chunk inside the array, unused
  const int64_t e = a.head + gi * kGroup;
#pragma unroll
  for (int r = 0; r < NR; ++r)
    G.r[r] = __ldcs(reinterpret_cast<const uint4*>(
        reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[r]) + e) - x.rphase[MIXED ? r : 0]));
  if (lane < kRun) {
    const int64_t gb = gi < nvec - 2 ? gi : nvec - 2;  // the state of a body group
    const int64_t es = a.head + gb * kGroup;
    G.s[0] = __ldcs(reinterpret_cast<const float4*>(a.master + es));
    G.s[1] = __ldcs(reinterpret_cast<const float4*>(a.master + es) + 1);
    G.s[2] = __ldcs(reinterpret_cast<const float4*>(a.m + es));
    G.s[3] = __ldcs(reinterpret_cast<const float4*>(a.m + es) + 1);
    G.s[4] = __ldcs(reinterpret_cast<const float4*>(a.v + es));
    G.s[5] = __ldcs(reinterpret_cast<const float4*>(a.v + es) + 1);
  }
}

// L2 prefetch of run `run`'s bytes, one bulk prefetch per array (lane r < n_ranks
// takes rank r's gradient chunks, the next three lanes master, m and v): the
// same chunks and state the run's loads read, so every range lies inside its
// array, starts on a 16-byte boundary and is a multiple of 16 bytes. Hints only.
template <int MAXR>
__device__ __forceinline__ void shift_prefetch(const ShiftArgs<MAXR>& x, int64_t run, int lane, int n_ranks,
                                               int64_t nvec) {
  const StepArgs<MAXR>& a = x.s;
  if (lane >= n_ranks + 3) return;
  const int64_t g0 = 1 + run * kRun;
  if (lane < n_ranks) {
    const int64_t gl = g0 + kRun < nvec - 1 ? g0 + kRun : nvec - 1;  // the chunk after the run, if any
    prefetch_l2(reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[lane]) + a.head + g0 * kGroup) -
                    x.rphase[lane],
                static_cast<uint32_t>((gl - g0 + 1) * 16));
  } else {
    const int64_t gb = g0 + kRun - 1 < nvec - 2 ? g0 + kRun - 1 : nvec - 2;  // the run's last body group
    const int k = lane - n_ranks;
    prefetch_l2((k == 0 ? a.master : (k == 1 ? a.m : a.v)) + a.head + g0 * kGroup,
                static_cast<uint32_t>((gb - g0 + 1) * 32));
  }
}

// The update of one body group from its (shifted) gradient sums and its state;
// the options and the param16 store at its phase, as in the aligned kernels.
template <int PT, bool WRITE_P16, int MAXR>
__device__ __forceinline__ void shift_update(const ShiftArgs<MAXR>& x, int64_t e, float (&g)[8], float (&p)[8],
                                             float (&m)[8], float (&v)[8], float gs, bool& bad) {
  const StepArgs<MAXR>& a = x.s;
  if (a.post_scale != 1.0f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = g[j] * a.post_scale;
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
#pragma unroll
  for (int j = 0; j < 8; ++j) adamw_elem(a.k, g[j], p[j], m[j], v[j]);
  st8f(a.master + e, p);
  st8f(a.m + e, m);
  st8f(a.v + e, v);
  if constexpr (WRITE_P16) st16_at_phase(static_cast<uint16_t*>(a.p16) + e, narrow8<PT>(p), x.pphase);
}

// Everything outside the vector body [1, nvec - 1), one element per thread (< 31 elements).
template <int GT, int PT, bool WRITE_P16, int MAXR>
__device__ __forceinline__ void shift_edges(const ShiftArgs<MAXR>& x, int64_t nvec, float gs, bool& bad) {
  const StepArgs<MAXR>& a = x.s;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t lo_end = a.head + kGroup, hi_start = a.head + (nvec - 1) * kGroup;
  const int64_t n_edge = lo_end + (a.n - hi_start);
  if (tid < n_edge) step1<GT, PT, false, WRITE_P16>(a, tid < lo_end ? tid : hi_start + (tid - lo_end), gs, bad);
}

template <int GT, int PT, bool WRITE_P16, bool MIXED, int MAXR, int NR>
__global__ void __launch_bounds__(ShiftShape<NR>::kThreadsPerBlock, ShiftShape<NR>::kBlocksPerSm)
    adam_shift_pipe_kernel(const __grid_constant__ ShiftArgs<MAXR> x) {
  __shared__ unsigned next_run;
  if (threadIdx.x == 0) next_run = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const StepArgs<MAXR>& a = x.s;
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t nvec = (a.n - a.head) / kGroup;  // >= 3 on this path
  const int64_t runs = (nvec - 2 + kRun - 1) / kRun;
  const int sh = x.rphase[0] >> 1;                // the groups' element offset into their first chunk
  const int lane = threadIdx.x & 31;
  const ChunkMap<ShiftShape<NR>::kThreadsPerBlock / 32> map(runs * 32);  // one "chunk" per run
  constexpr bool kPrefetch = NR <= SS_SHIFT_PF_RANKS;
  bool bad = false;
  ShiftGroup<NR> cur, nxt;
  // The warp's runs in the order it takes them: `run` (in cur), the next one (loaded into
  // nxt during run's update) and, with the L2 prefetch, the one after (asked of the L2).
  // Every run taken is processed; the counter is read by whole warps.
  int64_t run = map.template take<false>(&next_run, lane);
  int64_t rpf = (kPrefetch && run < runs) ? map.template take<false>(&next_run, lane) : runs;
  if (run < runs) shift_pipe_load<GT, NR, MIXED>(x, run, lane, nvec, cur);
  while (run < runs) {  // warp-uniform
    int64_t rload;
    if constexpr (kPrefetch) {
      rload = rpf;
      rpf = rload < runs ? map.template take<false>(&next_run, lane) : runs;
    } else {
      rload = map.template take<false>(&next_run, lane);
    }
    if (rload < runs) shift_pipe_load<GT, NR, MIXED>(x, rload, lane, nvec, nxt);
    if constexpr (kPrefetch) {
      if (rpf < runs) shift_prefetch(x, rpf, lane, NR, nvec);
    }
    float g[8];
    if constexpr (MIXED) {
      // each rank's packed values moved into place by its own phase, then added in rank order
      widen8<GT>(shift_chunk(cur.r[0], x.rphase[0] >> 1), g);
#pragma unroll
      for (int r = 1; r < NR; ++r) add8<GT>(shift_chunk(cur.r[r], x.rphase[r] >> 1), g);
    } else {
      widen8<GT>(cur.r[0], g);
#pragma unroll
      for (int r = 1; r < NR; ++r) add8<GT>(cur.r[r], g);
      shift_down8(g, sh);
    }
    const int64_t gi = 1 + run * kRun + lane;
    if (lane < kRun && gi < nvec - 1) {
      float p[8] = {cur.s[0].x, cur.s[0].y, cur.s[0].z, cur.s[0].w, cur.s[1].x, cur.s[1].y, cur.s[1].z, cur.s[1].w};
      float m[8] = {cur.s[2].x, cur.s[2].y, cur.s[2].z, cur.s[2].w, cur.s[3].x, cur.s[3].y, cur.s[3].z, cur.s[3].w};
      float v[8] = {cur.s[4].x, cur.s[4].y, cur.s[4].z, cur.s[4].w, cur.s[5].x, cur.s[5].y, cur.s[5].z, cur.s[5].w};
      shift_update<PT, WRITE_P16>(x, a.head + gi * kGroup, g, p, m, v, gs, bad);
    }
    cur = nxt;
    run = rload;
  }
  shift_edges<GT, PT, WRITE_P16>(x, nvec, gs, bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && lane == 0) *a.nonfinite = 1;
  }
}

#ifndef SS_SHIFT_VEC_BATCH
#define SS_SHIFT_VEC_BATCH 8  // rank chunks loaded per batch in the single-buffered form
#endif
#ifndef SS_SHIFT_VEC_THREADS
#define SS_SHIFT_VEC_THREADS 512  // one block per SM: up to 128 registers
#endif
constexpr int kShiftVecBatch = SS_SHIFT_VEC_BATCH;
constexpr int kShiftVecThreads = SS_SHIFT_VEC_THREADS;

template <int GT, int PT, bool WRITE_P16, bool MIXED, int MAXR>
__global__ void __launch_bounds__(kShiftVecThreads, 1)
    adam_shift_vec_kernel(const __grid_constant__ ShiftArgs<MAXR> x) {
  __shared__ unsigned next_run;
  if (threadIdx.x == 0) next_run = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const StepArgs<MAXR>& a = x.s;
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t nvec = (a.n - a.head) / kGroup;  // >= 3 on this path
  const int64_t runs = (nvec - 2 + kRun - 1) / kRun;
  const int sh = x.rphase[0] >> 1;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kShiftVecThreads / 32> map(runs * 32);
  const bool prefetch = a.n_ranks <= SS_SHIFT_VEC_PF_RANKS;
  bool bad = false;
  int64_t run = map.template take<false>(&next_run, lane);
  while (run < runs) {  // warp-uniform
    const int64_t rn = map.template take<false>(&next_run, lane);
    if (prefetch && rn < runs) shift_prefetch(x, rn, lane, a.n_ranks, nvec);
    const int64_t gi = 1 + run * kRun + lane;
    const int64_t gl = gi < nvec - 1 ? gi : nvec - 1;  // past the body: a chunk inside the array, unused
    const int64_t el = a.head + gl * kGroup;
    const bool body = lane < kRun && gi < nvec - 1;
    const int64_t e = a.head + gi * kGroup;
    // the group's state is requested with the first batch of rank chunks, so both arrive
    // in one round trip; the ranks' chunks come in batches, all loads of a batch first
    float4 s4[6];
    float g[8];
    for (int r0 = 0; r0 < a.n_ranks; r0 += kShiftVecBatch) {
      uint4 w[kShiftVecBatch];
#pragma unroll
      for (int j = 0; j < kShiftVecBatch; ++j)
        if (r0 + j < a.n_ranks)
          w[j] = __ldcs(reinterpret_cast<const uint4*>(
              reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[r0 + j]) + el) -
              x.rphase[MIXED ? r0 + j : 0]));
      if (r0 == 0 && body) {
        s4[0] = __ldcs(reinterpret_cast<const float4*>(a.master + e));
        s4[1] = __ldcs(reinterpret_cast<const float4*>(a.master + e) + 1);
        s4[2] = __ldcs(reinterpret_cast<const float4*>(a.m + e));
        s4[3] = __ldcs(reinterpret_cast<const float4*>(a.m + e) + 1);
        s4[4] = __ldcs(reinterpret_cast<const float4*>(a.v + e));
        s4[5] = __ldcs(reinterpret_cast<const float4*>(a.v + e) + 1);
      }
#pragma unroll
      for (int j = 0; j < kShiftVecBatch; ++j) {
        if (r0 + j < a.n_ranks) {
          // at mixed phases each rank's packed values are moved into place before they are added
          const uint4 c = MIXED ? shift_chunk(w[j], x.rphase[r0 + j] >> 1) : w[j];
          if (r0 + j == 0) widen8<GT>(c, g);
          else add8<GT>(c, g);
        }
      }
    }
    if constexpr (!MIXED) shift_down8(g, sh);
    if (body) {
      float p[8] = {s4[0].x, s4[0].y, s4[0].z, s4[0].w, s4[1].x, s4[1].y, s4[1].z, s4[1].w};
      float m[8] = {s4[2].x, s4[2].y, s4[2].z, s4[2].w, s4[3].x, s4[3].y, s4[3].z, s4[3].w};
      float v[8] = {s4[4].x, s4[4].y, s4[4].z, s4[4].w, s4[5].x, s4[5].y, s4[5].z, s4[5].w};
      shift_update<PT, WRITE_P16>(x, e, g, p, m, v, gs, bad);
    }
    run = rn;
  }
  shift_edges<GT, PT, WRITE_P16>(x, nvec, gs, bad);
  if (a.nonfinite) {
    const unsigned any = __ballot_sync(0xFFFFFFFFu, bad);
    if (any && lane == 0) *a.nonfinite = 1;
  }
}

// ---- dispatch

template <int G, int P, bool W, bool MIXED, int MAXR, int NR>
ss_status launch_shift_pipe_n(const ShiftArgs<MAXR>& x, void* stream) {
  auto* fn = adam_shift_pipe_kernel<G, P, W, MIXED, MAXR, NR>;
  constexpr int threads = ShiftShape<NR>::kThreadsPerBlock;
  const int64_t runs = ((x.s.n - x.s.head) / kGroup - 2 + kRun - 1) / kRun;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), runs * 32, threads), x, stream, threads);
}

template <int G, int P, bool W, bool MIXED, int MAXR>
ss_status launch_shift_vec(const ShiftArgs<MAXR>& x, void* stream) {
  auto* fn = adam_shift_vec_kernel<G, P, W, MIXED, MAXR>;
  const int64_t runs = ((x.s.n - x.s.head) / kGroup - 2 + kRun - 1) / kRun;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), runs * 32, kShiftVecThreads), x, stream,
                kShiftVecThreads);
}

template <int G, int P, bool W, bool MIXED, int MAXR>
ss_status launch_shift_warp(const ShiftArgs<MAXR>& x, void* stream) {
  if constexpr (MAXR == kSmallRanks) {
    constexpr int kMax = MIXED ? SS_SHIFT_MIXED_MAX_RANKS : SS_SHIFT_PIPE_MAX_RANKS;
#define SS_SHIFT_PIPE_CASE(R) \
  case R:                     \
    if constexpr (R <= kMax) return launch_shift_pipe_n<G, P, W, MIXED, MAXR, R>(x, stream); \
    break;
    switch (x.s.n_ranks) {
      SS_SHIFT_PIPE_CASE(1) SS_SHIFT_PIPE_CASE(2) SS_SHIFT_PIPE_CASE(3) SS_SHIFT_PIPE_CASE(4)
      SS_SHIFT_PIPE_CASE(5) SS_SHIFT_PIPE_CASE(6) SS_SHIFT_PIPE_CASE(7) SS_SHIFT_PIPE_CASE(8)
      SS_SHIFT_PIPE_CASE(9) SS_SHIFT_PIPE_CASE(10) SS_SHIFT_PIPE_CASE(11) SS_SHIFT_PIPE_CASE(12)
      SS_SHIFT_PIPE_CASE(13) SS_SHIFT_PIPE_CASE(14) SS_SHIFT_PIPE_CASE(15) SS_SHIFT_PIPE_CASE(16)
      default: break;
    }
#undef SS_SHIFT_PIPE_CASE
  }
  if constexpr (MIXED && !SS_SHIFT_MIXED_VEC) return SS_ERR_INVALID_ARG;  // not reached: see launch_shift
  else return launch_shift_vec<G, P, W, MIXED, MAXR>(x, stream);
}

template <int G, int P, bool F, bool W, int MAXR>
ss_status launch_shift(const StepArgs<MAXR>& a, const uint8_t* rphase, uint8_t pphase, void* stream) {
  ShiftArgs<MAXR> x;
  std::memset(&x, 0, sizeof x);
  x.s = a;
  for (int32_t r = 0; r < a.n_ranks; ++r) x.rphase[r] = rphase[r];
  x.pphase = pphase;
  // 16-bit gradients at one phase: the warp-cooperative forms (double-buffered up to 16
  // ranks, single-buffered above), summing first and shifting once. At mixed phases, up
  // to 12 ranks: the double-buffered form shifting each rank's packed chunk by its own
  // phase (on GB300 at 2^26 elements 1-8 ranks 0.92-0.98 of the copy peak against
  // 0.71-0.81 per-thread); more ranks: the per-thread form, which the warp-cooperative
  // single-buffered form with per-rank shifts did not beat there (13-64 ranks 0.75-0.83
  // against 0.78-0.82)
  if constexpr (!F) {
    bool same = true;
    for (int32_t r = 1; r < a.n_ranks; ++r) same = same && rphase[r] == rphase[0];
    if (same) return launch_shift_warp<G, P, W, false, MAXR>(x, stream);
    if constexpr (MAXR == kSmallRanks) {
      if (a.n_ranks <= SS_SHIFT_MIXED_MAX_RANKS) return launch_shift_warp<G, P, W, true, MAXR>(x, stream);
    }
#if SS_SHIFT_MIXED_VEC
    return launch_shift_vec<G, P, W, true, MAXR>(x, stream);
#endif
  }
  // more ranks at mixed phases, or an fp32 gradient with param16 off phase: the per-thread form
  auto* fn = adam_shift_kernel<G, P, F, W, MAXR>;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup), x, stream);
}

}  // namespace

template <int MAXR>
ss_status shift_step(const StepArgs<MAXR>& a, ss_dtype gt, ss_dtype pt, bool from_g32, bool p16,
                     const uint8_t* rphase, uint8_t pphase, void* stream) {
  // An fp32 gradient (gt is then the placeholder SS_BF16) travels with the small rank table.
#define SS_SHIFT_CASE(G, P, F, W) \
  if (gt == G && pt == P && from_g32 == F && p16 == W) return launch_shift<G, P, F, W, MAXR>(a, rphase, pphase, stream);
#define SS_SHIFT_P(G, P) SS_SHIFT_CASE(G, P, false, true) SS_SHIFT_CASE(G, P, false, false)
  SS_SHIFT_P(SS_BF16, SS_BF16)
  SS_SHIFT_P(SS_BF16, SS_FP16)
  SS_SHIFT_P(SS_FP16, SS_BF16)
  SS_SHIFT_P(SS_FP16, SS_FP16)
  if constexpr (MAXR == kSmallRanks) {
    SS_SHIFT_CASE(SS_BF16, SS_BF16, true, true)
    SS_SHIFT_CASE(SS_BF16, SS_BF16, true, false)
    SS_SHIFT_CASE(SS_BF16, SS_FP16, true, true)
    SS_SHIFT_CASE(SS_BF16, SS_FP16, true, false)
  }
#undef SS_SHIFT_P
#undef SS_SHIFT_CASE
  return SS_ERR_DTYPE;
}

template ss_status shift_step<kSmallRanks>(const StepArgs<kSmallRanks>&, ss_dtype, ss_dtype, bool, bool,
                                           const uint8_t*, uint8_t, void*);
template ss_status shift_step<kLargeRanks>(const StepArgs<kLargeRanks>&, ss_dtype, ss_dtype, bool, bool,
                                           const uint8_t*, uint8_t, void*);

}  // namespace ss
