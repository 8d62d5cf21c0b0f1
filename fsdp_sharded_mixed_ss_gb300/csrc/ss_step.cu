// ss_step.cu -- the fused shard step (ss_adam_step): rank-ordered fp32 reduce of
// the ranks' gradient shards, AdamW on the fp32 master and moments, and the
// 16-bit parameter cast, in one pass over HBM. This file holds the entry point
// and the kernel forms for arrays that share the fp32 state's 16-byte phase:
// register double-buffered (up to 8 ranks or an fp32 gradient),
// single-buffered vector (more ranks) and element-wise (no common phase). The
// forms for 16-bit arrays off that phase are in ss_step_shift.cu. All share
// the per-element arithmetic of ss_math.cuh.
#include "ss_step.cuh"

namespace ss {
namespace {

// Rank counts up to which the single-buffered kernel also prefetches its
// warp's next groups into L2 (measured on GB300 at 2^26 elements: +3-12% for
// N = 5-13, none at 14, -3% at 15, -6% at 16).
#ifndef SS_VEC_PF_RANKS
#define SS_VEC_PF_RANKS 13
#endif
constexpr int kVecPrefetchRanks = SS_VEC_PF_RANKS;

template <int GT, int PT, bool FROM_G32, bool WRITE_P16, int MAXR>
__global__ void __launch_bounds__(kChunkThreads, kChunkBlocksPerSm) adam_vec_kernel(const __grid_constant__ StepArgs<MAXR> a) {
  __shared__ unsigned next_chunk;
  if (threadIdx.x == 0) next_chunk = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const ChunkMap<kChunkWarps> map(nvec);
  bool bad = false;
  // moderate rank counts: the warp also asks the L2 for its next chunk, one bulk prefetch per
  // array (lane k takes array k), as the double-buffered kernel does for few ranks
  const int npf = (!FROM_G32 && a.n_ranks <= kVecPrefetchRanks) ? a.n_ranks + 3 : 0;
  int64_t c = map.take<false>(&next_chunk, lane);
  while (c < map.nchunk) {
    const int64_t cn = map.take<false>(&next_chunk, lane);
    if (npf && cn < map.nchunk && lane < npf) {
      const int64_t b = cn * 32;
      const int64_t cnt = nvec - b < 32 ? nvec - b : 32;
      const int64_t eb = a.head + b * kGroup;
      if (lane < a.n_ranks) {
        prefetch_l2(static_cast<const uint16_t*>(a.ranks.p[lane]) + eb, static_cast<uint32_t>(cnt * 16));
      } else {
        const int k = lane - a.n_ranks;
        prefetch_l2((k == 0 ? a.master : (k == 1 ? a.m : a.v)) + eb, static_cast<uint32_t>(cnt * 32));
      }
    }
    const int64_t gi = c * 32 + lane;
    if (gi < nvec) {
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
    c = cn;
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

// Register double-buffered form for small rank counts: the loads of a warp's
// next chunk are issued before the update of its current one, so each thread
// keeps two groups of bytes in flight (for small N, where one group alone is
// too few bytes to cover HBM latency at the residency the update's registers
// allow). NR is the rank count; with F the gradient is the fp32 array g32,
// held as NR = 2 raw 16-byte chunks.
// The rank counts (bit N set: N ranks) that take this form; the others take
// the single-buffered kernel, which with its L2 prefetch measured faster on
// GB300 for 5 and 6 ranks at 2^26 elements.
#ifndef SS_PIPE_RANK_MASK
#define SS_PIPE_RANK_MASK ((1u << 1) | (1u << 2) | (1u << 3) | (1u << 4) | (1u << 7) | (1u << 8))
#endif
constexpr unsigned kPipeRankMask = SS_PIPE_RANK_MASK;
constexpr bool pipe_ranks(int n) { return n >= 1 && n <= 8 && ((kPipeRankMask >> n) & 1u) != 0; }
// Rank counts up to which the kernel also prefetches into L2 (measured on
// GB300 at 2^26 elements: +2-9% for an fp32 gradient and N <= 6, -5% at N = 8,
// where a group's own loads already keep enough bytes in flight).
#ifndef SS_PIPE_PF_RANKS
#define SS_PIPE_PF_RANKS 6
#endif
constexpr int kPipePrefetchRanks = SS_PIPE_PF_RANKS;
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
__global__ void __launch_bounds__(kChunkThreads, kChunkBlocksPerSm) adam_pipe_kernel(const __grid_constant__ StepArgs<MAXR> a) {
  __shared__ unsigned next_chunk;
  if (threadIdx.x == 0) next_chunk = 0;
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (a.dev_skip != nullptr && *a.dev_skip != 0) return;
  const float gs = a.dev_scale ? *a.dev_scale : 1.0f;
  const int64_t nvec = (a.n - a.head) / kGroup;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  constexpr bool kPrefetch = F || NR <= kPipePrefetchRanks;
  const ChunkMap<kChunkWarps> map(nvec);
  const int64_t nchunk = map.nchunk;
  auto take = [&]() -> int64_t { return map.take<kPrefetch>(&next_chunk, lane); };
  bool bad = false;
  PipeGroup<NR> cur, nxt;
  int64_t c = take();
  int64_t cn = c < nchunk ? take() : nchunk;
  if (c < nchunk && c * 32 + lane < nvec) pipe_load<GT, NR, F>(a, c * 32 + lane, cur);
  while (c < nchunk) {
    const int64_t cnn = cn < nchunk ? take() : nchunk;
    if (cn < nchunk && cn * 32 + lane < nvec) pipe_load<GT, NR, F>(a, cn * 32 + lane, nxt);
    if constexpr (kPrefetch) {
      // L2 prefetch of the warp's chunk after next, one bulk prefetch per array (lane k takes
      // array k): more bytes in flight without registers, for groups whose own loads are few.
      // Hints only; every range lies inside its array.
      constexpr int kArrays = (F ? 1 : NR) + 3;
      const int64_t b = cnn * 32;
      if (cnn < nchunk && lane < kArrays) {
        const int64_t cnt = nvec - b < 32 ? nvec - b : 32;
        const int64_t e = a.head + b * kGroup;
        const char* base;
        int64_t bytes = cnt * 32;  // 8 fp32 per group
        if (lane < kArrays - 3) {
          if constexpr (F) {
            base = reinterpret_cast<const char*>(a.g32 + e);
          } else {
            base = reinterpret_cast<const char*>(static_cast<const uint16_t*>(a.ranks.p[lane]) + e);
            bytes = cnt * 16;  // 8 16-bit per group
          }
        } else {
          const int k = lane - (kArrays - 3);
          base = reinterpret_cast<const char*>((k == 0 ? a.master : (k == 1 ? a.m : a.v)) + e);
        }
        prefetch_l2(base, static_cast<uint32_t>(bytes));
      }
    }
    const int64_t gi = c * 32 + lane;
    if (gi < nvec) {
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
    }
    cur = nxt;
    c = cn;
    cn = cnn;
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
  pdl_wait();
  pdl_trigger();
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

// The rank counts (bit N set: N ranks) whose aligned steps take the warp-cooperative kernel.
#ifndef SS_WARP_COOP_RANK_MASK
#define SS_WARP_COOP_RANK_MASK ((1u << 4) | (1u << 5) | (0xFFu << 9))
#endif
constexpr unsigned kWarpCoopRankMask = SS_WARP_COOP_RANK_MASK;

template <int G, int P, bool W, int MAXR, int NR, bool F = false>
ss_status launch_pipe_n(const StepArgs<MAXR>& a, void* stream) {
  auto* fn = adam_pipe_kernel<G, P, F, W, MAXR, NR>;
  return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup, kChunkThreads), a, stream,
                kChunkThreads);
}

template <int G, int P, bool W, int MAXR>
ss_status launch_pipe(const StepArgs<MAXR>& a, void* stream) {
#define SS_PIPE_CASE(R)                                                     \
  case R:                                                                   \
    if constexpr (pipe_ranks(R)) return launch_pipe_n<G, P, W, MAXR, R>(a, stream); \
    else return SS_ERR_INVALID_ARG;
  switch (a.n_ranks) {
    SS_PIPE_CASE(1) SS_PIPE_CASE(2) SS_PIPE_CASE(3) SS_PIPE_CASE(4)
    SS_PIPE_CASE(5) SS_PIPE_CASE(6) SS_PIPE_CASE(7) SS_PIPE_CASE(8)
    default: return SS_ERR_INVALID_ARG;
  }
#undef SS_PIPE_CASE
}

template <int MAXR>
ss_status run_adam(const StepArgs<MAXR>& a, Path path, bool from_g32, bool p16, ss_dtype gt, ss_dtype pt,
                   const uint8_t* rphase, uint8_t pphase, void* stream) {
  if (path == Path::kShift) return shift_step<MAXR>(a, gt, pt, from_g32, p16, rphase, pphase, stream);
  // Only reachable forms are instantiated: an fp32 gradient (gt is then the
  // placeholder SS_BF16) always travels with the small rank table and takes the
  // double-buffered, shifted or element-wise form; the double-buffered form is
  // chosen only for at most 8 ranks, so only with the small table.
#define SS_ADAM_CASE(G, P, F, W)                                                          \
  if (gt == G && pt == P && from_g32 == F && p16 == W) {                                  \
    if (path == Path::kPipe) {                                                            \
      if constexpr (MAXR != kSmallRanks) return SS_ERR_INVALID_ARG;                       \
      else if constexpr (F) return launch_pipe_n<G, P, W, MAXR, 2, true>(a, stream);      \
      else return launch_pipe<G, P, W, MAXR>(a, stream);                                  \
    }                                                                                     \
    if (path == Path::kVector) {                                                          \
      if constexpr (F) return SS_ERR_INVALID_ARG;                                         \
      else {                                                                              \
        auto* fn = adam_vec_kernel<G, P, F, W, MAXR>;                                     \
        return launch(fn, grid_for(reinterpret_cast<const void*>(fn), (a.n - a.head) / kGroup, kChunkThreads), a, \
                      stream, kChunkThreads);                                             \
      }                                                                                   \
    }                                                                                     \
    auto* fn = adam_scalar_kernel<G, P, F, W, MAXR>;                                      \
    return launch(fn, grid_for(reinterpret_cast<const void*>(fn), a.n), a, stream);       \
  }
#define SS_ADAM_P(G, P) SS_ADAM_CASE(G, P, false, true) SS_ADAM_CASE(G, P, false, false)
  SS_ADAM_P(SS_BF16, SS_BF16)
  SS_ADAM_P(SS_BF16, SS_FP16)
  SS_ADAM_P(SS_FP16, SS_BF16)
  SS_ADAM_P(SS_FP16, SS_FP16)
  if constexpr (MAXR == kSmallRanks) {
    SS_ADAM_CASE(SS_BF16, SS_BF16, true, true)
    SS_ADAM_CASE(SS_BF16, SS_BF16, true, false)
    SS_ADAM_CASE(SS_BF16, SS_FP16, true, true)
    SS_ADAM_CASE(SS_BF16, SS_FP16, true, false)
  }
#undef SS_ADAM_P
#undef SS_ADAM_CASE
  return SS_ERR_DTYPE;
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" {

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
  Path path = !vec ? Path::kScalar : ((from_g32 || pipe_ranks(n_ranks)) ? Path::kPipe : Path::kVector);
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
  // Some rank counts whose 16-bit arrays share the state's phase take the warp-cooperative
  // double-buffered kernel of ss_step_shift.cu too, every phase 0 (same results). Measured
  // on GB300 at 2^26 elements: 9-16 ranks 0.99-1.05 of the copy peak there, against
  // 0.97-0.99 single-buffered here and 0.80-0.91 for this file's double-buffered kernel
  // in 256-thread blocks; 5 ranks 1.00 against 0.96; 4 ranks 1.00 against 0.98.
  if (vec && !from_g32 && n_ranks <= 16 && ((kWarpCoopRankMask >> n_ranks) & 1u) && n - h >= 3 * kGroup) {
    path = Path::kShift;
    for (int32_t r = 0; r < n_ranks; ++r)
      rphase[r] = static_cast<uint8_t>((reinterpret_cast<uintptr_t>(rank_grads[r]) + 2u * h) & 15u);
    if (param16) pphase = static_cast<uint8_t>((reinterpret_cast<uintptr_t>(param16) + 2u * h) & 15u);
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

}  // extern "C"
