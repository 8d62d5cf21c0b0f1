// ss_copy.cu -- unshard / reshard: the gather copy of the ranks' shards into the
// flat unit buffer and its inverse, one launch over all shards: 16-byte
// vectors aligned on the destination, the source read directly when it shares
// the destination's 16-byte phase and warp-cooperatively shifted otherwise.
#include "ss_common.cuh"

namespace ss {
namespace {

// ------------------------------------------------------------------ unshard / reshard copies

template <int MAXR>
struct CopyArgs {
  const void* src[MAXR];
  void* dst[MAXR];
  int64_t bytes[MAXR];
  int32_t n_seg;
  int32_t esize;
};

// Destination-aligned 16-byte vectors, kCopyUnroll per thread per iteration
// with their loads issued first, when source and destination share a 16-byte
// phase (vectors past the end re-read vector j0, in range, and are not stored).
// Sixteen vectors (256 bytes) in flight per thread measured fastest on GB300:
// 2-5% above a cp.async.bulk (TMA) global -> shared -> global copy with four
// 16 KB chunks in flight per block, on every size and shard count tried.
constexpr int kCopyUnroll = 16;
// Threads per block: 256, one block per SM at this register count. Blocks of
// 128 or 64 threads (a finer grid when many segments leave SMs idle) measured
// 3-6% slower on every copy tried.
#ifndef SS_COPY_THREADS
#define SS_COPY_THREADS 256
#endif
constexpr int kCopyThreads = SS_COPY_THREADS;

__device__ __forceinline__ void copy_body_aligned(const char* s, char* d, int64_t h, int64_t nvec, int64_t tid,
                                                  int64_t stride) {
  for (int64_t j0 = tid; j0 < nvec; j0 += stride * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t j = j0 + u * stride;
      v[u] = __ldcs(reinterpret_cast<const uint4*>(s + h + 16 * (j < nvec ? j : j0)));
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t j = j0 + u * stride;
      if (j < nvec) __stcs(reinterpret_cast<uint4*>(d + h + 16 * j), v[u]);
    }
  }
}

// Destination-aligned vectors whose source lies SOFF (2..14) bytes past a
// 16-byte boundary, warp-cooperatively: vector j's 16 bytes are the window at
// SOFF into source chunks j and j + 1 (aligned, chunk j at s + h - SOFF + 16 j).
// A warp takes blocks of 32 x kCopyUnroll consecutive vectors; lane l loads
// chunk (block start + 32 u + l) for each u and takes chunk + 1 from lane l + 1
// by shuffle (lane 31 from lane 0's next chunk, or, after the last u, from one
// extra load), so each source byte is loaded once. Body: vectors 1 .. nvec-2,
// whose chunks 1 .. nvec-1 all lie inside the segment's source range; vectors
// 0 and nvec - 1 are copied element by element with the head and tail.
template <int SOFF>
__device__ __forceinline__ void copy_body_shifted(const char* s, char* d, int64_t h, int64_t nvec, int64_t warp,
                                                  int64_t nwarps, int lane) {
  constexpr int U = kCopyUnroll;
  const char* c0 = s + h - SOFF;
  const int64_t last = nvec - 1;  // the highest chunk index read
  for (int64_t v0 = 1 + warp * 32 * U; v0 < last; v0 += nwarps * 32 * U) {  // warp-uniform
    uint4 c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      int64_t j = v0 + u * 32 + lane;
      j = j < last ? j : last;
      c[u] = __ldcs(reinterpret_cast<const uint4*>(c0 + 16 * j));
    }
    uint4 extra = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 31) {
      int64_t j = v0 + U * 32;
      j = j < last ? j : last;
      extra = __ldcs(reinterpret_cast<const uint4*>(c0 + 16 * j));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint4 nb = make_uint4(__shfl_down_sync(0xFFFFFFFFu, c[u].x, 1), __shfl_down_sync(0xFFFFFFFFu, c[u].y, 1),
                            __shfl_down_sync(0xFFFFFFFFu, c[u].z, 1), __shfl_down_sync(0xFFFFFFFFu, c[u].w, 1));
      if (u + 1 < U) {
        const uint4 f = make_uint4(__shfl_sync(0xFFFFFFFFu, c[u + 1 < U ? u + 1 : u].x, 0),
                                   __shfl_sync(0xFFFFFFFFu, c[u + 1 < U ? u + 1 : u].y, 0),
                                   __shfl_sync(0xFFFFFFFFu, c[u + 1 < U ? u + 1 : u].z, 0),
                                   __shfl_sync(0xFFFFFFFFu, c[u + 1 < U ? u + 1 : u].w, 0));
        if (lane == 31) nb = f;
      } else if (lane == 31) {
        nb = extra;
      }
      const int64_t v = v0 + u * 32 + lane;
      if (v < last) __stcs(reinterpret_cast<uint4*>(d + h + 16 * v), window16<SOFF>(c[u], nb));
    }
  }
}

template <int MAXR>
__global__ void __launch_bounds__(kCopyThreads) copy_segments_kernel(const __grid_constant__ CopyArgs<MAXR> a) {
  pdl_wait();
  pdl_trigger();
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
  const int64_t warp = tid >> 5, nwarps = stride >> 5;
  const int lane = threadIdx.x & 31;
  switch (soff) {
    case 0: copy_body_aligned(s, d, h, nvec, tid, stride); break;
    case 2: copy_body_shifted<2>(s, d, h, nvec, warp, nwarps, lane); break;
    case 4: copy_body_shifted<4>(s, d, h, nvec, warp, nwarps, lane); break;
    case 6: copy_body_shifted<6>(s, d, h, nvec, warp, nwarps, lane); break;
    case 8: copy_body_shifted<8>(s, d, h, nvec, warp, nwarps, lane); break;
    case 10: copy_body_shifted<10>(s, d, h, nvec, warp, nwarps, lane); break;
    case 12: copy_body_shifted<12>(s, d, h, nvec, warp, nwarps, lane); break;
    default: copy_body_shifted<14>(s, d, h, nvec, warp, nwarps, lane); break;
  }
  // Element by element: the head (h bytes) and the tail (bytes - t0), and with
  // a shifted source also vectors 0 and nvec - 1 (or every vector when nvec <
  // 3): at most 62 bytes, one element per thread of the segment's first block.
  const int64_t ve = soff == 0 ? 0 : (nvec < 3 ? nvec : 2);  // edge vectors copied here
  const int64_t eb = 16 / a.esize;                            // elements per vector
  const int64_t nh = h / a.esize, nt = (bytes - t0) / a.esize;
  if (blockIdx.x == 0 && threadIdx.x < nh + nt + ve * eb) {
    const int64_t i = threadIdx.x;
    int64_t off;
    if (i < nh) {
      off = i * a.esize;
    } else if (i < nh + nt) {
      off = t0 + (i - nh) * a.esize;
    } else {
      const int64_t q = i - nh - nt;                  // element q of the edge vectors
      const int64_t vec = q / eb;                     // 0, 1 (or up to 2 when nvec < 3)
      const int64_t vi = (nvec < 3) ? vec : (vec == 0 ? 0 : nvec - 1);
      off = h + 16 * vi + (q % eb) * a.esize;
    }
    if (a.esize == 2) *reinterpret_cast<uint16_t*>(d + off) = *reinterpret_cast<const uint16_t*>(s + off);
    else *reinterpret_cast<uint32_t*>(d + off) = *reinterpret_cast<const uint32_t*>(s + off);
  }
}

template <int MAXR>
ss_status run_copy(const void* const* src, void* const* dst, const int64_t* bytes, int32_t n_seg, int32_t esize,
                   int64_t total_bytes, void* stream) {
  CopyArgs<MAXR> a;
  std::memset(&a, 0, sizeof a);
  for (int32_t k = 0; k < n_seg; ++k) {
    a.src[k] = src[k];
    a.dst[k] = dst[k];
    a.bytes[k] = bytes[k];
  }
  a.n_seg = n_seg;
  a.esize = esize;
  auto* fn = copy_segments_kernel<MAXR>;
  const int64_t cap = std::max<int64_t>(
      1, static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(fn), kCopyThreads));
  const int64_t per_seg_work = (total_bytes / std::max(1, n_seg)) / 16 + 1;
  // one wave: at most cap / n_seg blocks per segment (a partial second wave would double the tail)
  int64_t gx = std::min<int64_t>(cap / n_seg, (per_seg_work + kCopyThreads - 1) / kCopyThreads);
  gx = std::max<int64_t>(gx, 1);
  return launch_dependent(fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(n_seg)), dim3(kCopyThreads), 0,
                          stream, a);
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" {

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
