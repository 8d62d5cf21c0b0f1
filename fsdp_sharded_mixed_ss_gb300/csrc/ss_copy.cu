// ss_copy.cu -- unshard / reshard: the gather copy of the ranks' shards into the
// flat unit buffer and its inverse, on the bulk-copy (TMA) engine when every
// segment keeps its 16-byte phase, else on SIMT threads; and the library's
// device error word raised by the bulk copy's bounded waits.
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
constexpr int kCopyUnroll = 8;

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
__global__ void __launch_bounds__(kThreads) copy_segments_kernel(const __grid_constant__ CopyArgs<MAXR> a) {
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

// Wait for the phase of the given parity to complete, for at most limit_ns
// (~1 s by default); on expiry set the timeout bit of the device error word
// and return false.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      atomicOr(&g_device_error, SS_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives at, so the wait runs out after limit_ns and reports through the
// device error word, exactly as a bulk-copy wait would. Nothing is in flight
// on the barrier, so the block simply returns.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint64_t limit_ns) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1u);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  mbar_wait(b, 0u, limit_ns);
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
  pdl_wait();
  pdl_trigger();
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

// Raise a kernel's dynamic shared memory limit once per device (cached per device and kernel).
bool allow_smem(const void* fn, size_t bytes) {
  struct Done {
    int dev;
    const void* fn;
    size_t bytes;
  };
  static std::mutex mu;
  static std::vector<Done> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (const Done& d : done)
    if (d.dev == dev && d.fn == fn && d.bytes >= bytes) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess)
    return false;
  done.push_back({dev, fn, bytes});
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
    return launch_dependent(fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(n_seg)), dim3(32), smem, stream, a);
  }
  auto* fn = copy_segments_kernel<MAXR>;
  const int64_t cap = std::max<int64_t>(1, static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(fn)));
  const int64_t per_seg_work = (total_bytes / std::max(1, n_seg)) / 16 + 1;
  int64_t gx = std::min<int64_t>((cap + n_seg - 1) / n_seg, (per_seg_work + kThreads - 1) / kThreads);
  gx = std::max<int64_t>(gx, 1);
  return launch_dependent(fn, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(n_seg)), dim3(kThreads), 0, stream, a);
}

}  // namespace
}  // namespace ss

using namespace ss;

extern "C" {

ss_status ss_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns < 1000000 || limit_ns > 2000000000) return SS_ERR_INVALID_ARG;
  return launch_dependent(wait_timeout_selftest_kernel, dim3(1), dim3(32), 0, stream,
                          static_cast<uint64_t>(limit_ns));
}

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
