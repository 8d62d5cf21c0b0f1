/* c_abi_consumer.c -- a plain C99 program using the shard-step library through
 * include/ss.h alone (no Python, no PyTorch): the boundary is usable from C.
 *
 *   consumer          host-only calls: layout, accounting, status strings and
 *                     argument errors reported before any launch
 *   consumer gpu      also device calls on cudaMalloc'd buffers and the
 *                     legacy default stream: an exact rank-ordered reduce, the
 *                     first AdamW step against its closed form, and an
 *                     unshard/reshard round trip
 *
 * Prints "OK" and exits 0 when every check holds. Built by the tests with
 * gcc (-DSS_WITH_CUDA for the device part) and linked against libss.so.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ss.h"

#ifdef SS_WITH_CUDA
#include <cuda_runtime_api.h>
#endif

static int fails = 0;
#define CHECK(c)                                                        \
  do {                                                                  \
    if (!(c)) {                                                         \
      fprintf(stderr, "FAIL %s:%d: %s\n", __FILE__, __LINE__, #c);      \
      ++fails;                                                          \
    }                                                                   \
  } while (0)

static void host_checks(void) {
  /* layout: three tensors of 5, 0, 3 elements over 7 ranks */
  const int64_t numels[3] = {5, 0, 3};
  int64_t offs[4], bounds[8];
  CHECK(ss_flatten_layout(numels, 3, 7, offs, bounds) == SS_OK);
  CHECK(offs[0] == 0 && offs[1] == 5 && offs[2] == 5 && offs[3] == 8);
  for (int k = 0; k <= 7; ++k) CHECK(bounds[k] == (int64_t)k * 8 / 7);
  for (int64_t i = 0; i < 8; ++i) {
    const int32_t k = ss_shard_of(8, 7, i);
    CHECK(k >= 0 && k < 7 && bounds[k] <= i && i < bounds[k + 1]);
  }
  CHECK(ss_shard_of(8, 7, 8) == -1 && ss_shard_of(8, 7, -1) == -1);
  int32_t count = -1;
  CHECK(ss_shard_segments(offs, 3, bounds, 7, 6, NULL, 0, &count) == SS_OK && count == 1);
  ss_segment seg;
  CHECK(ss_shard_segments(offs, 3, bounds, 7, 6, &seg, 1, &count) == SS_OK);
  CHECK(seg.tensor == 2 && seg.tensor_offset == bounds[6] - 5 && seg.shard_offset == 0 &&
        seg.length == bounds[7] - bounds[6]);
  CHECK(ss_flatten_layout(NULL, 3, 7, offs, bounds) == SS_ERR_INVALID_ARG);
  CHECK(ss_flatten_layout(numels, 3, 0, offs, bounds) == SS_ERR_INVALID_ARG);

  /* accounting: the pages' 16 bytes per parameter, and the ZeRO-1 share */
  ss_bytes b;
  CHECK(ss_state_bytes(1000, 8, 1, &b) == SS_OK);
  CHECK(b.mp_total == 16000.0 && b.fp32_total == 16000.0 && b.optimizer_state == 12000.0);
  CHECK(b.zero1_optimizer_per_gpu == 1500.0 && b.full_shard_per_gpu == 2000.0);

  /* status strings and version */
  for (int s = SS_OK; s <= SS_ERR_CUDA; ++s) CHECK(ss_status_string((ss_status)s) != NULL);
  CHECK(ss_abi_version() == SS_ABI_VERSION);

  /* argument errors are found on the host: these pointers are never dereferenced */
  float* const fake = (float*)(uintptr_t)0x7000000000ull;
  ss_adamw_hparams hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, 0, 0}; /* step 0 */
  CHECK(ss_adam_step(&hp, 64, fake, NULL, 0, SS_BF16, 1.0f, fake + 64, fake + 128, fake + 192, NULL, SS_BF16,
                     NULL, NULL) == SS_ERR_INVALID_ARG);
  hp.step = 1;
  CHECK(ss_adam_step(&hp, 64, fake, NULL, 0, SS_BF16, 1.0f, fake + 64, fake + 96, fake + 192, NULL, SS_BF16, NULL,
                     NULL) == SS_ERR_OVERLAP);
  CHECK(ss_adam_step(&hp, 64, fake, NULL, 0, SS_BF16, 1.0f, (float*)((char*)fake + 258), fake + 128, fake + 192, NULL,
                     SS_BF16, NULL, NULL) == SS_ERR_ALIGN);
  const void* ranks[2] = {fake, fake + 64};
  CHECK(ss_grad_reduce(ranks, 2, SS_FP32, 64, 1.0f, 0, fake + 128, NULL, NULL) == SS_ERR_DTYPE);
  CHECK(ss_grad_reduce(ranks, 2, SS_BF16, -1, 1.0f, 0, fake + 128, NULL, NULL) == SS_ERR_INVALID_ARG);
  CHECK(ss_grad_sumsq_workspace(-1) == -1 && ss_grad_sumsq_workspace(16384) == 8 * 3);
}

#ifdef SS_WITH_CUDA
/* bf16 bits of a small integer (exact) */
static uint16_t bf16_bits(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  return (uint16_t)(u >> 16);
}

static float rank_value(int64_t i, int r) { return (float)((i * 7 + r * 3) % 201 - 100); }

static void gpu_checks(void) {
  enum { N = 3 };
  const int64_t n = 1000003;
  uint16_t* h16 = (uint16_t*)malloc((size_t)n * 2);
  float* h32 = (float*)malloc((size_t)n * 4);
  void* d_ranks[N];
  float *d_g, *d_p, *d_m, *d_v, *d_flat;
  for (int r = 0; r < N; ++r) {
    CHECK(cudaMalloc(&d_ranks[r], (size_t)n * 2) == cudaSuccess);
    for (int64_t i = 0; i < n; ++i) h16[i] = bf16_bits(rank_value(i, r));
    CHECK(cudaMemcpy(d_ranks[r], h16, (size_t)n * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  }
  CHECK(cudaMalloc((void**)&d_g, (size_t)n * 4) == cudaSuccess);

  /* reduce: small integers, so the rank-ordered fp32 sum is exact */
  CHECK(ss_grad_reduce((const void* const*)d_ranks, N, SS_BF16, n, 1.0f, 0, d_g, NULL, NULL) == SS_OK);
  CHECK(cudaMemcpy(h32, d_g, (size_t)n * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  int64_t bad = 0;
  for (int64_t i = 0; i < n; ++i)
    bad += h32[i] != rank_value(i, 0) + rank_value(i, 1) + rank_value(i, 2);
  CHECK(bad == 0);

  /* AdamW, first step from zero moments: p1 = p0 (1 - lr wd) - lr g / (|g| + eps) */
  const ss_adamw_hparams hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, 0, 1};
  CHECK(cudaMalloc((void**)&d_p, (size_t)n * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&d_m, (size_t)n * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&d_v, (size_t)n * 4) == cudaSuccess);
  for (int64_t i = 0; i < n; ++i) h32[i] = 0.02f * (float)((i % 97) - 48) / 48.0f;
  CHECK(cudaMemcpy(d_p, h32, (size_t)n * 4, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemset(d_m, 0, (size_t)n * 4) == cudaSuccess);
  CHECK(cudaMemset(d_v, 0, (size_t)n * 4) == cudaSuccess);
  CHECK(ss_adam_step(&hp, n, NULL, (const void* const*)d_ranks, N, SS_BF16, 0.001f, d_p, d_m, d_v, NULL, SS_BF16,
                     NULL, NULL) == SS_OK);
  float* hp1 = (float*)malloc((size_t)n * 4);
  CHECK(cudaMemcpy(hp1, d_p, (size_t)n * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  bad = 0;
  for (int64_t i = 0; i < n; ++i) {
    const double g = (double)(float)((rank_value(i, 0) + rank_value(i, 1) + rank_value(i, 2)) * 0.001f);
    const double lr = (double)hp.lr, wd = (double)hp.weight_decay, eps = (double)hp.eps;
    const double ref = (double)h32[i] * (1.0 - lr * wd) - lr * g / (fabs(g) + eps);
    const double tol = fmax(1e-6 * fabs(ref), 1e-9);
    bad += fabs((double)hp1[i] - ref) > tol;
  }
  CHECK(bad == 0);

  /* unshard then reshard: fp32 shards of a 7-way cut, bit-exact round trip */
  const int64_t P = 2000011;
  int64_t numel[1] = {P}, offs[2], bnd[8];
  CHECK(ss_flatten_layout(numel, 1, 7, offs, bnd) == SS_OK);
  void* shards[7];
  float* hp32 = (float*)malloc((size_t)P * 4);
  for (int64_t i = 0; i < P; ++i) hp32[i] = (float)i;
  for (int k = 0; k < 7; ++k) {
    const int64_t len = bnd[k + 1] - bnd[k];
    CHECK(cudaMalloc(&shards[k], (size_t)len * 4) == cudaSuccess);
    CHECK(cudaMemcpy(shards[k], hp32 + bnd[k], (size_t)len * 4, cudaMemcpyHostToDevice) == cudaSuccess);
  }
  CHECK(cudaMalloc((void**)&d_flat, (size_t)P * 4) == cudaSuccess);
  CHECK(ss_unshard((const void* const*)shards, bnd, 7, SS_FP32, d_flat, NULL) == SS_OK);
  for (int k = 0; k < 7; ++k) CHECK(cudaMemset(shards[k], 0, (size_t)(bnd[k + 1] - bnd[k]) * 4) == cudaSuccess);
  CHECK(ss_reshard(d_flat, bnd, 7, SS_FP32, shards, NULL) == SS_OK);
  bad = 0;
  for (int k = 0; k < 7; ++k) {
    const int64_t len = bnd[k + 1] - bnd[k];
    CHECK(cudaMemcpy(h32, shards[k], (size_t)len * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
    for (int64_t j = 0; j < len; ++j) bad += h32[j] != (float)(bnd[k] + j);
  }
  CHECK(bad == 0);
  CHECK(cudaDeviceSynchronize() == cudaSuccess);

  for (int k = 0; k < 7; ++k) cudaFree(shards[k]);
  for (int r = 0; r < N; ++r) cudaFree(d_ranks[r]);
  cudaFree(d_g);
  cudaFree(d_p);
  cudaFree(d_m);
  cudaFree(d_v);
  cudaFree(d_flat);
  free(h16);
  free(h32);
  free(hp1);
  free(hp32);
}
#endif

int main(int argc, char** argv) {
  host_checks();
  if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
#ifdef SS_WITH_CUDA
    gpu_checks();
#else
    fprintf(stderr, "built without SS_WITH_CUDA\n");
    return 2;
#endif
  }
  if (fails) {
    printf("FAILED %d\n", fails);
    return 1;
  }
  printf("OK\n");
  return 0;
}
