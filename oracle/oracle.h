/* oracle.h -- declarations of the CPU oracle (test infrastructure only).
 * Independent of the product library's header: its own types and codes. */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

enum { ORA_OK = 0, ORA_EINVAL = 1, ORA_EOVERFLOW = 5 };
enum { ORA_BF16 = 0, ORA_FP16 = 1, ORA_FP32 = 2 };

typedef struct ora_segment {
  int32_t tensor;
  int32_t pad_;
  int64_t tensor_offset;
  int64_t shard_offset;
  int64_t length;
} ora_segment;

typedef struct ora_bytes {
  double fp32_params, fp32_grads, fp32_adam, fp32_total;
  double mp_params16, mp_grads16, mp_master32, mp_adam32, mp_total;
  double optimizer_state, zero1_optimizer_per_gpu;
  double full_shard_per_gpu, shard_grad_op_per_gpu, no_shard_per_gpu;
  double unit_gather, full_shard_peak, full_shard_saving, shard_grad_op_saving;
  double mp_full_shard_per_gpu, mp_unit_gather16;
} ora_bytes;

typedef struct ora_adamw_hp {
  float lr, beta1, beta2, eps, weight_decay;
  int32_t pad_;
  int64_t step;
} ora_adamw_hp;

int ora_flatten_layout(const int64_t* numels, int32_t n_tensors, int32_t n_ranks, int64_t* offsets,
                       int64_t* bounds);
int32_t ora_shard_of(int64_t P, int32_t n_ranks, int64_t i);
int ora_shard_segments(const int64_t* offsets, int32_t n_tensors, const int64_t* bounds, int32_t shard,
                       ora_segment* out, int32_t* count);
int ora_state_bytes(int64_t P, int32_t n_ranks, int32_t n_units, ora_bytes* out);
float ora_widen16(uint16_t h, int32_t dtype);
uint16_t ora_round_bf16(float f);
uint16_t ora_round_fp16(float f);
uint16_t ora_round16(float f, int32_t dtype);
int ora_round16_array(const float* x, int64_t n, int32_t dtype, uint16_t* out);
int ora_widen16_array(const uint16_t* h, int64_t n, int32_t dtype, float* out);
int ora_grad_reduce(const uint16_t* const* ranks, int32_t n_ranks, int32_t dtype, int64_t n, float post_scale,
                    int32_t accumulate, float* out);
int ora_adamw(const ora_adamw_hp* hp, int64_t n, const float* g, float grad_scale, float* master, float* m,
              float* v, uint16_t* p16, int32_t p16_dtype);
int ora_unshard(const void* const* shards, const int64_t* bounds, int32_t n_ranks, int32_t elem_size, void* flat);
int ora_reshard(const void* flat, const int64_t* bounds, int32_t n_ranks, int32_t elem_size, void* const* shards);
double ora_sumsq(const float* g, int64_t n);
float ora_clip_coef(double total_sumsq, float max_norm);
int32_t ora_all_finite(const float* g, int64_t n);
void ora_set_threads(int32_t n);
int32_t ora_max_threads(void);
#endif
