// ss_step.cuh -- pieces shared by the two CUDA sources of the fused shard step:
// ss_step.cu (the entry point ss_adam_step and the kernels for arrays that share
// the fp32 state's 16-byte phase) and ss_step_shift.cu (the kernels for 16-bit
// arrays off that phase).
#pragma once

#include "ss_common.cuh"

namespace ss {

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

// The 16-bit arrays' byte phases at the fp32 group starts, for the shifted-load kernels.
// When the fp32 arrays share a 16-byte phase but some 16-bit arrays (rank gradients,
// param16) do not, groups start where the fp32 arrays are 16-byte aligned and the 16-bit
// arrays are read as aligned chunks shifted into place.
template <int MAXR>
struct ShiftArgs {
  StepArgs<MAXR> s;
  uint8_t rphase[MAXR];  // byte offset of each rank's group starts past a 16-byte boundary (even)
  uint8_t pphase;        // the same for param16
};

// The shifted-load step (ss_step_shift.cu): picks the kernel form for the ranks' phases
// and the formats. rphase[r] is rank r's byte phase, pphase param16's.
template <int MAXR>
ss_status shift_step(const StepArgs<MAXR>& a, ss_dtype gt, ss_dtype pt, bool from_g32, bool p16,
                     const uint8_t* rphase, uint8_t pphase, void* stream);

}  // namespace ss
