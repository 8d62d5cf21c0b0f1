// synth_dev.cu -- device side of the seeded input generator (see synth_core.h).
// One grid-stride kernel writes elements [start, start+count) of a stream into
// a device buffer; the bits equal those of synth_fill_range on the host.
#include <cuda_runtime.h>
#include "synth_core.h"

__global__ void synth_fill_kernel(synth_spec s, uint64_t key, uint64_t sel, uint64_t start,
                                  uint64_t count, void* out) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t k = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k < count; k += stride) {
    uint32_t bits = synth_bits(&s, key, sel, start + k);
    if (s.fmt == SYNTH_FMT_FP32) ((uint32_t*)out)[k] = bits;
    else ((uint16_t*)out)[k] = (uint16_t)bits;
  }
}

extern "C" int synth_fill_range_dev(const synth_spec* s, uint64_t start, uint64_t count, void* out,
                                    void* stream) {
  if (!s || (!out && count)) return 1;
  if (count == 0) return 0;
  uint64_t key = synth_key(s->seed, s->stream);
  uint64_t sel = synth_key(s->seed, s->outlier_stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 2;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 2;
  uint64_t blocks = (count + 255) / 256;
  uint64_t cap = (uint64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  synth_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(*s, key, sel, start, count, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
