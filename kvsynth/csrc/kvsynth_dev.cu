/* Device side of the synthetic-input generator; see kvsynth_gen.h.  Same
 * definition as kvsynth_host.c, so host and device produce identical bits. */
#include <cuda_runtime.h>
#include "kvsynth_gen.h"

__global__ void kvs_fill_kernel(uint16_t* __restrict__ out, int64_t n_elem, int32_t H, int32_t D,
                                uint64_t seed, uint32_t tensor, uint32_t stream, int64_t tok0,
                                const float* __restrict__ chan_mult, const float* __restrict__ row_mult) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_elem; e += stride) {
    int64_t t = e / ((int64_t)H * D);
    int32_t hd = (int32_t)(e - t * (int64_t)H * D);
    uint64_t idx = (uint64_t)(tok0 * (int64_t)H * D) + (uint64_t)e;
    float x = kvs_base_value(seed, tensor, stream, idx);
    float cm = chan_mult ? chan_mult[hd] : 1.0f;
    float rm = row_mult ? row_mult[t] : 1.0f;
    out[e] = kvs_f32_to_bf16_rne(x * cm * rm);
  }
}

extern "C" int kvs_fill_bf16_dev(void* out, int64_t n_tok, int32_t H, int32_t D, uint64_t seed,
                                 uint32_t tensor, uint32_t stream, int64_t tok0,
                                 const float* chan_mult_dev, const float* row_mult_dev, void* cuda_stream) {
  int64_t n = n_tok * (int64_t)H * D;
  if (n <= 0) return 0;
  int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  kvs_fill_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)cuda_stream>>>(
      (uint16_t*)out, n, H, D, seed, tensor, stream, tok0, chan_mult_dev, row_mult_dev);
  return (int)cudaGetLastError();
}
