/* Host (CPU) side of the synthetic-input generator; see kvsynth_gen.h. */
#include <stddef.h>
#include "kvsynth_gen.h"

/* out[t][h][d] (bf16 bits) for local tokens t in [0, n_tok); the element index
 * fed to the generator is ((tok0 + t) * H + h) * D + d.  chan_mult is [H][D]
 * (NULL = 1), row_mult is [n_tok] (NULL = 1). */
void kvs_fill_bf16(uint16_t* out, int64_t n_tok, int32_t H, int32_t D, uint64_t seed,
                   uint32_t tensor, uint32_t stream, int64_t tok0,
                   const float* chan_mult, const float* row_mult) {
  for (int64_t t = 0; t < n_tok; ++t) {
    float rm = row_mult ? row_mult[t] : 1.0f;
    for (int32_t h = 0; h < H; ++h) {
      for (int32_t d = 0; d < D; ++d) {
        uint64_t idx = ((uint64_t)(tok0 + t) * (uint64_t)H + (uint64_t)h) * (uint64_t)D + (uint64_t)d;
        float x = kvs_base_value(seed, tensor, stream, idx);
        float cm = chan_mult ? chan_mult[h * D + d] : 1.0f;
        out[(t * H + h) * (int64_t)D + d] = kvs_f32_to_bf16_rne(x * cm * rm);
      }
    }
  }
}

/* Raw Philox4x32-10 blocks, for known-answer tests. */
void kvs_philox_blocks(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) kvs_philox4x32_10(ctr + 4 * i, key + 2 * i, out + 4 * i);
}

/* Same values as kvs_fill_bf16 restricted to the heads listed in `heads`:
 * out[t][j][d] = element (tok0 + t, heads[j], d) of the [*][H][D] tensor. */
void kvs_fill_bf16_heads(uint16_t* out, int64_t n_tok, int32_t H, int32_t D, uint64_t seed, uint32_t tensor,
                         uint32_t stream, int64_t tok0, const float* chan_mult, const float* row_mult,
                         const int32_t* heads, int32_t n_heads) {
  for (int64_t t = 0; t < n_tok; ++t) {
    float rm = row_mult ? row_mult[t] : 1.0f;
    for (int32_t j = 0; j < n_heads; ++j) {
      int32_t h = heads[j];
      for (int32_t d = 0; d < D; ++d) {
        uint64_t idx = ((uint64_t)(tok0 + t) * (uint64_t)H + (uint64_t)h) * (uint64_t)D + (uint64_t)d;
        float x = kvs_base_value(seed, tensor, stream, idx);
        float cm = chan_mult ? chan_mult[h * D + d] : 1.0f;
        out[(t * n_heads + j) * (int64_t)D + d] = kvs_f32_to_bf16_rne(x * cm * rm);
      }
    }
  }
}
