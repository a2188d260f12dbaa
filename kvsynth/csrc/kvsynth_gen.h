/* Seeded synthetic-input generator shared by the CUDA path's tests/benchmark
 * and by the CPU oracle's tests.  It holds no arithmetic of the KV-cache
 * method: it only turns (seed, tensor, stream, element index) into a bf16
 * value that is approximately N(0,1).
 *
 * Definition (identical on host and device, integer-exact):
 *   r0 = Philox4x32-10(ctr = {idx_lo, idx_hi, tensor, 2*stream + 0}, key = {seed_lo, seed_hi})
 *   r1 = Philox4x32-10(ctr = {idx_lo, idx_hi, tensor, 2*stream + 1}, key)
 *   S  = sum of the twelve 16-bit halves of r0[0..3], r1[0..1]      (Irwin-Hall, n = 12)
 *   x  = (S - 6*65536) / 65536            exact in fp32, mean 0, variance 1, |x| <= 6
 *   y  = x * chan_mult * row_mult         fp32 (the multipliers used are 1, 8, 20: exact)
 *   bf16 = round-to-nearest-even(y)
 * Philox4x32-10 follows Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
 * as easy as 1, 2, 3" (SC'11): multipliers 0xD2511F53 / 0xCD9E8D57, Weyl
 * key increments 0x9E3779B9 / 0xBB67AE85, ten rounds.
 */
#ifndef KVSYNTH_GEN_H
#define KVSYNTH_GEN_H
#include <stdint.h>

#ifdef __CUDACC__
#define KVS_HD __host__ __device__ __forceinline__
#else
#define KVS_HD static inline
#endif

KVS_HD void kvs_mulhilo(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  *hi = (uint32_t)(p >> 32);
  *lo = (uint32_t)p;
}

KVS_HD void kvs_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    uint32_t hi0, lo0, hi1, lo1;
    kvs_mulhilo(0xD2511F53u, c0, &hi0, &lo0);
    kvs_mulhilo(0xCD9E8D57u, c2, &hi1, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

KVS_HD float kvs_base_value(uint64_t seed, uint32_t tensor, uint32_t stream, uint64_t idx) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {(uint32_t)idx, (uint32_t)(idx >> 32), tensor, 2u * stream};
  uint32_t r0[4], r1[4];
  kvs_philox4x32_10(ctr, key, r0);
  ctr[3] = 2u * stream + 1u;
  kvs_philox4x32_10(ctr, key, r1);
  int32_t s = 0;
  for (int i = 0; i < 4; ++i) s += (int32_t)(r0[i] & 0xFFFFu) + (int32_t)(r0[i] >> 16);
  for (int i = 0; i < 2; ++i) s += (int32_t)(r1[i] & 0xFFFFu) + (int32_t)(r1[i] >> 16);
  return (float)(s - 6 * 65536) * (1.0f / 65536.0f);
}

KVS_HD uint16_t kvs_f32_to_bf16_rne(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  u += 0x7FFFu + ((u >> 16) & 1u);   /* inputs are finite by construction */
  return (uint16_t)(u >> 16);
}

#endif
