/* A plain C11 client of libkvq.so, used by the tests to drive the whole C ABI
 * without the Python binding: pool create, request open, one
 * kv_append_quant call per request, evictions by position, the INT2-first
 * reorder, kv_decode_attn, kv_pool_sync, kv_request_info, kv_pool_destroy.
 *
 * usage: kvq_c_client <in.bin> <out.bin>
 *
 * in.bin (little endian):
 *   int32 num_kv_heads, num_q_heads, n_req
 *   int32 n_tok[n_req]
 *   float softmax_scale
 *   per request r: uint8 bits[n_tok[r]],
 *                  uint16 k[n_tok[r]][num_kv_heads][128] (bf16), uint16 v[same]
 *   int64 n_evict; int32 evict_req[n_evict] (request index); int64 evict_pos[n_evict]
 *   uint16 q[n_req][num_q_heads][128] (bf16)
 * out.bin: float out[n_req][num_q_heads][128], then int64 n_tokens[n_req] as
 * kv_request_info reports them.
 *
 * Every status is checked; on an error the client prints kv_last_error() and
 * exits with status 1. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvq.h"

#define KV_CHECK(call)                                                                       \
  do {                                                                                       \
    kv_status_t st_ = (call);                                                                \
    if (st_ != KV_OK) {                                                                      \
      fprintf(stderr, "%s: status %d: %s\n", #call, (int)st_, kv_last_error());              \
      return 1;                                                                              \
    }                                                                                        \
  } while (0)
#define CUDA_CHECK(call)                                                                     \
  do {                                                                                       \
    cudaError_t e_ = (call);                                                                 \
    if (e_ != cudaSuccess) {                                                                 \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                            \
      return 1;                                                                              \
    }                                                                                        \
  } while (0)
#define READ(f, p, n)                                                                        \
  do {                                                                                       \
    if (fread((p), 1, (n), (f)) != (size_t)(n)) {                                            \
      fprintf(stderr, "short read: %s\n", #p);                                               \
      return 1;                                                                              \
    }                                                                                        \
  } while (0)

static void* xmalloc(size_t n) {
  void* p = malloc(n ? n : 1);
  if (!p) {
    fprintf(stderr, "out of host memory\n");
    exit(1);
  }
  return p;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s in.bin out.bin\n", argv[0]);
    return 2;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) {
    fprintf(stderr, "cannot open %s\n", argv[1]);
    return 1;
  }
  int32_t hdr[3];
  READ(in, hdr, sizeof hdr);
  const int32_t hkv = hdr[0], hq = hdr[1], n_req = hdr[2];
  if (hkv < 1 || hq < hkv || n_req < 1) {
    fprintf(stderr, "bad header\n");
    return 1;
  }
  int32_t* n_tok = (int32_t*)xmalloc((size_t)n_req * sizeof(int32_t));
  READ(in, n_tok, (size_t)n_req * sizeof(int32_t));
  float scale;
  READ(in, &scale, sizeof scale);
  int64_t total = 0;
  int32_t longest = 0;
  for (int32_t r = 0; r < n_req; ++r) {
    total += n_tok[r];
    if (n_tok[r] > longest) longest = n_tok[r];
  }

  kv_pool_config_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.num_kv_heads = hkv;
  cfg.head_dim = 128;
  cfg.page_tokens = 32;
  cfg.group = 32;
  cfg.n_int2_pages = total / 32 + 4;
  cfg.n_int4_pages = total / 32 + 2 * (int64_t)n_req + longest / 32 + 8;   /* tails, staging, transient staging */
  cfg.max_requests = n_req;
  cfg.max_pages_per_request = longest / 32 + 8;
  cfg.device = 0;
  kv_pool_t* pool = NULL;
  KV_CHECK(kv_pool_create(&cfg, &pool));

  int32_t* rid = (int32_t*)xmalloc((size_t)n_req * sizeof(int32_t));
  for (int32_t r = 0; r < n_req; ++r) KV_CHECK(kv_request_open(pool, &rid[r]));

  /* device K/V rows of every request stay allocated until the pool has synced */
  const size_t row = (size_t)hkv * 128 * sizeof(uint16_t);
  void** dk = (void**)xmalloc((size_t)n_req * sizeof(void*));
  void** dv = (void**)xmalloc((size_t)n_req * sizeof(void*));
  for (int32_t r = 0; r < n_req; ++r) {
    const size_t n = (size_t)n_tok[r];
    uint8_t* bits = (uint8_t*)xmalloc(n);
    uint16_t* hk = (uint16_t*)xmalloc(n * row);
    uint16_t* hv = (uint16_t*)xmalloc(n * row);
    int32_t* ids = (int32_t*)xmalloc(n * sizeof(int32_t));
    READ(in, bits, n);
    READ(in, hk, n * row);
    READ(in, hv, n * row);
    for (size_t t = 0; t < n; ++t) ids[t] = rid[r];
    CUDA_CHECK(cudaMalloc(&dk[r], n * row));
    CUDA_CHECK(cudaMalloc(&dv[r], n * row));
    CUDA_CHECK(cudaMemcpy(dk[r], hk, n * row, cudaMemcpyHostToDevice));
    CUDA_CHECK(cudaMemcpy(dv[r], hv, n * row, cudaMemcpyHostToDevice));
    KV_CHECK(kv_append_quant(pool, dk[r], dv[r], ids, bits, (int64_t)n, NULL));
    free(bits);
    free(hk);
    free(hv);
    free(ids);
  }

  int64_t n_ev = 0;
  READ(in, &n_ev, sizeof n_ev);
  if (n_ev < 0) {
    fprintf(stderr, "bad eviction count\n");
    return 1;
  }
  if (n_ev > 0) {
    int32_t* ev_req = (int32_t*)xmalloc((size_t)n_ev * sizeof(int32_t));
    int64_t* ev_pos = (int64_t*)xmalloc((size_t)n_ev * sizeof(int64_t));
    READ(in, ev_req, (size_t)n_ev * sizeof(int32_t));
    READ(in, ev_pos, (size_t)n_ev * sizeof(int64_t));
    for (int64_t i = 0; i < n_ev; ++i) {
      if (ev_req[i] < 0 || ev_req[i] >= n_req) {
        fprintf(stderr, "bad eviction request\n");
        return 1;
      }
      ev_req[i] = rid[ev_req[i]];
    }
    KV_CHECK(kv_evict_slots(pool, ev_req, ev_pos, n_ev, NULL));
    free(ev_req);
    free(ev_pos);
  }
  KV_CHECK(kv_reorder_pages(pool, rid, n_req, NULL));

  const size_t nq = (size_t)n_req * hq * 128;
  uint16_t* hqv = (uint16_t*)xmalloc(nq * sizeof(uint16_t));
  READ(in, hqv, nq * sizeof(uint16_t));
  fclose(in);
  void* dq = NULL;
  float* dout = NULL;
  CUDA_CHECK(cudaMalloc(&dq, nq * sizeof(uint16_t)));
  CUDA_CHECK(cudaMalloc((void**)&dout, nq * sizeof(float)));
  CUDA_CHECK(cudaMemcpy(dq, hqv, nq * sizeof(uint16_t), cudaMemcpyHostToDevice));
  KV_CHECK(kv_decode_attn(pool, dq, rid, n_req, hq, scale, dout, NULL));
  KV_CHECK(kv_pool_sync(pool));

  float* out = (float*)xmalloc(nq * sizeof(float));
  CUDA_CHECK(cudaMemcpy(out, dout, nq * sizeof(float), cudaMemcpyDeviceToHost));
  int64_t* ntok_out = (int64_t*)xmalloc((size_t)n_req * sizeof(int64_t));
  for (int32_t r = 0; r < n_req; ++r) {
    int32_t pages = 0;
    KV_CHECK(kv_request_info(pool, rid[r], &pages, &ntok_out[r]));
  }
  FILE* fo = fopen(argv[2], "wb");
  if (!fo || fwrite(out, sizeof(float), nq, fo) != nq ||
      fwrite(ntok_out, sizeof(int64_t), (size_t)n_req, fo) != (size_t)n_req || fclose(fo) != 0) {
    fprintf(stderr, "cannot write %s\n", argv[2]);
    return 1;
  }
  for (int32_t r = 0; r < n_req; ++r) KV_CHECK(kv_request_close(pool, rid[r]));
  KV_CHECK(kv_pool_destroy(pool));
  for (int32_t r = 0; r < n_req; ++r) {
    CUDA_CHECK(cudaFree(dk[r]));
    CUDA_CHECK(cudaFree(dv[r]));
  }
  CUDA_CHECK(cudaFree(dq));
  CUDA_CHECK(cudaFree(dout));
  free(dk);
  free(dv);
  free(hqv);
  free(out);
  free(ntok_out);
  free(rid);
  free(n_tok);
  return 0;
}
