// Quantize-on-append (INT4 tail / staging pages), INT2 repack and table
// scatter kernels.
//
// Quantization follows TriAxialKV, key design 3 (asymmetric group
// quantization, G = 32): for a group with minimum mn and maximum mx,
//   scale = half_rn((mx - mn) / (2^b - 1)),  zero = half_rn(mn),
//   code  = clamp(rint((x - zero) / scale), 0, 2^b - 1)   (0 when scale == 0),
// with IEEE fp32 subtraction and division (no fast-math, no FTZ) and binary16
// round-to-nearest-even storage.  INT4 K and V are per token (32 consecutive
// channels); the INT2 repack dequantizes a full 32-token staging page with
// fmaf(code, scale, zero) and requantizes K per channel (across the 32 tokens)
// and V per token.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ bool out_of_range(float x) { return !(fabsf(x) <= 65504.0f); }

struct GroupMeta {
  __half s, z;
  float sf, zf;
  bool nz;
};

__device__ __forceinline__ GroupMeta make_meta(float mn, float mx, float qmax) {
  GroupMeta m;
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), qmax);
  m.s = __float2half_rn(s32);
  m.z = __float2half_rn(mn);
  m.sf = __half2float(m.s);
  m.zf = __half2float(m.z);
  m.nz = (__half_as_ushort(m.s) & 0x7FFFu) != 0;
  return m;
}

// code = clamp(rint(fl((x - zero) / scale)), 0, qmax) (0 when scale == 0),
// without a division in the common case.  rs = approximate
// reciprocal of m.sf (relative error < 2^-22), so q0 = u * rs lies within
// 4e-6 of the correctly rounded quotient fl(u / s) for |u / s| < 64 (here
// |u / s| <= qmax + 1).  When q0 is more than 1e-5 from every half-integer,
// fl(u / s) rounds to the same integer; otherwise the quotient is computed
// exactly.  Same result as the division form, bit for bit.
__device__ __forceinline__ float approx_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t qcode_fast(float x, const GroupMeta& m, float rs, float qmax) {
  if (!m.nz) return 0u;
  const float u = __fsub_rn(x, m.zf);
  const float q0 = u * rs;
  float c = rintf(q0);
  if (!(fabsf(fabsf(q0 - c) - 0.5f) > 1e-5f)) c = rintf(__fdiv_rn(u, m.sf));
  return (uint32_t)fminf(fmaxf(c, 0.0f), qmax);
}

// min / max over the 8 lanes of one 32-channel group (lanes 8*gr .. 8*gr + 7)
__device__ __forceinline__ void group8_minmax(float& mn, float& mx) {
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
}

__device__ __forceinline__ void st_half(uint8_t* img, int byte_off, __half h) {
  *reinterpret_cast<__half*>(img + byte_off) = h;
}

__device__ __forceinline__ void or_bits(uint8_t* img, int byte_off, int shift, uint32_t val) {
  atomicOr(reinterpret_cast<uint32_t*>(img) + (byte_off >> 2), val << (8 * (byte_off & 3) + shift));
}

// Quantize one token (a warp: lane = channels 4*lane .. 4*lane+3) into slot
// `slot` of an INT4 block image `img` (shared or global memory).  V nibbles
// are OR-ed in: the block's unfilled slots hold zeros.
// With vcodes (shared memory, [slot][channel] bytes) the V codes go there
// for a later word-wise packing (pack_i4v) instead of being OR-ed into img.
// vmax: the warp's running maximum of V scales (one atomic per warp at the
// end instead of one per token on the pool's single maximum word).
// A token's K and V rows of one kv head, as each lane holds them (4 bf16
// channels 4*lane .. 4*lane+3 of each).
struct RawRows {
  uint2 kr, vr;
};
__device__ __forceinline__ RawRows load_rows(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                                             int t, int h, int hkv) {
  const size_t row = ((size_t)t * hkv + h) * kHeadDim + 4 * (threadIdx.x & 31);
  return RawRows{*reinterpret_cast<const uint2*>(k + row), *reinterpret_cast<const uint2*>(v + row)};
}

__device__ __forceinline__ bool quantize_rows(uint8_t* img, const RawRows& rr, int slot, float& vmax,
                                              uint8_t* vcodes = nullptr) {
  const int lane = threadIdx.x & 31, gr = lane >> 3;
  const uint2 kr = rr.kr, vr = rr.vr;
  float xk[4], xv[4];
  xk[0] = __uint_as_float(kr.x << 16); xk[1] = __uint_as_float(kr.x & 0xFFFF0000u);
  xk[2] = __uint_as_float(kr.y << 16); xk[3] = __uint_as_float(kr.y & 0xFFFF0000u);
  xv[0] = __uint_as_float(vr.x << 16); xv[1] = __uint_as_float(vr.x & 0xFFFF0000u);
  xv[2] = __uint_as_float(vr.y << 16); xv[3] = __uint_as_float(vr.y & 0xFFFF0000u);
  bool bad = false;
  float kmn = xk[0], kmx = xk[0], vmn = xv[0], vmx = xv[0];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    bad |= out_of_range(xk[a]) | out_of_range(xv[a]);
    kmn = fminf(kmn, xk[a]); kmx = fmaxf(kmx, xk[a]);
    vmn = fminf(vmn, xv[a]); vmx = fmaxf(vmx, xv[a]);
  }
  group8_minmax(kmn, kmx);
  group8_minmax(vmn, vmx);
  const GroupMeta km = make_meta(kmn, kmx, 15.0f);
  const GroupMeta vm = make_meta(vmn, vmx, 15.0f);
  uint32_t ck[4], cv[4];
  const float krs = approx_rcp(km.sf), vrs = approx_rcp(vm.sf);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ck[a] = qcode_fast(xk[a], km, krs, 15.0f);
    cv[a] = qcode_fast(xv[a], vm, vrs, 15.0f);
  }
  // K: channels 4*lane .. 4*lane+3 are nibbles 0..3 or 4..7 of one word -> 2 bytes
  const int kb = i4k_byte(slot, 4 * lane);
  *reinterpret_cast<uint16_t*>(img + kb) = (uint16_t)(ck[0] | (ck[1] << 4) | (ck[2] << 8) | (ck[3] << 12));
  // V: channel-major, one nibble per channel
  if (vcodes) {
    *reinterpret_cast<uint32_t*>(vcodes + kHeadDim * slot + 4 * lane) = cv[0] | (cv[1] << 8) | (cv[2] << 16) | (cv[3] << 24);
  } else {
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int c = 4 * lane + a;
      or_bits(img, i4v_byte(slot, c), i4v_shift(slot), cv[a]);
    }
  }
  vmax = fmaxf(vmax, vm.sf);   // per lane; reduced over the warp by flush_vmax
  if ((lane & 7) == 0) {
    st_half(img, kI4KMeta + 16 * slot + 4 * gr, km.s);
    st_half(img, kI4KMeta + 16 * slot + 4 * gr + 2, km.z);
    st_half(img, kI4VMeta + 2 * v_meta_index(slot, gr), vm.s);
    st_half(img, kI4VMeta + 256 + 2 * v_meta_index(slot, gr), vm.z);
  }
  return bad;
}

// The tokens j = warp, warp + W, ... < n of a job (W = warps per CTA), each
// into slot first + j: their indices are read at once (lane q holds the q-th)
// and the next token's rows are loaded while the current one is quantized.
template <int W>
__device__ __forceinline__ bool quantize_tokens(uint8_t* img, const __nv_bfloat16* __restrict__ k,
                                                const __nv_bfloat16* __restrict__ v,
                                                const int32_t* __restrict__ tk, int n, int first, int h, int hkv,
                                                float& vmax, uint8_t* vcodes) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mine = n > warp ? (n - warp + W - 1) / W : 0;   // <= 32 / W
  const int t_l = lane < mine ? tk[warp + W * lane] : 0;
  bool bad = false;
  if (mine == 0) return bad;
  RawRows cur = load_rows(k, v, __shfl_sync(0xFFFFFFFFu, t_l, 0), h, hkv);
  for (int q = 0; q < mine; ++q) {
    RawRows nxt = cur;
    if (q + 1 < mine) nxt = load_rows(k, v, __shfl_sync(0xFFFFFFFFu, t_l, q + 1), h, hkv);
    bad |= quantize_rows(img, cur, first + warp + W * q, vmax, vcodes);
    cur = nxt;
  }
  return bad;
}

// One atomic per warp for the pool's running maximum of V scales
// (non-negative floats order as their bits).
__device__ __forceinline__ void flush_vmax(float vmax, uint32_t* __restrict__ status) {
#pragma unroll
  for (int o = 16; o; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
  if ((threadIdx.x & 31) == 0 && vmax > 0.0f) atomicMax(status + 2, __float_as_uint(vmax));
}

// INT4 V words from [slot][channel] code bytes: word (channel c, slot chunk j)
// holds slots 8j .. 8j+7 in nibbles 0..7; every word is built by one thread.
__device__ __forceinline__ void pack_i4v(uint8_t* __restrict__ img, const uint8_t* __restrict__ vcodes) {
  for (int x = threadIdx.x; x < kHeadDim * (kPage / 8); x += kThreads) {
    const int c = x & (kHeadDim - 1), j = x >> 7;
    uint32_t w = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) w |= (uint32_t)vcodes[kHeadDim * (8 * j + k) + c] << (4 * k);
    *reinterpret_cast<uint32_t*>(img + i4v_byte(8 * j, c)) = w;
  }
}

// One CTA per (job, kv head), a warp per token.  A new page (job starting at
// slot 0) is built as an image in shared memory from zeros and written whole,
// so its unfilled slots read as code 0, scale 0, zero 0; a page that already
// holds tokens gets only its new slots written in place (the V words by
// atomic OR).  The kv-head-0 CTA also writes the page's table entry and the
// request's table length, so an append that only fills or adds tail pages
// needs no separate table update.
template <bool kByValue>
__global__ void __launch_bounds__(kThreads) append_int4_kernel(
    uint8_t* __restrict__ pool, size_t int4_off, int64_t n2, int hkv, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const AppendJob* __restrict__ jobs, const int32_t* __restrict__ toks,
    Entry* __restrict__ table, int32_t* __restrict__ ntab, uint32_t* __restrict__ status,
    const __grid_constant__ SmallAppend small) {
  __shared__ __align__(16) uint8_t img[kInt4Block];
  __shared__ __align__(16) uint8_t vcodes[kPage * kHeadDim];   // V codes of a new page, packed after
  asm volatile("griddepcontrol.wait;" ::: "memory");   // earlier work on the stream (the previous decode) is done
  asm volatile("griddepcontrol.launch_dependents;");
  const AppendJob job = kByValue ? small.jobs[blockIdx.x] : jobs[blockIdx.x];
  const int32_t* tk = kByValue ? small.toks : toks;
  const int h = blockIdx.y;
  uint8_t* blk = pool + int4_off + ((size_t)(job.page - n2) * hkv + h) * kInt4Block;
  const bool fresh = job.first_slot == 0;
  bool bad = false;
  float vmax = 0.0f;
  if (fresh) {
    uint4* img4 = reinterpret_cast<uint4*>(img);
    for (int i = threadIdx.x; i < kInt4Block / 16; i += kThreads) img4[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < kPage * kHeadDim / 16; i += kThreads)
      reinterpret_cast<uint4*>(vcodes)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    bad |= quantize_tokens<kThreads / 32>(img, k, v, tk + job.tok_off, job.n_slots, job.first_slot, h, hkv, vmax,
                                          vcodes);
    __syncthreads();
    pack_i4v(img, vcodes);
    __syncthreads();
    uint4* out4 = reinterpret_cast<uint4*>(blk);
    for (int i = threadIdx.x; i < kInt4Block / 16; i += kThreads) out4[i] = img4[i];
  } else {
    bad |= quantize_tokens<kThreads / 32>(blk, k, v, tk + job.tok_off, job.n_slots, job.first_slot, h, hkv, vmax,
                                          nullptr);
  }
  flush_vmax(vmax, status);
  if (bad) atomicOr(status, kStatusRange);
  if (h == 0 && threadIdx.x == 0) {
    if (job.tab_index >= 0) table[job.tab_index] = Entry{job.page, job.live};
    if (job.ntab_req >= 0) ntab[job.ntab_req] = job.ntab_len;
  }
}

// Requantize a 32-token INT4 block image (shared memory) into an INT2 block
// image (shared memory): K per channel across the 32 tokens, V per token and
// group, both from the INT4-dequantized values fmaf(code, scale, zero); tracks
// the largest INT2 K and V scales.  The codes go through `codes` ([slot]
// [channel] bytes, shared memory) and are packed so that every output byte is
// written by one thread.  128 threads.
__device__ __forceinline__ void repack_image(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                             uint32_t* __restrict__ smax_bits, uint8_t* __restrict__ codes) {
  // K: thread c owns channel c; its group is the 32 tokens of the page.
  {
    const int c = threadIdx.x;
    const int gr = c >> 5;
    float x[kPage];
    float mn, mx;
#pragma unroll
    for (int t = 0; t < kPage; ++t) {
      const uint32_t code = (src[i4k_byte(t, c)] >> i4k_shift(c)) & 15u;
      const float sf = __half2float(*reinterpret_cast<const __half*>(src + kI4KMeta + 16 * t + 4 * gr));
      const float zf = __half2float(*reinterpret_cast<const __half*>(src + kI4KMeta + 16 * t + 4 * gr + 2));
      x[t] = __fmaf_rn((float)code, sf, zf);
      mn = t ? fminf(mn, x[t]) : x[t];
      mx = t ? fmaxf(mx, x[t]) : x[t];
    }
    const GroupMeta m = make_meta(mn, mx, 3.0f);
    const float rs = approx_rcp(m.sf);
#pragma unroll
    for (int t = 0; t < kPage; ++t) codes[kHeadDim * t + c] = (uint8_t)qcode_fast(x[t], m, rs, 3.0f);
    st_half(dst, kI2KMeta + 2 * i2k_meta_index(c), m.s);
    st_half(dst, kI2KMeta + 256 + 2 * i2k_meta_index(c), m.z);
    // running maximum of INT2 K scales (non-negative floats order as their bits)
    float smx = m.sf;
#pragma unroll
    for (int o = 16; o; o >>= 1) smx = fmaxf(smx, __shfl_xor_sync(0xFFFFFFFFu, smx, o));
    if ((threadIdx.x & 31) == 0) atomicMax(smax_bits, __float_as_uint(smx));
  }
  __syncthreads();
  // K codes: byte (slot t, b) holds channels 4b .. 4b+3
  for (int x = threadIdx.x; x < kPage * (kHeadDim / 4); x += kThreads) {
    const int t = x >> 5, b = x & 31;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + kHeadDim * t + 4 * b);
    dst[i2k_byte(t, 4 * b)] = (uint8_t)((w & 3u) | ((w >> 6) & 0xCu) | ((w >> 12) & 0x30u) | ((w >> 18) & 0xC0u));
  }
  __syncthreads();
  // V: thread -> (slot t, group gr), 32 channels each.
  {
    const int t = threadIdx.x >> 2, gr = threadIdx.x & 3;
    const int mi = v_meta_index(t, gr);
    const float sf = __half2float(*reinterpret_cast<const __half*>(src + kI4VMeta + 2 * mi));
    const float zf = __half2float(*reinterpret_cast<const __half*>(src + kI4VMeta + 256 + 2 * mi));
    float x[kGroup];
    float mn, mx;
#pragma unroll
    for (int cc = 0; cc < kGroup; ++cc) {
      const int c = kGroup * gr + cc;
      const uint32_t code = (src[i4v_byte(t, c)] >> i4v_shift(t)) & 15u;
      x[cc] = __fmaf_rn((float)code, sf, zf);
      mn = cc ? fminf(mn, x[cc]) : x[cc];
      mx = cc ? fmaxf(mx, x[cc]) : x[cc];
    }
    const GroupMeta m = make_meta(mn, mx, 3.0f);
    const float rs = approx_rcp(m.sf);
#pragma unroll
    for (int cc = 0; cc < kGroup; ++cc) codes[kHeadDim * t + kGroup * gr + cc] = (uint8_t)qcode_fast(x[cc], m, rs, 3.0f);
    st_half(dst, kI2VMeta + 2 * mi, m.s);
    st_half(dst, kI2VMeta + 256 + 2 * mi, m.z);
    float vmx = m.sf;
#pragma unroll
    for (int o = 16; o; o >>= 1) vmx = fmaxf(vmx, __shfl_xor_sync(0xFFFFFFFFu, vmx, o));
    if ((threadIdx.x & 31) == 0) atomicMax(smax_bits + 1, __float_as_uint(vmx));
  }
  __syncthreads();
  // V codes: the 8 slots of chunk i of channel c fill two bytes (4 slots each)
  for (int x = threadIdx.x; x < kHeadDim * (kPage / 8); x += kThreads) {
    const int c = x & (kHeadDim - 1), i = x >> 7;
    const int b0 = i2v_byte(8 * i, c);
    int b1 = b0;
    uint32_t v0 = 0u, v1 = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int t = 8 * i + k, b = i2v_byte(t, c);
      const uint32_t code = (uint32_t)codes[kHeadDim * t + c] << i2v_shift(t);
      if (b == b0) {
        v0 |= code;
      } else {
        v1 |= code;
        b1 = b;
      }
    }
    dst[b0] = (uint8_t)v0;
    dst[b1] = (uint8_t)v1;
  }
}

// One CTA per (repack job, kv head): INT4 staging block -> INT2 block.
__global__ void __launch_bounds__(kThreads) repack_int2_kernel(uint8_t* __restrict__ pool, size_t int4_off,
                                                              int64_t n2, int hkv,
                                                              const RepackJob* __restrict__ jobs,
                                                              uint32_t* __restrict__ smax_bits) {
  __shared__ __align__(16) uint8_t src[kInt4Block];
  __shared__ __align__(16) uint8_t dst[kInt2Block];
  __shared__ __align__(16) uint8_t codes[kPage * kHeadDim];
  const RepackJob job = jobs[blockIdx.x];
  const int h = blockIdx.y;
  const uint8_t* sblk = pool + int4_off + ((size_t)(job.src - n2) * hkv + h) * kInt4Block;
  uint8_t* dblk = pool + ((size_t)job.dst * hkv + h) * kInt2Block;
  for (int i = threadIdx.x; i < kInt4Block / 16; i += kThreads)
    reinterpret_cast<uint4*>(src)[i] = reinterpret_cast<const uint4*>(sblk)[i];
  for (int i = threadIdx.x; i < kInt2Block / 16; i += kThreads)
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  repack_image(src, dst, smax_bits, codes);
  __syncthreads();
  for (int i = threadIdx.x; i < kInt2Block / 16; i += kThreads)
    reinterpret_cast<uint4*>(dblk)[i] = reinterpret_cast<const uint4*>(dst)[i];
}

// One CTA per (direct job, kv head): 32 tokens that fill a fresh staging page
// within one call.  The staging page's INT4 image is built in shared memory
// exactly as the append kernel builds a new page (a warp per token), then
// requantized to INT2 as the repack kernel does; only the INT2 block is
// written to memory.  Launched as a programmatic dependent of the append
// kernel, which signals after its own wait: the earlier work on the stream
// (the previous decode, the uploads) is complete when this grid starts, and
// it touches nothing the append kernel writes, so the two run side by side.
// Every thread waits for the append grid before it exits, so the kernels
// that follow in stream order (the repack reads staging pages the append
// kernel fills) see both.
__global__ void __launch_bounds__(kThreads) direct_int2_kernel(
    uint8_t* __restrict__ pool, int hkv, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const DirectJob* __restrict__ jobs, const int32_t* __restrict__ toks, uint32_t* __restrict__ status) {
  __shared__ __align__(16) uint8_t img[kInt4Block];
  __shared__ __align__(16) uint8_t dst[kInt2Block];
  __shared__ __align__(16) uint8_t codes[kPage * kHeadDim];
  const DirectJob job = jobs[blockIdx.x];
  const int h = blockIdx.y;
  bool bad = false;
  float vmax = 0.0f;
  // every slot is written: no zeroing
  bad |= quantize_tokens<kThreads / 32>(img, k, v, toks + job.tok_off, kPage, 0, h, hkv, vmax, codes);
  flush_vmax(vmax, status);
  if (bad) atomicOr(status, kStatusRange);
  __syncthreads();
  pack_i4v(img, codes);
  __syncthreads();
  repack_image(img, dst, status + 1, codes);
  __syncthreads();
  uint8_t* dblk = pool + ((size_t)job.dst * hkv + h) * kInt2Block;
  for (int i = threadIdx.x; i < kInt2Block / 16; i += kThreads)
    reinterpret_cast<uint4*>(dblk)[i] = reinterpret_cast<const uint4*>(dst)[i];
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void scatter_kernel(Entry* __restrict__ table, int32_t* __restrict__ ntab, uint32_t* __restrict__ hdead,
                               int hkv, const TableUpd* __restrict__ upd, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const TableUpd u = upd[i];
  if (u.kind == 0) table[u.index] = Entry{u.a, u.b};
  else if (u.kind == 1) ntab[u.index] = u.a;
  else if (hdead) hdead[(size_t)u.index * hkv + u.a] = u.b;   // kind 2: per-head exclusion word
}

}  // namespace

cudaError_t launch_append(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                          const int32_t* d_toks, const SmallAppend* small, cudaStream_t s) {
  if (n_jobs <= 0) return cudaSuccess;
  dim3 grid((unsigned)n_jobs, (unsigned)P->cfg.num_kv_heads);
  ++P->launches;
  const AppendJob* no_jobs = nullptr;
  const int32_t* no_toks = nullptr;
  if (small)
    return launch_pdl(append_int4_kernel<true>, grid, dim3(kThreads), 0, s, P->d_pool, P->int4_offset,
                      P->cfg.n_int2_pages, P->cfg.num_kv_heads, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
                      no_jobs, no_toks, P->d_table, P->d_ntab, P->d_status, *small);
  static const SmallAppend none{};
  return launch_pdl(append_int4_kernel<false>, grid, dim3(kThreads), 0, s, P->d_pool, P->int4_offset,
                    P->cfg.n_int2_pages, P->cfg.num_kv_heads, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
                    d_jobs, d_toks, P->d_table, P->d_ntab, P->d_status, none);
}

cudaError_t launch_repack(kv_pool* P, const RepackJob* d_jobs, int n_jobs, cudaStream_t s) {
  if (n_jobs <= 0) return cudaSuccess;
  dim3 grid((unsigned)n_jobs, (unsigned)P->cfg.num_kv_heads);
  ++P->launches;
  repack_int2_kernel<<<grid, kThreads, 0, s>>>(P->d_pool, P->int4_offset, P->cfg.n_int2_pages,
                                               P->cfg.num_kv_heads, d_jobs, P->d_status + 1);
  return cudaGetLastError();
}

cudaError_t launch_direct_int2(kv_pool* P, const void* k, const void* v, const DirectJob* d_jobs, int n_jobs,
                               const int32_t* d_toks, cudaStream_t s) {
  if (n_jobs <= 0) return cudaSuccess;
  dim3 grid((unsigned)n_jobs, (unsigned)P->cfg.num_kv_heads);
  ++P->launches;
  return launch_pdl(direct_int2_kernel, grid, dim3(kThreads), 0, s, P->d_pool, P->cfg.num_kv_heads,
                    (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, d_jobs, d_toks, P->d_status);
}

cudaError_t launch_scatter(kv_pool* P, const TableUpd* d_upd, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  ++P->launches;
  scatter_kernel<<<(n + 255) / 256, 256, 0, s>>>(P->d_table, P->d_ntab, P->d_hdead, P->cfg.num_kv_heads, d_upd, n);
  return cudaGetLastError();
}

}  // namespace kvq
