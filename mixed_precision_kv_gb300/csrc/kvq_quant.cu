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

// ---- INT3 pages (TriAxialKV, limitations and outlook: INT3 as a further
// width): the INT4 per-token rule with 2^3 - 1 levels, codes stored as a
// 2-bit low plane and a 1-bit high plane.  A warp quantizes one token of one
// kv head, lane = channels 4*lane .. 4*lane+3 (one group per 8 lanes).
// K: a lane's four low-bit fields are one byte of the token's low plane and
// its four high bits one nibble of the high plane, whose byte it shares with
// the lane of the neighbouring group (lane ^ 8): the even group's lane writes
// the byte.  V (channel-major) goes to vcodes for a fresh page (packed by
// pack_i3v), else its bits are OR-ed into the block.
__device__ __forceinline__ bool quantize_rows3(uint8_t* img, const RawRows& rr, int slot, float& vmax,
                                               uint8_t* vcodes) {
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
  const GroupMeta km = make_meta(kmn, kmx, 7.0f);
  const GroupMeta vm = make_meta(vmn, vmx, 7.0f);
  uint32_t ck[4], cv[4];
  const float krs = approx_rcp(km.sf), vrs = approx_rcp(vm.sf);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ck[a] = qcode_fast(xk[a], km, krs, 7.0f);
    cv[a] = qcode_fast(xv[a], vm, vrs, 7.0f);
  }
  const int c0 = 4 * lane;
  img[i3k_lo_byte(slot, c0)] = (uint8_t)((ck[0] & 3u) | ((ck[1] & 3u) << 2) | ((ck[2] & 3u) << 4) | ((ck[3] & 3u) << 6));
  const uint32_t hi = (ck[0] >> 2) | ((ck[1] >> 2) << 1) | ((ck[2] >> 2) << 2) | ((ck[3] >> 2) << 3);
  const uint32_t hi_odd = __shfl_xor_sync(0xFFFFFFFFu, hi, 8);
  if ((gr & 1) == 0) img[i3k_hi_byte(slot, c0)] = (uint8_t)(hi | (hi_odd << 4));
  if (vcodes) {
    *reinterpret_cast<uint32_t*>(vcodes + kHeadDim * slot + c0) = cv[0] | (cv[1] << 8) | (cv[2] << 16) | (cv[3] << 24);
  } else {
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int c = c0 + a;
      or_bits(img, i3v_lo_byte(slot, c), i3v_lo_shift(slot), cv[a] & 3u);
      or_bits(img, i3v_hi_byte(slot, c), i3v_hi_shift(slot, c), cv[a] >> 2);
    }
  }
  vmax = fmaxf(vmax, vm.sf);
  if ((lane & 7) == 0) {
    st_half(img, kI3KMeta + 16 * slot + 4 * gr, km.s);
    st_half(img, kI3KMeta + 16 * slot + 4 * gr + 2, km.z);
    st_half(img, kI3VMeta + 2 * v_meta_index(slot, gr), vm.s);
    st_half(img, kI3VMeta + 256 + 2 * v_meta_index(slot, gr), vm.z);
  }
  return bad;
}

// INT3 V planes from [slot][channel] code bytes, every word by one thread:
// low-plane word (chunk X, h) and high-plane word X of the layout.
__device__ __forceinline__ void pack_i3v(uint8_t* __restrict__ img, const uint8_t* __restrict__ vcodes) {
  for (int x = threadIdx.x; x < 3 * 128; x += kThreads) {
    const int X = x < 256 ? x >> 1 : x - 256;
    const int mh = X >> 5, r = (X >> 2) & 7, j = X & 3;   // chunk X = 32 (m >> 1) + 4 r + j
    uint32_t w = 0u;
    if (x < 256) {
      const int h = x & 1, m = 2 * mh + h;
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w |= ((uint32_t)vcodes[kHeadDim * (8 * j + k) + 16 * m + 8 * e + r] & 3u) << (8 * e + 2 * (k & 3) + 16 * (k >> 2));
      *reinterpret_cast<uint32_t*>(img + kI3VCodes + 8 * X + 4 * h) = w;
    } else {
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        const int m = 2 * mh + (wd >> 1), e = wd & 1;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w |= ((uint32_t)vcodes[kHeadDim * (8 * j + k) + 16 * m + 8 * e + r] >> 2) << (4 * wd + (k & 3) + 16 * (k >> 2));
      }
      *reinterpret_cast<uint32_t*>(img + kI3VHigh + 4 * X) = w;
    }
  }
}

// One CTA per (job, kv head) of INT3 tail pages, a warp per token; a new page
// is built in shared memory from zeros and written whole, a page that
// already holds tokens gets its new slots in place (V bits by atomic OR).
// Table entry and length as in append_int4_kernel.
__global__ void __launch_bounds__(kThreads) append_int3_kernel(
    uint8_t* __restrict__ pool, size_t int3_off, int64_t n3b, int hkv, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const AppendJob* __restrict__ jobs, const int32_t* __restrict__ toks,
    Entry* __restrict__ table, int32_t* __restrict__ ntab, uint32_t* __restrict__ status) {
  __shared__ __align__(16) uint8_t img[kInt3Block];
  __shared__ __align__(16) uint8_t vcodes[kPage * kHeadDim];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const AppendJob job = jobs[blockIdx.x];
  const int h = blockIdx.y;
  uint8_t* blk = pool + int3_off + ((size_t)(job.page - n3b) * hkv + h) * kInt3Block;
  const bool fresh = job.first_slot == 0;
  uint8_t* dst = fresh ? img : blk;
  if (fresh) {
    for (int i = threadIdx.x; i < kInt3Block / 16; i += kThreads) reinterpret_cast<uint4*>(img)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < kPage * kHeadDim / 16; i += kThreads)
      reinterpret_cast<uint4*>(vcodes)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
  }
  const int warp = threadIdx.x >> 5;
  const int32_t* tk = toks + job.tok_off;
  bool bad = false;
  float vmax = 0.0f;
  for (int q = warp; q < job.n_slots; q += kThreads / 32)
    bad |= quantize_rows3(dst, load_rows(k, v, tk[q], h, hkv), job.first_slot + q, vmax, fresh ? vcodes : nullptr);
  if (fresh) {
    __syncthreads();
    pack_i3v(img, vcodes);
    __syncthreads();
    for (int i = threadIdx.x; i < kInt3Block / 16; i += kThreads)
      reinterpret_cast<uint4*>(blk)[i] = reinterpret_cast<const uint4*>(img)[i];
  }
  flush_vmax(vmax, status);
  if (bad) atomicOr(status, kStatusRange);
  if (h == 0 && threadIdx.x == 0) {
    if (job.tab_index >= 0) table[job.tab_index] = Entry{job.page, job.live};
    if (job.ntab_req >= 0) ntab[job.ntab_req] = job.ntab_len;
  }
}

// ---- FP4 pages (TriAxialKV, limitations and outlook: non-uniform FP
// formats; HyQuant background: s = max|X| / c_B with c_B = 6 for E2M1):
// per token and 32-channel group s = half_rn(max|x| / 6), code = the E2M1
// value nearest to x / s (IEEE fp32 quotient), ties to the even mantissa,
// saturating at 6, zero coded +0; s = 0 codes everything 0.  The midpoints of
// the E2M1 grid are exact in fp32, so comparisons decide the rounding.
__device__ __forceinline__ uint32_t e2m1_code(float x, float sf, bool nz) {
  if (!nz) return 0u;
  const float u = __fdiv_rn(x, sf);
  const float a = fabsf(u);
  const uint32_t m = a <= 0.25f ? 0u : a < 0.75f ? 1u : a <= 1.25f ? 2u : a < 1.75f ? 3u
                   : a <= 2.5f  ? 4u : a < 3.5f  ? 5u : a <= 5.0f  ? 6u : 7u;
  return m == 0u ? 0u : ((u < 0.0f ? 8u : 0u) | m);
}

// A warp quantizes one token of one kv head (lane = channels 4*lane ..
// 4*lane+3).  K: a lane's four codes are the low (lane even) or high (lane
// odd) nibbles of one word; the even lane writes the word with its
// neighbour's nibbles.  V as in quantize_rows3.
__device__ __forceinline__ bool quantize_rows_fp4(uint8_t* img, const RawRows& rr, int slot, float& vmax,
                                                  uint8_t* vcodes) {
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
  const __half ks = __float2half_rn(__fdiv_rn(fmaxf(-kmn, kmx), 6.0f));
  const __half vs = __float2half_rn(__fdiv_rn(fmaxf(-vmn, vmx), 6.0f));
  const float ksf = __half2float(ks), vsf = __half2float(vs);
  const bool knz = (__half_as_ushort(ks) & 0x7FFFu) != 0, vnz = (__half_as_ushort(vs) & 0x7FFFu) != 0;
  uint32_t ck[4], cv[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    ck[a] = e2m1_code(xk[a], ksf, knz);
    cv[a] = e2m1_code(xv[a], vsf, vnz);
  }
  const int c0 = 4 * lane;
  const uint32_t kw = ck[0] | (ck[1] << 8) | (ck[2] << 16) | (ck[3] << 24);
  const uint32_t kw_odd = __shfl_xor_sync(0xFFFFFFFFu, kw, 1);
  if ((lane & 1) == 0) *reinterpret_cast<uint32_t*>(img + f4k_byte(slot, c0)) = kw | (kw_odd << 4);
  if (vcodes) {
    *reinterpret_cast<uint32_t*>(vcodes + kHeadDim * slot + c0) = cv[0] | (cv[1] << 8) | (cv[2] << 16) | (cv[3] << 24);
  } else {
#pragma unroll
    for (int a = 0; a < 4; ++a) or_bits(img, f4v_byte(slot, c0 + a), f4v_shift(slot), cv[a]);
  }
  vmax = fmaxf(vmax, vsf);
  if ((lane & 7) == 0) {
    st_half(img, kF4KScale + 8 * slot + 2 * gr, ks);
    st_half(img, kF4VScale + 2 * v_meta_index(slot, gr), vs);
  }
  return bad;
}

// FP4 V words from [slot][channel] code bytes, each word by one thread.
__device__ __forceinline__ void pack_f4v(uint8_t* __restrict__ img, const uint8_t* __restrict__ vcodes) {
  for (int x = threadIdx.x; x < 512; x += kThreads) {
    const int X = x >> 2, w = x & 3;
    const int m = 2 * (X >> 5) + (w >> 1), e = w & 1, r = (X >> 2) & 7, j = X & 3;
    const int c = 16 * m + 8 * e + r;
    uint32_t v = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) v |= (uint32_t)vcodes[kHeadDim * (8 * j + k) + c] << (8 * (k & 3) + 4 * (k >> 2));
    *reinterpret_cast<uint32_t*>(img + kF4VCodes + 16 * X + 4 * w) = v;
  }
}

// One CTA per (job, kv head) of FP4 tail pages, a warp per token (as
// append_int3_kernel).
__global__ void __launch_bounds__(kThreads) append_fp4_kernel(
    uint8_t* __restrict__ pool, size_t fp4_off, int64_t nfb, int hkv, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const AppendJob* __restrict__ jobs, const int32_t* __restrict__ toks,
    Entry* __restrict__ table, int32_t* __restrict__ ntab, uint32_t* __restrict__ status) {
  __shared__ __align__(16) uint8_t img[kFp4Block];
  __shared__ __align__(16) uint8_t vcodes[kPage * kHeadDim];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const AppendJob job = jobs[blockIdx.x];
  const int h = blockIdx.y;
  uint8_t* blk = pool + fp4_off + ((size_t)(job.page - nfb) * hkv + h) * kFp4Block;
  const bool fresh = job.first_slot == 0;
  uint8_t* dst = fresh ? img : blk;
  if (fresh) {
    for (int i = threadIdx.x; i < kFp4Block / 16; i += kThreads) reinterpret_cast<uint4*>(img)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < kPage * kHeadDim / 16; i += kThreads)
      reinterpret_cast<uint4*>(vcodes)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
  }
  const int warp = threadIdx.x >> 5;
  const int32_t* tk = toks + job.tok_off;
  bool bad = false;
  float vmax = 0.0f;
  for (int q = warp; q < job.n_slots; q += kThreads / 32)
    bad |= quantize_rows_fp4(dst, load_rows(k, v, tk[q], h, hkv), job.first_slot + q, vmax, fresh ? vcodes : nullptr);
  if (fresh) {
    __syncthreads();
    pack_f4v(img, vcodes);
    __syncthreads();
    for (int i = threadIdx.x; i < kFp4Block / 16; i += kThreads)
      reinterpret_cast<uint4*>(blk)[i] = reinterpret_cast<const uint4*>(img)[i];
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

// ---- bulk kernels: a CTA of 4 warps per (page, kv head), warp gr = the
// 32-channel group gr, lane t = slot t (its token's 32 channels of the group
// held in registers).  A token's group is quantized without any cross-lane
// step; INT4 metadata comes from packed bf16 min/max, per-channel INT2 K
// statistics from warp reductions across the 32 tokens.  The arithmetic of
// every code, scale and zero is the one qcode_fast / make_meta apply (same
// operations, same order), so the results are bit-identical.
constexpr int kBulkThreads = 128;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf2_min(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float redux_min(float x) {
  float d;
  asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(d) : "f"(x));
  return d;
}
__device__ __forceinline__ float redux_max(float x) {
  float d;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(d) : "f"(x));
  return d;
}

// The 32 bf16 channels 32gr .. 32gr + 31 of token T, kv head h (16 words).
__device__ __forceinline__ void load_group(const __nv_bfloat16* __restrict__ src, int T, int h, int hkv, int gr,
                                           uint32_t (&w)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(src + ((size_t)T * hkv + h) * kHeadDim + 32 * gr);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = __ldg(p + q);
    w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
  }
}

// Group metadata of 32 bf16 values (INT4): min / max exactly, NaN carried so
// that the range check sees it (NaN, Inf or |x| > 65504 sets `bad`).
__device__ __forceinline__ GroupMeta meta_i4(const uint32_t (&w)[16], bool& bad) {
  uint32_t mn2 = w[0], mx2 = w[0];
#pragma unroll
  for (int j = 1; j < 16; ++j) {
    mn2 = bf2_min(mn2, w[j]);
    mx2 = bf2_max(mx2, w[j]);
  }
  const float a = bf_lo(mn2), b = bf_hi(mn2), c = bf_lo(mx2), d = bf_hi(mx2);
  bad |= out_of_range(a) | out_of_range(b) | out_of_range(c) | out_of_range(d);
  return make_meta(fminf(a, b), fmaxf(c, d), 15.0f);
}

// Codes of 8 values of one group: qcode_fast for each (same operations), the
// exact division redone for the whole chunk when any of its quotients lies
// near a rounding tie (rare).
template <int QMAX>
__device__ __forceinline__ void codes8(const float (&x)[8], const GroupMeta& m, float rs, float (&c)[8]) {
  bool tie = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float u = __fsub_rn(x[j], m.zf);
    const float q0 = u * rs;
    const float r = rintf(q0);
    tie |= !(fabsf(fabsf(q0 - r) - 0.5f) > 1e-5f);
    c[j] = fminf(fmaxf(r, 0.0f), (float)QMAX);
  }
  if (tie) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float u = __fsub_rn(x[j], m.zf);
      const float q0 = u * rs;
      float r = rintf(q0);
      if (!(fabsf(fabsf(q0 - r) - 0.5f) > 1e-5f)) r = rintf(__fdiv_rn(u, m.sf));
      c[j] = fminf(fmaxf(r, 0.0f), (float)QMAX);
    }
  }
  if (!m.nz) {
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = 0.0f;
  }
}
// 8 bf16 values of words w[4q .. 4q + 3] as floats
__device__ __forceinline__ void bf8(const uint32_t (&w)[16], int q, float (&x)[8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = bf_lo(w[4 * q + j]);
    x[2 * j + 1] = bf_hi(w[4 * q + j]);
  }
}

// Pack 8 integer-valued floats (0..15) as nibbles 0..7 of a word (exact:
// the two halves are integers below 2^16, read off after adding 2^23).
__device__ __forceinline__ uint32_t pack_nib8(const float (&c)[8]) {
  float lo = c[0], hi = c[4];
#pragma unroll
  for (int n = 1; n < 4; ++n) {
    lo = fmaf(c[n], (float)(1 << (4 * n)), lo);
    hi = fmaf(c[4 + n], (float)(1 << (4 * n)), hi);
  }
  const uint32_t l = __float_as_uint(lo + 8388608.0f) & 0xFFFFu, h = __float_as_uint(hi + 8388608.0f) & 0xFFFFu;
  return l | (h << 16);
}
// Pack 8 integer-valued floats (0..3) as 2-bit fields 0..7 (16 bits).
__device__ __forceinline__ uint32_t pack_crumb8(const float (&c)[8]) {
  float a = c[0];
#pragma unroll
  for (int n = 1; n < 8; ++n) a = fmaf(c[n], (float)(1 << (2 * n)), a);
  return __float_as_uint(a + 8388608.0f) & 0xFFFFu;
}

// Transpose of an 8 x 8 matrix of nibbles held in 8 words (word k = row k,
// nibble n = column n): on return word n holds column n (nibble k = row k).
__device__ __forceinline__ void transpose_nib8x8(uint32_t (&r)[8]) {
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    const uint32_t t = ((r[k] >> 4) ^ r[k + 1]) & 0x0F0F0F0Fu;
    r[k + 1] ^= t;
    r[k] ^= t << 4;
  }
#pragma unroll
  for (int k = 0; k < 8; k += 4)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t t = ((r[k + q] >> 8) ^ r[k + q + 2]) & 0x00FF00FFu;
      r[k + q + 2] ^= t;
      r[k + q] ^= t << 8;
    }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t t = ((r[q] >> 16) ^ r[q + 4]) & 0x0000FFFFu;
    r[q + 4] ^= t;
    r[q] ^= t << 16;
  }
}

// INT4 V codes of one group into the block image: lane t holds its slot's
// codes as nibbles of cw[o] (channels 32gr + 8o + n); word (channel, slot chunk j) gets
// slots 8j .. 8j + 7 in nibbles 0..7.  `wbuf`: 128 words of the warp's own
// shared memory.
__device__ __forceinline__ void store_i4v_group(uint8_t* img, const uint32_t (&cw)[4], int gr, uint32_t* wbuf) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 0; o < 4; ++o) wbuf[32 * o + lane] = cw[o];   // channels 8o .. 8o+7 of slot lane, as nibbles
  __syncwarp();
  if (lane < 16) {
    const int o = lane >> 2, j = lane & 3;
    const uint4 a = *reinterpret_cast<const uint4*>(wbuf + 32 * o + 8 * j);
    const uint4 b = *reinterpret_cast<const uint4*>(wbuf + 32 * o + 8 * j + 4);
    uint32_t r[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};   // row k = slot 8j + k
    transpose_nib8x8(r);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<uint32_t*>(img + i4v_byte(8 * j, 32 * gr + 8 * o + k)) = r[k];
  }
  __syncwarp();
}

// INT4 quantization of one token's group (K or V): the metadata and the codes
// as nibble words cw[q] (channels 8q .. 8q + 7 of the group in nibbles 0..7).
__device__ __forceinline__ GroupMeta quant_i4_words(const uint32_t (&w)[16], uint32_t (&cw)[4], bool& bad) {
  const GroupMeta m = meta_i4(w, bad);
  const float rs = approx_rcp(m.sf);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float x[8], c[8];
    bf8(w, q, x);
    codes8<15>(x, m, rs, c);
    cw[q] = pack_nib8(c);
  }
  return m;
}
// fmaf(code, scale, zero) of the 8 nibbles of a code word
__device__ __forceinline__ void deq8(uint32_t cw, const GroupMeta& m, float (&y)[8]) {
#pragma unroll
  for (int n = 0; n < 8; ++n) y[n] = __fmaf_rn((float)((cw >> (4 * n)) & 15u), m.sf, m.zf);
}

// Fresh INT4 pages filled with 32 tokens within one call.  Grid (jobs, kv heads).
__global__ void __launch_bounds__(kBulkThreads, 8) bulk_int4_kernel(
    uint8_t* __restrict__ pool, size_t int4_off, int64_t n2, int hkv, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const AppendJob* __restrict__ jobs, const int32_t* __restrict__ toks,
    Entry* __restrict__ table, int32_t* __restrict__ ntab, uint32_t* __restrict__ status) {
  __shared__ __align__(16) uint8_t img[kInt4Block];
  __shared__ __align__(16) uint32_t wbuf[4][128];
  asm volatile("griddepcontrol.wait;" ::: "memory");   // token lists and earlier stream work are done
  asm volatile("griddepcontrol.launch_dependents;");
  const AppendJob job = jobs[blockIdx.x];
  const int h = blockIdx.y, gr = threadIdx.x >> 5, t = threadIdx.x & 31;
  const int T = toks[job.tok_off + t];
  bool bad = false;
  {
    // K: slot t's row, words (i, gr) i = 0..3 hold channels 32gr + 8i + n in nibble n
    uint32_t w[16], cw[4];
    load_group(k, T, h, hkv, gr, w);
    const GroupMeta m = quant_i4_words(w, cw, bad);
#pragma unroll
    for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(img + kI4KCodes + 64 * t + 16 * i + 4 * gr) = cw[i];
    *reinterpret_cast<uint32_t*>(img + kI4KMeta + 16 * t + 4 * gr) =
        (uint32_t)__half_as_ushort(m.s) | ((uint32_t)__half_as_ushort(m.z) << 16);
  }
  {
    uint32_t w[16], cw[4];
    load_group(v, T, h, hkv, gr, w);
    const GroupMeta m = quant_i4_words(w, cw, bad);
    store_i4v_group(img, cw, gr, wbuf[gr]);
    st_half(img, kI4VMeta + 2 * v_meta_index(t, gr), m.s);
    st_half(img, kI4VMeta + 256 + 2 * v_meta_index(t, gr), m.z);
    flush_vmax(m.sf, status);
  }
  if (__any_sync(0xFFFFFFFFu, bad) && t == 0) atomicOr(status, kStatusRange);
  __syncthreads();
  uint4* out4 = reinterpret_cast<uint4*>(pool + int4_off + ((size_t)(job.page - n2) * hkv + h) * kInt4Block);
  const uint4* img4 = reinterpret_cast<const uint4*>(img);
  for (int x = threadIdx.x; x < kInt4Block / 16; x += kBulkThreads) out4[x] = img4[x];
  if (h == 0 && threadIdx.x == 0) {
    if (job.tab_index >= 0) table[job.tab_index] = Entry{job.page, job.live};
    if (job.ntab_req >= 0) ntab[job.ntab_req] = job.ntab_len;
  }
}

// Direct INT2 groups: 32 tokens that fill a staging page within one call,
// quantized to INT4 (per token and group), dequantized with fmaf(code, scale,
// zero) and requantized to INT2: K per channel across the 32 tokens, V per
// token and group.  Only the INT2 block is written.  Grid (jobs, kv heads).
// Launched as a programmatic dependent of the INT4 kernels, as the
// warp-per-token direct kernel is (it touches nothing they write).
__global__ void __launch_bounds__(kBulkThreads, 6) bulk_int2_kernel(
    uint8_t* __restrict__ pool, int hkv, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const DirectJob* __restrict__ jobs, const int32_t* __restrict__ toks, uint32_t* __restrict__ status) {
  __shared__ __align__(16) uint8_t img[kInt2Block];
  __shared__ __align__(16) float4 kmeta[4][32];          // per channel of the warp's group: zero, 1/scale, scale, nz
  __shared__ __align__(16) uint32_t vbuf[4][32][3];      // INT2 V codes [slot][channels 0..15, 16..31] (padded)
  const DirectJob job = jobs[blockIdx.x];
  const int h = blockIdx.y, gr = threadIdx.x >> 5, t = threadIdx.x & 31;
  const int T = toks[job.tok_off + t];
  bool bad = false;
  // ---- K: INT4 per token, dequantized, then INT2 per channel across the 32 slots
  {
    float xq[32];   // INT4-dequantized K of slot t's group
    {
      uint32_t w[16], cw[4];
      load_group(k, T, h, hkv, gr, w);
      const GroupMeta m = quant_i4_words(w, cw, bad);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float y[8];
        deq8(cw[q], m, y);
#pragma unroll
        for (int n = 0; n < 8; ++n) xq[8 * q + n] = y[n];
      }
    }
    float my_mn = 0.0f, my_mx = 0.0f;   // channel t of the group: min / max over the 32 slots
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float a = redux_min(xq[c]), b = redux_max(xq[c]);
      my_mn = t == c ? a : my_mn;
      my_mx = t == c ? b : my_mx;
    }
    const GroupMeta m2 = make_meta(my_mn, my_mx, 3.0f);
    kmeta[gr][t] = make_float4(m2.zf, approx_rcp(m2.sf), m2.sf, m2.nz ? 1.0f : 0.0f);
    const int ch = 32 * gr + t;
    st_half(img, kI2KMeta + 2 * i2k_meta_index(ch), m2.s);
    st_half(img, kI2KMeta + 256 + 2 * i2k_meta_index(ch), m2.z);
    float smx = m2.sf;
#pragma unroll
    for (int o = 16; o; o >>= 1) smx = fmaxf(smx, __shfl_xor_sync(0xFFFFFFFFu, smx, o));
    if (t == 0) atomicMax(status + 1, __float_as_uint(smx));
    __syncwarp();
    // slot t's codes, channel c with channel c's metadata (the repack's rule per element)
    uint32_t row[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float c2[8];
      bool tie = false;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float4 mm = kmeta[gr][8 * q + n];
        const float u = __fsub_rn(xq[8 * q + n], mm.x);
        const float q0 = u * mm.y;
        const float r = rintf(q0);
        tie |= mm.w != 0.0f && !(fabsf(fabsf(q0 - r) - 0.5f) > 1e-5f);
        c2[n] = mm.w != 0.0f ? fminf(fmaxf(r, 0.0f), 3.0f) : 0.0f;
      }
      if (tie) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const float4 mm = kmeta[gr][8 * q + n];
          const float u = __fsub_rn(xq[8 * q + n], mm.x);
          const float q0 = u * mm.y;
          float r = rintf(q0);
          if (!(fabsf(fabsf(q0 - r) - 0.5f) > 1e-5f)) r = rintf(__fdiv_rn(u, mm.z));
          c2[n] = mm.w != 0.0f ? fminf(fmaxf(r, 0.0f), 3.0f) : 0.0f;
        }
      }
      row[q >> 1] |= pack_crumb8(c2) << (16 * (q & 1));
    }
    // slot t's row: channel c at byte c >> 2, bits 2 (c & 3): the group's 8 bytes
    *reinterpret_cast<uint2*>(img + kI2KCodes + 32 * t + 8 * gr) = make_uint2(row[0], row[1]);
  }
  // ---- V: INT4 per token, then INT2 per token on the dequantized values
  {
    uint32_t cw[4];
    GroupMeta m;
    {
      uint32_t w[16];
      load_group(v, T, h, hkv, gr, w);
      m = quant_i4_words(w, cw, bad);
    }
    flush_vmax(m.sf, status);   // the INT4 V scales count toward the pool's V-scale maximum too
    float mn = 0.0f, mx = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float y[8];
      deq8(cw[q], m, y);
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        mn = (q == 0 && n == 0) ? y[0] : fminf(mn, y[n]);
        mx = (q == 0 && n == 0) ? y[0] : fmaxf(mx, y[n]);
      }
    }
    const GroupMeta m2 = make_meta(mn, mx, 3.0f);
    const float rs2 = approx_rcp(m2.sf);
    uint32_t row[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float y[8], c2[8];
      deq8(cw[q], m, y);
      codes8<3>(y, m2, rs2, c2);
      row[q >> 1] |= pack_crumb8(c2) << (16 * (q & 1));
    }
    st_half(img, kI2VMeta + 2 * v_meta_index(t, gr), m2.s);
    st_half(img, kI2VMeta + 256 + 2 * v_meta_index(t, gr), m2.z);
    float vmx = m2.sf;
#pragma unroll
    for (int o = 16; o; o >>= 1) vmx = fmaxf(vmx, __shfl_xor_sync(0xFFFFFFFFu, vmx, o));
    if (t == 0) atomicMax(status + 2, __float_as_uint(vmx));
    // codes [slot][channels 0..15, 16..31] as 2-bit fields
    vbuf[gr][t][0] = row[0];
    vbuf[gr][t][1] = row[1];
  }
  __syncwarp();
  // INT2 V bytes: lane = channel cc of the group; the 4 slot chunks i
  {
    const int c = 32 * gr + t;
    const int wsel = t >> 4, sh = 2 * (t & 15);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int b0 = i2v_byte(8 * i, c);
      int b1 = b0;
      uint32_t v0 = 0u, v1 = 0u;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int tt = 8 * i + kk, b = i2v_byte(tt, c);
        const uint32_t code = ((vbuf[gr][tt][wsel] >> sh) & 3u) << i2v_shift(tt);
        if (b == b0) v0 |= code;
        else { v1 |= code; b1 = b; }
      }
      img[b0] = (uint8_t)v0;
      img[b1] = (uint8_t)v1;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && t == 0) atomicOr(status, kStatusRange);
  __syncthreads();
  uint4* out4 = reinterpret_cast<uint4*>(pool + ((size_t)job.dst * hkv + h) * kInt2Block);
  const uint4* img4 = reinterpret_cast<const uint4*>(img);
  for (int x = threadIdx.x; x < kInt2Block / 16; x += kBulkThreads) out4[x] = img4[x];
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

cudaError_t launch_append_int3(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                               const int32_t* d_toks, cudaStream_t s) {
  if (n_jobs <= 0) return cudaSuccess;
  ++P->launches;
  return launch_pdl(append_int3_kernel, dim3((unsigned)n_jobs, (unsigned)P->cfg.num_kv_heads), dim3(kThreads), 0, s,
                    P->d_pool, P->int3_offset, (int64_t)(P->cfg.n_int2_pages + P->cfg.n_int4_pages),
                    P->cfg.num_kv_heads, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, d_jobs, d_toks,
                    P->d_table, P->d_ntab, P->d_status);
}

cudaError_t launch_append_fp4(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                              const int32_t* d_toks, cudaStream_t s) {
  if (n_jobs <= 0) return cudaSuccess;
  ++P->launches;
  return launch_pdl(append_fp4_kernel, dim3((unsigned)n_jobs, (unsigned)P->cfg.num_kv_heads), dim3(kThreads), 0, s,
                    P->d_pool, P->fp4_offset,
                    (int64_t)(P->cfg.n_int2_pages + P->cfg.n_int4_pages + P->cfg.n_int3_pages), P->cfg.num_kv_heads,
                    (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, d_jobs, d_toks, P->d_table, P->d_ntab,
                    P->d_status);
}

cudaError_t launch_bulk_int4(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                             const int32_t* d_toks, cudaStream_t s) {
  if (n_jobs <= 0) return cudaSuccess;
  ++P->launches;
  return launch_pdl(bulk_int4_kernel, dim3((unsigned)n_jobs, (unsigned)P->cfg.num_kv_heads), dim3(kBulkThreads), 0,
                    s, P->d_pool, P->int4_offset, P->cfg.n_int2_pages, P->cfg.num_kv_heads, (const __nv_bfloat16*)k,
                    (const __nv_bfloat16*)v, d_jobs, d_toks, P->d_table, P->d_ntab, P->d_status);
}

cudaError_t launch_bulk_int2(kv_pool* P, const void* k, const void* v, const DirectJob* d_jobs, int n_jobs,
                             const int32_t* d_toks, cudaStream_t s) {
  if (n_jobs <= 0) return cudaSuccess;
  ++P->launches;
  return launch_pdl(bulk_int2_kernel, dim3((unsigned)n_jobs, (unsigned)P->cfg.num_kv_heads), dim3(kBulkThreads), 0,
                    s, P->d_pool, P->cfg.num_kv_heads, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, d_jobs, d_toks,
                    P->d_status);
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
