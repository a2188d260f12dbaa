// Tensor-core split decode (mma.sync m16n8k16, fp16 inputs, fp32 accumulate).
//
// What it computes is the same as the CUDA-core kernel: per split (a page
// range of one (batch row, kv head) unit, one precision), the online-softmax
// state (m, l, acc) of the g packed query heads over dequantized K and V
// (TriAxialKV key design 4: fused Flash-Decoding with in-kernel dequant;
// HyQuant Algorithm 3: split-K, GQA query packing, ReduceSoftmax merge), with
// dead slots at logit -1e4 and V = 0 (IntentKV sentinel dead slot).
//
// How it computes it (the arithmetic is regrouped, not changed):
//  * A code word unpacks into mma A registers with one shift and one AND per
//    register: a 2- or 4-bit field at bits p.. of both 16-bit halves (zero
//    elsewhere) is the binary16 subnormal code * 2^(p-24).  The tensor core
//    keeps full precision for subnormal operands whose top set bit is at bit
//    7 or above, so fields sit at p = 6 or 8 (2-bit) and p = 4 or 6 (4-bit).
//    The factor 2^(6-p) is carried by the other operand (q fragments, or P
//    for INT2 V slot pairs at p = 8), and the common 2^-18 by the fp32 scale
//    applied to the sums.
//  * K dot products: s_t = sum_c q_c (scale * code_tc + zero).
//      INT4 K (per-token groups): per-group accumulators, scale applied per
//      token in fp32 afterwards, zero term sum_g zero_tg * Q_g by a small mma.
//      INT2 K (per-channel groups): the channel scale is folded into q as an
//      exact fp16 pair q*s = hi + lo (hi = rn(q*s), lo = fma(q, s, -hi)); the
//      zero term sum_c q_c zero_c is one fp32 dot product per page.
//  * P.V: out_c = sum_t p_t (scale_tg code_tc + zero_tg); p_t * scale_tg is
//      folded as an fp16 pair (p = p_hi + p_lo, then p_hi*s exactly and p_lo*s
//      rounded); the zero term sum_t p_t zero_tg is a small mma.
//  * For g <= 4 the eight N columns are (head, part) pairs: hi / lo of the
//    exact split (INT2 K, P.V) or even / odd channel group (INT4 K), so one
//    mma does both parts and each lane owns one head; for g > 4 hi and lo
//    are two mmas.
//  * q is scaled by a power of two per head so that q * scale stays inside
//    the binary16 range, and P by a power of two so that P * scale stays out
//    of the subnormal range (the pool tracks the largest INT2 K and V scales).
// Work layout: every warp is an independent worker.  The plan cuts all
// (unit, page) pairs into one contiguous, equal-cost range per warp; a warp
// walks its range across unit boundaries, writes one partial (m, l, acc) per
// unit it touched and never waits for another warp.  The q fragments of a
// unit are built once per call by frag_kernel and read through L1, so a unit
// boundary costs a partial store, not a prologue.  One CTA of 16 warps per SM
// (128 registers per thread): warps of one CTA are scheduled alike, so equal
// costs give equal finish times.
// Pages stream through a two-stage per-warp ring filled by cp.async.bulk with
// mbarrier completion; the ring runs across unit boundaries.  Every wait is
// bounded and reports a timeout status.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kWarps = kMmaWarpsPerCta;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 2;
constexpr int kStageBytes = kInt4Block;
constexpr int kPartStride = kHeadDim + 4;
constexpr float kDead2 = -1.0e4f * 1.4426950408889634f;
constexpr uint32_t kSpinLimit = 1u << 22;
constexpr uint32_t kN4 = 0x00F000F0u;   // 4-bit field at bit 4 of each half
constexpr uint32_t kN6 = 0x03C003C0u;   // 4-bit field at bit 6 of each half
constexpr uint32_t kC6 = 0x00C000C0u;   // 2-bit field at bit 6 of each half
constexpr uint32_t kC8 = 0x03000300u;   // 2-bit field at bit 8 of each half
constexpr uint32_t kB8 = 0x01000100u;   // 1-bit field at bit 8 of each half (INT3 code bit 2)
constexpr float kCodeUnit = 262144.0f;  // 2^18: a field at bit 6 is code * 2^-18

// One warp's shared memory: its copy ring and its P staging buffer.  Every
// stage starts on a 16-byte boundary (bulk-copy destinations and 16-byte
// shared loads require it).
struct alignas(16) WarpSmem {
  uint8_t stage[kStages][kStageBytes];
  float pbuf[8][kPage];                // P [head][slot] of the current page; V zero terms at a flush
  unsigned long long bar[kStages];
  const uint32_t* hdead;               // exclusion words (read from here at each refill, not kept in a register)
};
static_assert(sizeof(WarpSmem) % 16 == 0 && kStageBytes % 16 == 0, "stage buffers must stay 16-byte aligned");
static_assert(kInt2Block <= kStageBytes && kInt3Block <= kStageBytes && kFp4Block <= kStageBytes,
              "every block fits a stage");

// q-side operands of one unit (batch row, kv head), built by frag_kernel.
struct alignas(16) UnitFrag {
  uint4 bq2[4][32], bqn[4][32];        // INT2 K q fragments [word / 4][lane], negated copies (lo columns)
  uint4 bq4[4][32];                    // INT4 K q fragments
  uint32_t qzh[8][kHeadDim / 2];       // 2^Ez q as binary16 pairs in the INT2 K scale/zero pair order
  float acol2[8], acol4[8];            // 2^(18 - E) * scale * log2(e) for INT2 / INT4 K pages
  float qzs[8];                        // 2^(-Ez) * scale * log2(e)
  uint32_t bz[8][4];                   // fp16 pairs: hi(Q0,Q1), hi(Q2,Q3), lo(Q0,Q1), lo(Q2,Q3) of scale*log2(e)*Q_{h,group}
  uint4 bq3[4][32];                    // INT3 K q fragments (every field at bit 6)
};
static_assert(sizeof(UnitFrag) % 16 == 0, "unit fragments are copied as 16-byte words");

// frag_kernel's shared memory
struct FragSmem {
  float qraw[8][kHeadDim];             // q (fp32) of the packed heads
  int eh2[8], eh4[8];                  // per-head power-of-two q scales E for INT2 / INT4 K pages
  UnitFrag f;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t rotr8(uint32_t x) { return __funnelshift_r(x, x, 8); }
// x << s, or x >> -s for s < 0 (s is a constant once the callers unroll)
__device__ __forceinline__ uint32_t shl_s(uint32_t x, int s) { return s >= 0 ? x << s : x >> -s; }
// An INT3 A register: the low plane shifted by sl puts the code's low bits at
// bits 6..7 of both halves, the high plane shifted by sh puts bit 2 at bit 8:
// the 3-bit code at bit 6, as an INT4 code at bit 6.
__device__ __forceinline__ uint32_t i3reg(uint32_t lo, int sl, uint32_t hi, int sh) {
  return (shl_s(lo, sl) & kC6) | (shl_s(hi, sh) & kB8);
}
// An FP4 A register: the two E2M1 codes of the low byte of x (low nibble ->
// low half) as binary16 values (exact: E2M1 values have 2 significant bits).
// FP4 products are therefore 2^18 larger than the code * 2^-18 fields of the
// integer widths; the callers rescale them in fp32.
__device__ __forceinline__ uint32_t f4reg(uint32_t x) {
  uint32_t d;
  asm("{.reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(d) : "r"(x));
  return d;
}
constexpr float kFp4Unit = 1.0f / 262144.0f;   // 2^-18: FP4 products in the integer widths' units
// INT2 code word variants: variant jj puts two 2-bit fields of each half at
// bits 6 and 8.  Scale/zero pair index (register j of the pair order) of the
// field at bit 6 and at bit 8 of variant jj.
__device__ __forceinline__ uint32_t i2_variant(uint32_t x, int jj) {
  return jj == 0 ? x : (jj == 1 ? (x >> 4) : (jj == 2 ? (x << 4) : rotr8(x)));
}
__host__ __device__ constexpr int i2_reg6(int jj) { return jj == 0 ? 3 : (jj == 1 ? 5 : (jj == 2 ? 1 : 7)); }
__host__ __device__ constexpr int i2_reg8(int jj) { return jj == 0 ? 4 : (jj == 1 ? 6 : (jj == 2 ? 2 : 0)); }
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// -x for both binary16 halves (an fp16 negation, which ptxas can fold into
// the operand of the instruction that consumes it)
__device__ __forceinline__ uint32_t hneg2(uint32_t x) {
  uint32_t d;
  asm("neg.f16x2 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}
// pack two floats as binary16 (round to nearest even): lo -> bits 0..15
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// binary16 halves of a 32-bit register as fp32 (exact)
__device__ __forceinline__ float h_lo(uint32_t x) {
  float f;
  asm("{.reg .f16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, l;}" : "=f"(f) : "r"(x));
  return f;
}
__device__ __forceinline__ float h_hi(uint32_t x) {
  float f;
  asm("{.reg .f16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, h;}" : "=f"(f) : "r"(x));
  return f;
}
// acc + lo(a) * lo(b) + hi(a) * hi(b): binary16 products are exact in fp32,
// each addition rounds once.
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .f16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.f16 %0, al, bl, %0;\n fma.rn.f32.f16 %0, ah, bh, %0;}"
      : "+f"(acc) : "r"(a), "r"(b));
  return acc;
}
// 2^x (flushes results below 2^-126 to zero; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// x * 2^e for |e| <= 126, rounded once (as ldexpf): 2^e is a normal float
__device__ __forceinline__ float pow2_scale(float x, int e) { return x * __int_as_float((e + 127) << 23); }
__device__ __forceinline__ uint32_t comp(const uint4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}
// Packed fp32 pairs (one f32x2 instruction for two IEEE operations, each
// rounded as its scalar form): (a0, a1) += (b0, b1), (a0, a1) *= (b0, b1),
// (a0 - b0, a1 - b1).
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{.reg .b64 x, y;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n add.rn.f32x2 x, x, y;\n"
      " mov.b64 {%0, %1}, x;}"
      : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2(float& a0, float& a1, float b0, float b1) {
  asm("{.reg .b64 x, y;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n mul.rn.f32x2 x, x, y;\n"
      " mov.b64 {%0, %1}, x;}"
      : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float a0, float a1, float b0, float b1, float& d0, float& d1) {
  asm("{.reg .b64 x, y;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n sub.rn.f32x2 x, x, y;\n"
      " mov.b64 {%0, %1}, x;}"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// exact fp16 pair of the fp32 product x: hi = rn16(x), lo = rn16(x - hi)
__device__ __forceinline__ void split_f16(float x, unsigned short& hi, unsigned short& lo) {
  const __half h = __float2half_rn(x);
  hi = __half_as_ushort(h);
  lo = __half_as_ushort(__float2half_rn(x - __half2float(h)));
}

// ---- bulk copy + mbarrier (bounded waits) --------------------------------
__device__ __forceinline__ void bar_init(unsigned long long* b) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, unsigned long long* b) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(su32(dst)), "l"(src), "r"(bytes), "r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool bar_try(unsigned long long* b, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(su32(b)), "r"(phase) : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool bar_wait(unsigned long long* b, uint32_t phase, uint32_t limit = kSpinLimit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (bar_try(b, phase)) return true;
  return false;
}

// Lanes and heads.  A lane is (r, i) = (lane >> 2, lane & 3); its C fragment
// holds rows r and r + 8 of columns 2i and 2i + 1.  For g <= 4 ("paired
// columns") the eight N columns are (head, part) pairs, column n = 2 * head +
// part, where part is hi / lo of an exact fp16 split (INT2 K, P.V) or the
// even / odd channel group (INT4 K): lane (r, i) then owns head i and both
// parts meet in its registers.  For g > 4 the columns are heads and a lane
// owns heads 2i and 2i + 1.  NH = heads per lane.
template <int G>
struct Cols {
  static constexpr bool kPair = G <= 4;
  static constexpr int NH = kPair ? 1 : 2;
};

// ---- logits of one INT4 (kI3: INT3) page: lg[m][e][hh] for token 16m + r + 8e
// and the lane's head hh (log2 units, scale folded in).  An INT3 page has the
// INT4 page's per-token groups and scale/zero; only its code words differ.
template <int G, bool kI3 = false, bool kF4 = false>
__device__ __forceinline__ void qk_int4(const uint8_t* blk, const uint4* bq4, const uint32_t (&bz)[2],
                                        const float (&acol)[Cols<G>::NH], float (&lg)[2][2][Cols<G>::NH]) {
  constexpr bool kPair = Cols<G>::kPair;
  const int lane = threadIdx.x & 31, r = lane >> 2, i = lane & 3;
  uint32_t bq[16];
#pragma unroll
  for (int x4 = 0; x4 < 4; ++x4) {
    const uint4 b = __ldg(&bq4[x4 * 32 + lane]);
    bq[4 * x4] = b.x; bq[4 * x4 + 1] = b.y; bq[4 * x4 + 2] = b.z; bq[4 * x4 + 3] = b.w;
  }
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    uint4 kw[2], km[2];
    uint2 kl[2], ks[2];
    uint32_t kh[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 16 * m + r + 8 * e;
      if constexpr (kF4) {
        kw[e] = *reinterpret_cast<const uint4*>(blk + kF4KCodes + 64 * t + 16 * i);
        ks[e] = *reinterpret_cast<const uint2*>(blk + kF4KScale + 8 * t);
      } else if constexpr (kI3) {
        kl[e] = *reinterpret_cast<const uint2*>(blk + kI3KCodes + 48 * t + 8 * i);
        kh[e] = *reinterpret_cast<const uint32_t*>(blk + kI3KCodes + 48 * t + 32 + 4 * i);
        km[e] = *reinterpret_cast<const uint4*>(blk + kI3KMeta + 16 * t);
      } else {
        kw[e] = *reinterpret_cast<const uint4*>(blk + kI4KCodes + 64 * t + 16 * i);
        km[e] = *reinterpret_cast<const uint4*>(blk + kI4KMeta + 16 * t);
      }
    }
    // Group gr's k-steps: nibbles 0/4 at p = 6, 1/5 at p = 4, then 2/6 and 3/7 at p = 6.
    // INT3: channels n / n + 4 at p = 6 for every n (the q fragments carry no 2^2).
    auto group_mma = [&](float (&acc)[4], int gr) {
      if constexpr (kF4) {
        // FP4: byte n of a word holds channels n and n + 4
        const uint32_t x0 = comp(kw[0], gr), x1 = comp(kw[1], gr);
        mma16816(acc, f4reg(x0), f4reg(x1), f4reg(x0 >> 8), f4reg(x1 >> 8), bq[4 * gr], bq[4 * gr + 1]);
        mma16816(acc, f4reg(x0 >> 16), f4reg(x1 >> 16), f4reg(x0 >> 24), f4reg(x1 >> 24), bq[4 * gr + 2],
                 bq[4 * gr + 3]);
      } else if constexpr (kI3) {
        const uint32_t l0 = gr < 2 ? kl[0].x : kl[0].y, l1 = gr < 2 ? kl[1].x : kl[1].y;
        const int o = 8 * (gr & 1);
        auto reg = [&](uint32_t l, uint32_t h, int n) { return i3reg(l, 6 - o - 2 * n, h, 8 - 4 * gr - n); };
        mma16816(acc, reg(l0, kh[0], 0), reg(l1, kh[1], 0), reg(l0, kh[0], 1), reg(l1, kh[1], 1), bq[4 * gr],
                 bq[4 * gr + 1]);
        mma16816(acc, reg(l0, kh[0], 2), reg(l1, kh[1], 2), reg(l0, kh[0], 3), reg(l1, kh[1], 3), bq[4 * gr + 2],
                 bq[4 * gr + 3]);
      } else {
        const uint32_t x0 = comp(kw[0], gr), x1 = comp(kw[1], gr);   // tokens r, r + 8
        mma16816(acc, (x0 << 6) & kN6, (x1 << 6) & kN6, x0 & kN4, x1 & kN4, bq[4 * gr], bq[4 * gr + 1]);
        mma16816(acc, (x0 >> 2) & kN6, (x1 >> 2) & kN6, (x0 >> 6) & kN6, (x1 >> 6) & kN6, bq[4 * gr + 2],
                 bq[4 * gr + 3]);
      }
    };
    // zero term sum_g zero_tg * (scale log2e Q_g) by one mma: every lane feeds
    // (zero_0, zero_1) in k-slots 2i, 2i+1 and (zero_2, zero_3) in 2i+8, 2i+9;
    // B rows 0, 1 / 8, 9 hold the hi parts of Q, rows 2, 3 / 10, 11 the lo
    // parts, the other rows zero.  FP4 groups have no zero point.
    uint32_t az0 = 0u, az1 = 0u, az2 = 0u, az3 = 0u;
    if constexpr (!kF4) {
      az0 = __byte_perm(km[0].x, km[0].y, 0x7632); az2 = __byte_perm(km[0].z, km[0].w, 0x7632);
      az1 = __byte_perm(km[1].x, km[1].y, 0x7632); az3 = __byte_perm(km[1].z, km[1].w, 0x7632);
    }
    // the scale of group gr of token e (FP4: the products carry 2^18 more)
    auto ksc = [&](int e, int gr) -> float {
      if constexpr (kF4) {
        const uint32_t w = gr < 2 ? ks[e].x : ks[e].y;
        return ((gr & 1) ? h_hi(w) : h_lo(w)) * kFp4Unit;
      } else {
        return h_lo(comp(km[e], gr));
      }
    };
    if constexpr (kPair) {
      // acc[0]: groups 0 / 1 in columns 2h / 2h+1, acc[1]: groups 2 / 3
      float acc[2][4];
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        acc[pr][0] = acc[pr][1] = acc[pr][2] = acc[pr][3] = 0.0f;
        group_mma(acc[pr], 2 * pr);
        group_mma(acc[pr], 2 * pr + 1);
      }
      float T[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = ksc(e, 0) * acc[0][2 * e];
        v = fmaf(ksc(e, 1), acc[0][2 * e + 1], v);
        v = fmaf(ksc(e, 2), acc[1][2 * e], v);
        v = fmaf(ksc(e, 3), acc[1][2 * e + 1], v);
        T[2 * e] = v * acol[0];
      }
      if constexpr (!kF4) mma16816(T, az0, az1, az2, az3, bz[0], bz[1]);   // B: even columns only
      lg[m][0][0] = T[0];
      lg[m][1][0] = T[2];
    } else {
      float acc[4][4];
#pragma unroll
      for (int gr = 0; gr < 4; ++gr) {
        acc[gr][0] = acc[gr][1] = acc[gr][2] = acc[gr][3] = 0.0f;
        group_mma(acc[gr], gr);
      }
      float T[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = c >> 1;
        float v = 0.0f;
#pragma unroll
        for (int gr = 0; gr < 4; ++gr) v = fmaf(ksc(e, gr), acc[gr][c], v);
        T[c] = v * acol[c & 1];
      }
      if constexpr (!kF4) mma16816(T, az0, az1, az2, az3, bz[0], bz[1]);
#pragma unroll
      for (int c = 0; c < 4; ++c) lg[m][c >> 1][c & 1] = T[c];
    }
  }
}

// ---- logits of one INT2 page (same layout as qk_int4)
template <int G>
__device__ __forceinline__ void qk_int2(const uint8_t* blk, const UnitFrag* __restrict__ F,
                                        const float (&acol)[Cols<G>::NH], float (&lg)[2][2][Cols<G>::NH],
                                        float (&zc)[Cols<G>::NH]) {
  constexpr bool kPair = Cols<G>::kPair;
  const int lane = threadIdx.x & 31, r = lane >> 2, i = lane & 3;
  uint2 kw[2][2];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      kw[m][e] = *reinterpret_cast<const uint2*>(blk + kI2KCodes + 32 * (16 * m + r + 8 * e) + 8 * i);
  uint4 sv[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) sv[x] = *reinterpret_cast<const uint4*>(blk + kI2KMeta + 64 * i + 16 * x);
  // two accumulators per M tile so that consecutive mmas do not wait on each
  // other (g <= 4: alternating k-steps; g > 4: the hi and the lo pass)
  float acc[2][2][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int x = 0; x < 2; ++x) acc[m][x][0] = acc[m][x][1] = acc[m][x][2] = acc[m][x][3] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int wi = kk >> 2, jj = kk & 3;
    const int p0 = wi * 8 + i2_reg6(jj), p1 = wi * 8 + i2_reg8(jj);
    const uint32_t s0 = comp(sv[p0 >> 2], p0 & 3), s1 = comp(sv[p1 >> 2], p1 & 3);
    const uint4 qq = __ldg(&F->bq2[kk >> 1][lane]);
    const uint32_t q0 = (kk & 1) ? qq.z : qq.x, q1 = (kk & 1) ? qq.w : qq.y;
    // hi = rn(q s); lo = q s - hi (exact: the rounding error of an fp16 product)
    uint32_t b0, b1, u0, u1;
    if constexpr (kPair) {
      // bqn holds -q where the lo part is wanted and 0 elsewhere, so
      // u = fma(q, s, rn(bqn s)) is lo or hi
      const uint4 nq = __ldg(&F->bqn[kk >> 1][lane]);
      const uint32_t n0 = (kk & 1) ? nq.z : nq.x, n1 = (kk & 1) ? nq.w : nq.y;
      u0 = hfma2(q0, s0, hmul2(n0, s0));
      u1 = hfma2(q1, s1, hmul2(n1, s1));
      b0 = b1 = 0u;
    } else {
      // lo = fma(q, s, -hi)
      b0 = hmul2(q0, s0);
      b1 = hmul2(q1, s1);
      u0 = hfma2(q0, s0, hneg2(b0));
      u1 = hfma2(q1, s1, hneg2(b1));
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t x0 = i2_variant(wi ? kw[m][0].y : kw[m][0].x, jj);   // token 16m + r
      const uint32_t x1 = i2_variant(wi ? kw[m][1].y : kw[m][1].x, jj);   // token 16m + r + 8
      const uint32_t a0 = x0 & kC6, a1 = x1 & kC6, a2 = x0 & kC8, a3 = x1 & kC8;
      if constexpr (kPair) {
        mma16816(acc[m][kk & 1], a0, a1, a2, a3, u0, u1);
      } else {
        mma16816(acc[m][0], a0, a1, a2, a3, b0, b1);
        mma16816(acc[m][1], a0, a1, a2, a3, u0, u1);
      }
    }
  }
  // zero term Z_h = sum_c q_hc zero_c (fp32 sums of exact binary16 products),
  // returned per head (the softmax adds it to the page's logits as a scalar,
  // so its reduction overlaps the max reduction instead of preceding it)
  if constexpr (kPair) {
    // lane (r, i) sums head i over scale/zero pairs 8r .. 8r+7; the lanes of
    // one head (r = 0..7) reduce, and every lane ends with its own head's Z
    const uint4* zs = reinterpret_cast<const uint4*>(blk + kI2KMeta + 256 + 32 * r);
    const uint4* qs = reinterpret_cast<const uint4*>(&F->qzh[i][8 * r]);
    float zq[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // independent partial sums
#pragma unroll
    for (int x4 = 0; x4 < 2; ++x4) {
      const uint4 zz = zs[x4], qz = __ldg(&qs[x4]);
      zq[0] = fma2_f16_f32(zz.x, qz.x, zq[0]);
      zq[1] = fma2_f16_f32(zz.y, qz.y, zq[1]);
      zq[2] = fma2_f16_f32(zz.z, qz.z, zq[2]);
      zq[3] = fma2_f16_f32(zz.w, qz.w, zq[3]);
    }
    float zp = (zq[0] + zq[1]) + (zq[2] + zq[3]);
    zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 4);
    zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 8);
    zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 16);
    zc[0] = zp * __ldg(&F->qzs[i]);
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = (acc[m][0][2 * e] + acc[m][0][2 * e + 1]) + (acc[m][1][2 * e] + acc[m][1][2 * e + 1]);
        lg[m][e][0] = acol[0] * v;
      }
  } else {
    // lane (r, i) sums head r over chunk i; the 4 lanes of a head reduce and
    // the lanes of heads 2i, 2i+1 fetch theirs
    const uint4* zs = reinterpret_cast<const uint4*>(blk + kI2KMeta + 256 + 64 * i);
    const uint4* qs = reinterpret_cast<const uint4*>(&F->qzh[r][i * 16]);
    float zq[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // independent partial sums
#pragma unroll
    for (int x4 = 0; x4 < 4; ++x4) {
      const uint4 zz = zs[x4], qz = __ldg(&qs[x4]);
      zq[0] = fma2_f16_f32(zz.x, qz.x, zq[0]);
      zq[1] = fma2_f16_f32(zz.y, qz.y, zq[1]);
      zq[2] = fma2_f16_f32(zz.z, qz.z, zq[2]);
      zq[3] = fma2_f16_f32(zz.w, qz.w, zq[3]);
    }
    float zp = (zq[0] + zq[1]) + (zq[2] + zq[3]);
    zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 1);
    zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 2);
    zp *= __ldg(&F->qzs[r]);
    zc[0] = __shfl_sync(0xFFFFFFFFu, zp, 4 * (2 * i));
    zc[1] = __shfl_sync(0xFFFFFFFFu, zp, 4 * (2 * i + 1));
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) lg[m][e][hh] = acol[hh] * (acc[m][0][2 * e + hh] + acc[m][1][2 * e + hh]);
  }
}

// ---- online softmax update and P.V for one page (any width; kInt3: an INT3
// page, read as an INT4 page with INT3 code words)
template <int G, bool kInt2, bool kInt3 = false, bool kFp4 = false>
__device__ __forceinline__ void softmax_pv(const uint8_t* blk, uint32_t live, float pscale,
                                           float (&lg)[2][2][Cols<G>::NH], const float (&zc)[Cols<G>::NH],
                                           float (&o)[8][4], float (&zv)[4],
                                           float (&mrun)[Cols<G>::NH], float (&lsum)[Cols<G>::NH],
                                           float (*pbuf)[kPage]) {
  constexpr bool kPair = Cols<G>::kPair;
  constexpr int NH = Cols<G>::NH;
  constexpr int vmeta = kInt2 ? kI2VMeta : (kInt3 ? kI3VMeta : (kFp4 ? kF4VScale : kI4VMeta));
  const int lane = threadIdx.x & 31, r = lane >> 2, i = lane & 3;
  const bool full = live == 0xFFFFFFFFu;   // warp-uniform: no dead slot on this page
  if (!full) {
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (!((live >> (16 * m + r + 8 * e)) & 1u))
#pragma unroll
          for (int hh = 0; hh < NH; ++hh) lg[m][e][hh] = kDead2 - zc[hh];
  }
  // the page's logits are lg + zc (zc: a per-head constant of the page)
  float corr[NH], pv[2][2][NH];
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) {
    float pm = fmaxf(fmaxf(lg[0][0][hh], lg[0][1][hh]), fmaxf(lg[1][0][hh], lg[1][1][hh]));
    pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 16));
    const float mnew = fmaxf(mrun[hh], pm + zc[hh]);
    corr[hh] = ex2(mrun[hh] - mnew);
    mrun[hh] = mnew;
    const float mo = mnew - zc[hh];
    float ps = 0.0f;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pv[m][e][hh] = ex2(lg[m][e][hh] - mo);
        ps += pv[m][e][hh];
      }
    lsum[hh] = lsum[hh] * corr[hh] + ps;
  }
  if (!full) {   // dead slots carry V = 0
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (!((live >> (16 * m + r + 8 * e)) & 1u))
#pragma unroll
          for (int hh = 0; hh < NH; ++hh) pv[m][e][hh] = 0.0f;
  }
  {
    // INT2 V: even slots pair with code fields at p = 8, so their P carries 2^-2
    const float pmul = (kInt2 && !(r & 1)) ? 0.25f * pscale : pscale;
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      const int h = kPair ? i : 2 * i + hh;
      if (h < G)
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int e = 0; e < 2; ++e) pbuf[h][16 * m + r + 8 * e] = pv[m][e][hh] * pmul;
    }
  }
  const float c0 = corr[0], c1 = corr[NH - 1];
  if (__any_sync(0xFFFFFFFFu, c0 != 1.0f || c1 != 1.0f)) {
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      mul2(o[m][0], o[m][1], c0, c1);
      mul2(o[m][2], o[m][3], c0, c1);
    }
    mul2(zv[0], zv[1], c0, c1);
    mul2(zv[2], zv[3], c0, c1);
  }
  __syncwarp();

  // B operands: p of the head of column r at slots 8i..8i+7, pairs (8i+k, 8i+k+4)
  const int hp = kPair ? (r >> 1) : r;
  const bool lo_col = kPair && (r & 1);
  const float4 pa = *reinterpret_cast<const float4*>(&pbuf[hp][8 * i]);
  const float4 pb = *reinterpret_cast<const float4*>(&pbuf[hp][8 * i + 4]);
  const float pav[4] = {pa.x, pa.y, pa.z, pa.w}, pbv[4] = {pb.x, pb.y, pb.z, pb.w};
  uint32_t ph[4], pl[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ph[k] = pack_h2(pav[k], pbv[k]);
    float ra, rb;
    sub2(pav[k], pbv[k], h_lo(ph[k]), h_hi(ph[k]), ra, rb);
    pl[k] = pack_h2(ra, rb);
  }
  // V zero term: rows = groups (lanes r < 4), k = slots.  Lanes r >= 4 load
  // group r - 4 as well (no branch): their rows 4..7 of the product are
  // finite and never read (only lanes r < 4 store the zero terms).  FP4
  // groups have no zero point.
  if constexpr (!kFp4) {
    uint4 zz = *reinterpret_cast<const uint4*>(blk + vmeta + 256 + 64 * (r & 3) + 16 * i);
    if (kInt2) {   // undo the 2^-2 of the even slots' P: words 0 and 2 hold slot pairs (8i, 8i+4), (8i+2, 8i+6)
      zz.x = hmul2(zz.x, 0x44004400u);
      zz.z = hmul2(zz.z, 0x44004400u);
    }
    float zt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if constexpr (kPair) {
      mma16816(zt, zz.x, 0u, zz.y, 0u, lo_col ? pl[0] : ph[0], lo_col ? pl[1] : ph[1]);
      mma16816(zt, zz.z, 0u, zz.w, 0u, lo_col ? pl[2] : ph[2], lo_col ? pl[3] : ph[3]);
    } else {
      mma16816(zt, zz.x, 0u, zz.y, 0u, ph[0], ph[1]);
      mma16816(zt, zz.z, 0u, zz.w, 0u, ph[2], ph[3]);
      mma16816(zt, zz.x, 0u, zz.y, 0u, pl[0], pl[1]);
      mma16816(zt, zz.z, 0u, zz.w, 0u, pl[2], pl[3]);
    }
    add2(zv[0], zv[1], zt[0], zt[1]);
    add2(zv[2], zv[3], zt[2], zt[3]);
  }
  // Fold operands, hi = rn(p_hi s) and lo = rn(p_lo s + (p_hi s - hi)) (the
  // bracket is exact: the rounding error of an fp16 product).  g <= 4: one
  // B per lane, u = fma(p_hi, s, rn(x3 s)) with x3 = -p_hi in the lo columns
  // and 0 in the hi columns, then B = rn(x1 s + u) with x1 = p_lo or 0;
  // g > 4: hi and lo both, lo from -hi directly.
  uint32_t x3[4], x1[4];
  if constexpr (kPair) {
    const uint32_t lomask = lo_col ? 0xFFFFFFFFu : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x3[k] = (ph[k] ^ 0x80008000u) & lomask;   // -p_hi or 0 (one logic op)
      x1[k] = pl[k] & lomask;
    }
  }
#pragma unroll
  for (int gr = 0; gr < 4; ++gr) {
    const uint4 svv = *reinterpret_cast<const uint4*>(blk + vmeta + 64 * gr + 16 * i);
    const uint32_t sk[4] = {svv.x, svv.y, svv.z, svv.w};
    uint32_t bh[4], bl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (kPair) {
        bh[k] = hfma2(x1[k], sk[k], hfma2(ph[k], sk[k], hmul2(x3[k], sk[k])));
      } else {
        bh[k] = hmul2(ph[k], sk[k]);
        bl[k] = hfma2(pl[k], sk[k], hfma2(ph[k], sk[k], hneg2(bh[k])));
      }
    }
    uint32_t wv[4];
    uint32_t vh3 = 0u;
    if (kInt2) {
      const uint2 v2 = *reinterpret_cast<const uint2*>(blk + kI2VCodes + 16 * (32 * (gr >> 1) + 4 * r + i) + 8 * (gr & 1));
      wv[0] = v2.x; wv[1] = v2.y;
    } else if (kFp4) {
      const uint4 v4 = *reinterpret_cast<const uint4*>(blk + kF4VCodes + 16 * (32 * gr + 4 * r + i));
      wv[0] = v4.x; wv[1] = v4.y; wv[2] = v4.z; wv[3] = v4.w;
    } else if (kInt3) {
      const int X = 32 * gr + 4 * r + i;
      const uint2 v3 = *reinterpret_cast<const uint2*>(blk + kI3VCodes + 8 * X);
      wv[0] = v3.x; wv[1] = v3.y;
      vh3 = *reinterpret_cast<const uint32_t*>(blk + kI3VHigh + 4 * X);
    } else {
      const uint4 v4 = *reinterpret_cast<const uint4*>(blk + kI4VCodes + 16 * (32 * gr + 4 * r + i));
      wv[0] = v4.x; wv[1] = v4.y; wv[2] = v4.z; wv[3] = v4.w;
    }
#pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
      const int m = 2 * gr + mm;
      uint32_t a[2][4];
      if (kInt2) {
        // channel 16m+r in bytes 0/2, 16m+r+8 in bytes 1/3 (see the layout)
        const uint32_t x = wv[mm], xr = x >> 4, xl = x << 4, xo = rotr8(x);
        a[0][0] = xo & kC8; a[0][1] = x & kC8;     // slots (8i, 8i+4), p = 8
        a[0][2] = xl & kC6; a[0][3] = xr & kC6;    // slots (8i+1, 8i+5), p = 6
        a[1][0] = xl & kC8; a[1][1] = xr & kC8;    // slots (8i+2, 8i+6), p = 8
        a[1][2] = x & kC6; a[1][3] = xo & kC6;     // slots (8i+3, 8i+7), p = 6
      } else if (kFp4) {
        // slot 8i+k and 8i+k+4 of channel 16m+r (+8 for e = 1) in byte k of the word
        const uint32_t w0 = wv[2 * mm], w1 = wv[2 * mm + 1];
        a[0][0] = f4reg(w0); a[0][1] = f4reg(w1); a[0][2] = f4reg(w0 >> 8); a[0][3] = f4reg(w1 >> 8);
        a[1][0] = f4reg(w0 >> 16); a[1][1] = f4reg(w1 >> 16); a[1][2] = f4reg(w0 >> 24); a[1][3] = f4reg(w1 >> 24);
      } else if (kInt3) {
        // channel 16m+r (e = 0) and 16m+r+8 (e = 1): slot 8i+k's low bits at
        // 8e + 2k of plane word mm, bit 2 at 4(2mm + e) + k of the high word
        const uint32_t x = wv[mm];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int e = 0; e < 2; ++e) a[k >> 1][2 * (k & 1) + e] = i3reg(x, 6 - 8 * e - 2 * k, vh3, 8 - 4 * (2 * mm + e) - k);
      } else {
        // slot 8i+k in nibble k; nibbles k and k+4 moved to bit 6 of each half
        const uint32_t w0 = wv[2 * mm], w1 = wv[2 * mm + 1];   // channels 16m+r, 16m+r+8
        a[0][0] = (w0 << 6) & kN6; a[0][1] = (w1 << 6) & kN6; a[0][2] = (w0 << 2) & kN6; a[0][3] = (w1 << 2) & kN6;
        a[1][0] = (w0 >> 2) & kN6; a[1][1] = (w1 >> 2) & kN6; a[1][2] = (w0 >> 6) & kN6; a[1][3] = (w1 >> 6) & kN6;
      }
      // This page's products go to a fresh accumulator, added to the running
      // sum in fp32: the tensor core aligns products to the accumulator's
      // magnitude, so accumulating many pages in place would truncate the
      // small late contributions.
      float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      mma16816(t, a[0][0], a[0][1], a[0][2], a[0][3], bh[0], bh[1]);
      mma16816(t, a[1][0], a[1][1], a[1][2], a[1][3], bh[2], bh[3]);
      if constexpr (!kPair) {
        mma16816(t, a[0][0], a[0][1], a[0][2], a[0][3], bl[0], bl[1]);
        mma16816(t, a[1][0], a[1][1], a[1][2], a[1][3], bl[2], bl[3]);
      }
      if constexpr (kFp4) {
#pragma unroll
        for (int x = 0; x < 4; ++x) o[m][x] = fmaf(t[x], kFp4Unit, o[m][x]);
      } else {
        add2(o[m][0], o[m][1], t[0], t[1]);
        add2(o[m][2], o[m][3], t[2], t[3]);
      }
    }
  }
  __syncwarp();
}

// ---- q fragments (B operands of the K dot products), built once per unit
// INT2 K word x = 2 kk + e of lane L: k-slots of a0/a1 (e = 0) hold the field
// at bit 6, those of a2/a3 (e = 1) the field at bit 8 (factor 2^-2);
// register 0 of the pair order has its halves swapped.
template <int G>
__device__ __forceinline__ uint32_t frag_q2(const FragSmem& S, int L, int x) {
  const int r = L >> 2, i = L & 3;
  const int h = Cols<G>::kPair ? (r >> 1) : r;
  if (h >= G) return 0u;
  const int kk = x >> 1, e = x & 1, jj = kk & 3, wi = kk >> 2;
  const int j = e ? i2_reg8(jj) : i2_reg6(jj);
  const int c = 4 * (8 * i + 4 * wi + (j >> 2)) + (j & 3);
  const int clo = j == 0 ? c + 8 : c, chi = j == 0 ? c : c + 8;
  const int ex = S.eh2[h] - 2 * e;
  return pack_h2(pow2_scale(S.qraw[h][clo], ex), pow2_scale(S.qraw[h][chi], ex));
}
// INT4 K word x = 4 gr + 2 hf + e of lane L: nibbles (2hf + e, 2hf + e + 4)
// of group gr's words; the bit-4 field (hf = 0, e = 1) carries 2^2.  With
// paired columns, column 2h + part holds the groups of parity part.
template <int G>
__device__ __forceinline__ uint32_t frag_q4(const FragSmem& S, int L, int x) {
  const int r = L >> 2, i = L & 3;
  const int gr = x >> 2, hf = (x >> 1) & 1, e = x & 1;
  if (Cols<G>::kPair && (gr & 1) != (r & 1)) return 0u;
  const int h = Cols<G>::kPair ? (r >> 1) : r;
  if (h >= G) return 0u;
  const int c = 32 * gr + 8 * i + 2 * hf + e;
  const int ex = S.eh4[h] + ((hf == 0 && e == 1) ? 2 : 0);
  return pack_h2(pow2_scale(S.qraw[h][c], ex), pow2_scale(S.qraw[h][c + 4], ex));
}
// INT3 K word x: the INT4 word's channels, every field at bit 6 (no 2^2)
template <int G>
__device__ __forceinline__ uint32_t frag_q3(const FragSmem& S, int L, int x) {
  const int r = L >> 2, i = L & 3;
  const int gr = x >> 2, hf = (x >> 1) & 1, e = x & 1;
  if (Cols<G>::kPair && (gr & 1) != (r & 1)) return 0u;
  const int h = Cols<G>::kPair ? (r >> 1) : r;
  if (h >= G) return 0u;
  const int c = 32 * gr + 8 * i + 2 * hf + e;
  return pack_h2(pow2_scale(S.qraw[h][c], S.eh4[h]), pow2_scale(S.qraw[h][c + 4], S.eh4[h]));
}

// ---- per-unit q operands: one CTA of 8 warps per unit (batch row, kv head).
// It computes what the scan needs on the q side of a unit: the per-head
// power-of-two scales, the mma B fragments of both K formats, the INT2 K
// zero-term pairs and the INT4 K zero-term fragments.
template <int G>
__global__ void __launch_bounds__(256) frag_kernel(const __nv_bfloat16* __restrict__ q, int hq, float scale_log2,
                                                   const Unit* __restrict__ units,
                                                   const uint32_t* __restrict__ smax_bits,
                                                   UnitFrag* __restrict__ frags,
                                                   const GroupPool* __restrict__ gpools) {
  constexpr bool kPair = Cols<G>::kPair;
  __shared__ FragSmem S;
  // Launched as a programmatic dependent of the last kernel before the decode
  // (normally the append kernel, which signals after its own wait).  Nothing
  // it reads is written by that kernel: q and the plan are in place before
  // it, and the INT2 K scale maximum changes only in repacks, which finish
  // before their dependents start.  It waits for that grid only before it
  // exits, so the scan's wait (on this grid) covers the appends too.
  const Unit u = units[blockIdx.x];
  asm volatile("griddepcontrol.launch_dependents;");   // the scan may be staged
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  // a grouped decode: the unit's own pool bounds its INT2 K scales
  if (gpools) smax_bits = gpools[u.pad].smax;
  const float smax = fmaxf(__uint_as_float(smax_bits[0]), 1.0f);
  {
    // thread (h, 4 channels); q needs only its element alignment
    const int h = tid >> 5, c = 4 * (tid & 31);
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (h < G) {
      const __nv_bfloat16* qh = q + ((size_t)u.b * hq + (size_t)u.kvh * G + h) * kHeadDim + c;
      v = make_float4(__bfloat162float(qh[0]), __bfloat162float(qh[1]), __bfloat162float(qh[2]),
                      __bfloat162float(qh[3]));
    }
    *reinterpret_cast<float4*>(&S.qraw[h][c]) = v;
  }
  __syncthreads();
  {
    const int h = w;
    float mx = 0.0f, qg[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      qg[k] = S.qraw[h][lane + 32 * k];           // channel lane + 32k is in group k
      mx = fmaxf(mx, fabsf(qg[k]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
#pragma unroll
      for (int k = 0; k < 4; ++k) qg[k] += __shfl_xor_sync(0xFFFFFFFFu, qg[k], o);
    }
    if (lane == 0) {
      int E2 = 0, E4 = 0;
      if (mx > 0.0f) {
        // INT2 K folds q * scale: |q * scale| * 2^E2 <= 2^14
        E2 = max(-100, min(100, ilogbf(16384.0f / (mx * smax))));
        // INT4 K: |q| * 2^E4 < 2^13 (q of the bit-4 fields carries another 2^2)
        E4 = max(-100, min(100, 12 - ilogbf(mx)));
      }
      S.eh2[h] = E2;
      S.eh4[h] = E4;
      S.f.acol2[h] = pow2_scale(scale_log2, 18 - E2);
      S.f.acol4[h] = pow2_scale(scale_log2, 18 - E4);
      unsigned short hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) split_f16(scale_log2 * qg[k], hi[k], lo[k]);
      S.f.bz[h][0] = hi[0] | ((uint32_t)hi[1] << 16);
      S.f.bz[h][1] = hi[2] | ((uint32_t)hi[3] << 16);
      S.f.bz[h][2] = lo[0] | ((uint32_t)lo[1] << 16);
      S.f.bz[h][3] = lo[2] | ((uint32_t)lo[3] << 16);
    }
    // q as binary16 pairs in the INT2 K scale/zero pair order for the zero
    // term, scaled by 2^Ez so that max |q| lies in [2^14, 2^15)
    const int Ez = mx > 0.0f ? max(-100, min(100, 14 - ilogbf(mx))) : 0;
    for (int pr = lane; pr < kHeadDim / 2; pr += 32) {
      const int j = pr & 7, iw = pr >> 3;        // iw = chunk i * 2 + word wi
      const int c = 4 * (4 * iw + (j >> 2)) + (j & 3);
      const int clo = j == 0 ? c + 8 : c, chi = j == 0 ? c : c + 8;   // pair 0 is stored swapped
      S.f.qzh[h][pr] = pack_h2(pow2_scale(S.qraw[h][clo], Ez), pow2_scale(S.qraw[h][chi], Ez));
    }
    if (lane == 0) S.f.qzs[h] = pow2_scale(scale_log2, -Ez);
  }
  __syncthreads();
  {
    // q fragments of every lane: [x >> 2][lane][x & 3] for word x = 0..15
    uint32_t* f2 = reinterpret_cast<uint32_t*>(&S.f.bq2[0][0]);
    uint32_t* fn = reinterpret_cast<uint32_t*>(&S.f.bqn[0][0]);
    uint32_t* f4 = reinterpret_cast<uint32_t*>(&S.f.bq4[0][0]);
    uint32_t* f3 = reinterpret_cast<uint32_t*>(&S.f.bq3[0][0]);
    for (int y = tid; y < 16 * 32; y += 256) {
      const int x = 4 * (y >> 7) + (y & 3), L = (y >> 2) & 31;
      const uint32_t v2 = frag_q2<G>(S, L, x);
      f2[y] = v2;
      // negated copy for the exact hi/lo split (g <= 4: lo columns only)
      fn[y] = (!kPair || ((L >> 2) & 1)) ? (v2 ^ 0x80008000u) : 0u;
      f4[y] = frag_q4<G>(S, L, x);
      f3[y] = frag_q3<G>(S, L, x);
    }
  }
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(&S.f);
  uint4* dst = reinterpret_cast<uint4*>(frags + blockIdx.x);
  for (int x = tid; x < (int)(sizeof(UnitFrag) / 16); x += 256) dst[x] = src[x];
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- persistent scan: warp gw = blockIdx.x * kWarps + w of the n_workers
// workers owns the splits [wsplit[gw], wsplit[gw + 1]): contiguous page ranges
// of consecutive units, cut so that every warp gets about the same cost.  The
// warp writes one partial per split.  kHead: some slots are excluded for
// single kv heads (hdead, one word per page id x kv head); without it the
// scan does not carry the extra pointer.  kMulti: the splits come from
// several pools (head groups, each with its own pages and tables): a split
// names its pool and its kv head within the pool, the page stream reads the
// pool's addresses from gpools, and a page ticket carries its width.  kI3:
// the pool has INT3 pages (ids [n3b, nfb), blocks from int3_off) or FP4
// pages (ids from nfb, blocks from fp4_off).
template <int G, bool kHead, bool kMulti, bool kI3>
__global__ void __launch_bounds__(kThreads, 1) decode_mma_kernel(
    const uint8_t* __restrict__ pool, size_t int4_off, int64_t n2, int hkv, int max_pages,
    const Entry* __restrict__ table, const UnitFrag* __restrict__ frags, const Split* __restrict__ splits,
    const int32_t* __restrict__ wsplit, int n_workers, const int32_t* __restrict__ ntab,
    const uint32_t* __restrict__ hdead, float* __restrict__ part, const uint32_t* __restrict__ smax_bits,
    uint32_t* __restrict__ status, uint32_t first_spins, const GroupPool* __restrict__ gpools, size_t int3_off,
    int64_t n3b, size_t fp4_off, int64_t nfb) {
  constexpr bool kPair = Cols<G>::kPair;
  constexpr int NH = Cols<G>::NH;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, r = lane >> 2, i = lane & 3;
  WarpSmem& WS = reinterpret_cast<WarpSmem*>(smem_raw)[w];
  // neighbouring workers share an SM: they scan the same one or two units, so
  // the q operands they read stay in that SM's L1
  const int gw = blockIdx.x * kWarps + w;
  // the plan is copied in before the launch (not by a kernel): read it first
  const int s_begin = gw < n_workers ? wsplit[gw] : 0, s_end = gw < n_workers ? wsplit[gw + 1] : 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // fragments, and the appends before them, are done
  asm volatile("griddepcontrol.launch_dependents;");   // the merge may be staged
  if (s_begin >= s_end) return;   // no CTA-wide barrier below: idle warps may leave
  // P is carried as p * 2^sv in the fp16 folds so that p * scale stays clear
  // of the binary16 subnormal range; 2^sv * (largest V scale) <= 2^15.
  float vmax = fmaxf(__uint_as_float(smax_bits[1]), 1.0f / 1024.0f);
  if constexpr (kMulti) {
    // a warp may read pages of every pool: bound the V scales of all of them
    const int np = gpools[0].n_pools;
    for (int p = 0; p < np; ++p) vmax = fmaxf(vmax, __uint_as_float(gpools[p].smax[1]));
  }
  const int sv = max(0, min(15, ilogbf(32768.0f / vmax)));
  const float pscale = ldexpf(1.0f, sv), oscale = ldexpf(1.0f, -sv);
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) bar_init(&WS.bar[st]);
    if constexpr (kHead) WS.hdead = hdead;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // ---- the warp's page stream, read in batches of up to 32 pages: lane j of
  // a batch holds stream page bbase + j (its table entry, the address of its
  // block and tag = split << 6 | kv head; num_kv_heads <= 64), found with the
  // scan order in closed form, so that a page costs a few shuffles.  A batch
  // stops at the end of a split.  A ticket is one page; id < 0 ends the stream.
  struct Ticket {
    int32_t id;
    uint32_t live;
    int32_t tag;
  };
  int lsg = s_begin, lpos = 0, lend = 0, lkvh = 0, ln = 0, lm = 0;   // reader: split, next position, end, ...
  int lpl = 0;   // kMulti: pool of the split being read
  const Entry* ltab = table;
  auto enter = [&](int sg) {
    const Split sp = splits[sg];
    lpos = sp.page_begin;
    ln = sp.n_pos;
    lm = sp.n_lead;
    if constexpr (kMulti) {
      lpl = sp.pad[0];
      const GroupPool* gp = gpools + lpl;
      ltab = gp->table + (size_t)sp.req * gp->max_pages;
      lend = sp.page_end >= 0 ? sp.page_end : gp->ntab[sp.req];
      lkvh = sp.pad[1];
    } else {
      ltab = table + (size_t)sp.req * max_pages;
      lend = sp.page_end >= 0 ? sp.page_end : ntab[sp.req];   // open-ended: the table's length now
      lkvh = sp.unit % hkv;
    }
  };
  enter(lsg);
  int bbase = 0, bcount = 0;   // the batch holds stream pages [bbase, bbase + bcount)
  int32_t bid = -1, btag = 0;
  uint32_t blive = 0u;
  int32_t brank = -1;   // kHead: rank of this lane's page among the batch's pages with a live slot (-1: none)
  unsigned long long bsrc = 0ull;
  // kHead: a page whose every slot is dead for this kv head is skipped (no
  // copy, no work): it would add nothing, since a dead slot's weight
  // 2^(-1e4 log2 e - m) is 0 and its V is 0.  A unit left with no page reads
  // as empty, as an all-dead unit does.
  auto refill = [&](int k) {
    for (;;) {
    while (lpos >= lend && lsg + 1 < s_end) enter(++lsg);
    const int nb = max(0, min(32, lend - lpos));
    bbase = k;
    bcount = nb;
    bid = -1;
    if constexpr (kHead || kMulti) blive = 0u;
    if (lane < nb) {
      // scan-order position p -> table index: the next INT2-first entry when
      // floor((p+1) m / n) > floor(p m / n), else the next of the others
      const int p = lpos + lane;
      int idx = p;
      if (p < ln) {
        const int64_t n64 = ln;
        const int a0 = (int)((int64_t)p * lm / n64), a1 = (int)((int64_t)(p + 1) * lm / n64);
        idx = a1 > a0 ? a0 : lm + p - a1;
      }
      const Entry e = ltab[idx];
      bid = e.id;
      if constexpr (kMulti) {
        // the split's pool: width from its INT2 range, exclusion words if it has them
        const GroupPool* gp = gpools + lpl;
        const int64_t gn2 = gp->n2;
        const int ghkv = gp->hkv;
        const uint32_t* hd = gp->hdead;
        blive = hd ? e.live & ~hd[(size_t)e.id * ghkv + lkvh] : e.live;
        const bool i2 = e.id < gn2;
        int cls = i2 ? 1 : 0;   // width class in the ticket: 0 INT4, 1 INT2, 2 INT3, 3 FP4
        const uint8_t* src = i2 ? gp->pool + ((size_t)e.id * ghkv + lkvh) * kInt2Block
                                : gp->pool + gp->int4_off + ((size_t)(e.id - gn2) * ghkv + lkvh) * kInt4Block;
        if constexpr (kI3) {
          if (e.id >= gp->nfb) {
            cls = 3;
            src = gp->pool + gp->fp4_off + ((size_t)(e.id - gp->nfb) * ghkv + lkvh) * kFp4Block;
          } else if (e.id >= gp->n3b) {
            cls = 2;
            src = gp->pool + gp->int3_off + ((size_t)(e.id - gp->n3b) * ghkv + lkvh) * kInt3Block;
          }
        }
        btag = (lsg << 8) | (cls << 6) | lkvh;
        bsrc = (unsigned long long)(uintptr_t)src;
      } else {
        // slots excluded for this kv head only read as dead slots too
        if constexpr (kHead) {
          const uint32_t* hd = *reinterpret_cast<const uint32_t* const volatile*>(&WS.hdead);
          blive = e.live & ~hd[(size_t)e.id * hkv + lkvh];
        }
        else blive = e.live;
        btag = (lsg << 6) | lkvh;
        const uint8_t* src = e.id < n2 ? pool + ((size_t)e.id * hkv + lkvh) * kInt2Block
                                       : pool + int4_off + ((size_t)(e.id - n2) * hkv + lkvh) * kInt4Block;
        if constexpr (kI3) {
          if (e.id >= nfb) src = pool + fp4_off + ((size_t)(e.id - nfb) * hkv + lkvh) * kFp4Block;
          else if (e.id >= n3b) src = pool + int3_off + ((size_t)(e.id - n3b) * hkv + lkvh) * kInt3Block;
        }
        bsrc = (unsigned long long)(uintptr_t)src;
      }
    }
    lpos += nb;
    if constexpr (kHead || kMulti) {
      const bool keep = lane < nb && blive != 0u;
      const uint32_t kept = __ballot_sync(0xFFFFFFFFu, keep);
      brank = keep ? __popc(kept & ((1u << lane) - 1u)) : -1;
      bcount = __popc(kept);
      if (bcount > 0 || nb == 0) break;   // else the whole batch is dead: the next one
    } else {
      break;
    }
    }
  };
  bool more = true;   // the stream may hold pages past the current batch
  // ticket of stream page k (k >= bbase; refills when k is past the batch)
  auto ticket = [&](int k, unsigned long long& src) -> Ticket {
    if (k >= bbase + bcount) {
      if (!more) return Ticket{-1, 0u, 0};
      refill(k);
      if (bcount == 0) {
        more = false;
        return Ticket{-1, 0u, 0};
      }
    }
    int j = k - bbase;
    if constexpr (kHead || kMulti) j = __ffs(__ballot_sync(0xFFFFFFFFu, brank == j)) - 1;   // the lane of the j-th page kept
    src = __shfl_sync(0xFFFFFFFFu, bsrc, j);
    return Ticket{__shfl_sync(0xFFFFFFFFu, bid, j), __shfl_sync(0xFFFFFFFFu, blive, j),
                  __shfl_sync(0xFFFFFFFFu, btag, j)};
  };
  // a ticket's width and split
  auto tk_int2 = [&](const Ticket& t) { return kMulti ? ((t.tag >> 6) & 3) == 1 : t.id < n2; };
  auto tk_split = [&](const Ticket& t) { return kMulti ? t.tag >> 8 : t.tag >> 6; };
  auto tk_int3 = [&](const Ticket& t) {
    return kI3 && (kMulti ? ((t.tag >> 6) & 3) == 2 : (t.id >= n3b && t.id < nfb));
  };
  auto tk_fp4 = [&](const Ticket& t) { return kI3 && (kMulti ? ((t.tag >> 6) & 3) == 3 : t.id >= nfb); };
  // copy number n goes to stage n & 1 and completes phase (n >> 1) & 1
  auto issue = [&](const Ticket& t, unsigned long long src, uint32_t n) {   // lane 0
    const uint32_t st = n & (kStages - 1);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the stage was read generically
    bulk_load(WS.stage[st], (const void*)(uintptr_t)src,
              tk_int2(t)   ? (uint32_t)kInt2Block
              : tk_int3(t) ? (uint32_t)kInt3Block
              : tk_fp4(t)  ? (uint32_t)kFp4Block
                           : (uint32_t)kInt4Block,
              &WS.bar[st]);
  };
  static_assert(kStages == 2, "the ticket ring below serves a two-stage copy ring");
  unsigned long long src0 = 0ull, src1 = 0ull;
  Ticket t0 = ticket(0, src0);
  Ticket t1 = t0.id >= 0 ? ticket(1, src1) : Ticket{-1, 0u, 0};   // pages c, c+1 (copies issued)
  if (lane == 0) {
    if (t0.id >= 0) issue(t0, src0, 0u);
    if (t1.id >= 0) issue(t1, src1, 1u);
  }

  // ---- state of the split being scanned
  const UnitFrag* F = frags;
  float acol2[NH], acol4[NH];
  uint32_t bz[2];
  float o[8][4], zv[4], mrun[NH], lsum[NH];
  auto begin_split = [&](int sg) {
    F = frags + splits[sg].unit;
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      const int h = kPair ? i : 2 * i + hh;
      acol2[hh] = __ldg(&F->acol2[h]);
      acol4[hh] = __ldg(&F->acol4[h]);
      mrun[hh] = -INFINITY;
      lsum[hh] = 0.0f;
    }
    // INT4 K zero term B fragment: column r; with paired columns only the
    // even columns (part 0) carry Q
    const int hb = kPair ? (r >> 1) : r;
    const bool has = hb < G && i < 2 && (!kPair || !(r & 1));
    bz[0] = has ? __ldg(&F->bz[hb][2 * i]) : 0u;
    bz[1] = has ? __ldg(&F->bz[hb][2 * i + 1]) : 0u;
#pragma unroll
    for (int m = 0; m < 8; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.0f;
    zv[0] = zv[1] = zv[2] = zv[3] = 0.0f;
  };
  // partial of split sg: finish l, combine the column parts, add the V zero term
  auto flush = [&](int sg) {
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      lsum[hh] += __shfl_xor_sync(0xFFFFFFFFu, lsum[hh], 4);
      lsum[hh] += __shfl_xor_sync(0xFFFFFFFFu, lsum[hh], 8);
      lsum[hh] += __shfl_xor_sync(0xFFFFFFFFu, lsum[hh], 16);
    }
    float* zb = &WS.pbuf[0][0];   // [group][column]
    __syncwarp();
    if (r < 4) {
      if (kPair) {
        zb[r * 8 + i] = zv[0] + zv[1];
      } else {
        zb[r * 8 + 2 * i] = zv[0];
        zb[r * 8 + 2 * i + 1] = zv[1];
      }
    }
    __syncwarp();
    float* out = part + (size_t)sg * G * kPartStride;
    if constexpr (kPair) {
      if (i < G) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float zt = zb[(m >> 1) * 8 + i];
          out[i * kPartStride + 16 * m + r] = fmaf(o[m][0] + o[m][1], kCodeUnit, zt) * oscale;
          out[i * kPartStride + 16 * m + r + 8] = fmaf(o[m][2] + o[m][3], kCodeUnit, zt) * oscale;
        }
        if (r == 0) {
          out[i * kPartStride + kHeadDim] = mrun[0];
          out[i * kPartStride + kHeadDim + 1] = lsum[0];
        }
      }
    } else {
#pragma unroll
      for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int h = 2 * i + (cc & 1), ch = 16 * m + r + 8 * (cc >> 1);
          if (h < G) out[h * kPartStride + ch] = fmaf(o[m][cc], kCodeUnit, zb[(m >> 1) * 8 + h]) * oscale;
        }
      if (r == 0)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          if (2 * i + hh < G) {
            out[(2 * i + hh) * kPartStride + kHeadDim] = mrun[hh];
            out[(2 * i + hh) * kPartStride + kHeadDim + 1] = lsum[hh];
          }
    }
    __syncwarp();   // zb is P staging again for the next page
  };
  // partial of a split that adds nothing (no page scanned, or a timed-out scan)
  auto flush_empty = [&](int sg) {
    float* out = part + (size_t)sg * G * kPartStride;
    for (int x = lane; x < G * kPartStride; x += 32) out[x] = (x % kPartStride) == kHeadDim ? -INFINITY : 0.0f;
  };

  // ---- page loop
  int csg = -1;        // split being scanned
  uint32_t c = 0;      // copies consumed
  bool ok = true;
  while (t0.id >= 0) {
    const int sg = tk_split(t0);
    if (sg != csg) {
      if (csg >= 0) flush(csg);
      for (int x = csg < 0 ? s_begin : csg + 1; x < sg; ++x) flush_empty(x);
      csg = sg;
      begin_split(sg);
    }
    const uint32_t st = c & (kStages - 1);
    // the first wait's bound is kSpinLimit unless a test shortens it
    const bool got = bar_wait(&WS.bar[st], (c >> 1) & 1u, c == 0 ? first_spins : kSpinLimit);
    if (!__all_sync(0xFFFFFFFFu, got)) {
      ok = false;
      break;
    }
    const uint8_t* blk = WS.stage[st];
    float lg[2][2][NH], zc[NH];
    if (tk_int2(t0)) {
      qk_int2<G>(blk, F, acol2, lg, zc);
      softmax_pv<G, true>(blk, t0.live, pscale, lg, zc, o, zv, mrun, lsum, WS.pbuf);
    } else if (tk_int3(t0)) {
      if constexpr (kI3) {
        qk_int4<G, true>(blk, &F->bq3[0][0], bz, acol4, lg);
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) zc[hh] = 0.0f;
        softmax_pv<G, false, true>(blk, t0.live, pscale, lg, zc, o, zv, mrun, lsum, WS.pbuf);
      }
    } else if (tk_fp4(t0)) {
      if constexpr (kI3) {
        // FP4 codes pair channels n, n + 4 with no 2^2: the INT3 q fragments
        qk_int4<G, false, true>(blk, &F->bq3[0][0], bz, acol4, lg);
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) zc[hh] = 0.0f;
        softmax_pv<G, false, false, true>(blk, t0.live, pscale, lg, zc, o, zv, mrun, lsum, WS.pbuf);
      }
    } else {
      qk_int4<G>(blk, &F->bq4[0][0], bz, acol4, lg);
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) zc[hh] = 0.0f;
      softmax_pv<G, false>(blk, t0.live, pscale, lg, zc, o, zv, mrun, lsum, WS.pbuf);
    }
    ++c;
    unsigned long long src2 = 0ull;
    const Ticket t2 = t1.id >= 0 ? ticket((int)c + 1, src2) : Ticket{-1, 0u, 0};   // page c + 2 of the old c
    if (t2.id >= 0 && lane == 0) issue(t2, src2, c + 1);
    t0 = t1;
    t1 = t2;
  }
  if (!ok) {
    if (lane == 0) atomicOr(status, kStatusTimeout);
    // let the copies in flight land before the warp leaves
    if (t0.id >= 0) bar_wait(&WS.bar[c & (kStages - 1)], (c >> 1) & 1u);
    if (t1.id >= 0) bar_wait(&WS.bar[(c + 1) & (kStages - 1)], ((c + 1) >> 1) & 1u);
    for (int x = csg; x < s_end; ++x) flush_empty(x);
    return;
  }
  if (csg >= 0) flush(csg);
  for (int x = csg < 0 ? s_begin : csg + 1; x < s_end; ++x) flush_empty(x);
}

constexpr int kScanSmem = kWarps * (int)sizeof(WarpSmem);

// The scan reads its q operands and its spilled registers through L1, which
// shares the SM's memory with shared memory: ask for the smallest shared
// carveout that holds one CTA (the default takes the largest, leaving L1 too
// small for 16 warps' q operands; the scan then ran up to 1.45x slower).
template <int G, bool kHead, bool kMulti, bool kI3>
cudaError_t set_scan_attributes() {
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<G, kHead, kMulti, kI3>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, per_sm = 0, reserved = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
  if (per_sm <= 0) return cudaErrorInvalidValue;
  const int pct = std::min(100, (int)(((int64_t)(kScanSmem + reserved) * 100 + per_sm - 1) / per_sm));
  return cudaFuncSetAttribute(decode_mma_kernel<G, kHead, kMulti, kI3>, cudaFuncAttributePreferredSharedMemoryCarveout,
                              pct);
}

template <int G>
cudaError_t launch_mma_g(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units, int n_units,
                         const Split* d_splits, const int32_t* d_wsplit, int n_workers, void* d_frags, float* d_part,
                         cudaStream_t s, const GroupPool* d_gpools, bool groups_extra) {
  // function attributes are set once per device (bit = device ordinal)
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(attr_set.load() >> dev & 1u)) {
    cudaError_t e = set_scan_attributes<G, false, false, false>();
    if (e == cudaSuccess) e = set_scan_attributes<G, true, false, false>();
    if (e == cudaSuccess) e = set_scan_attributes<G, false, true, false>();
    if (e == cudaSuccess) e = set_scan_attributes<G, false, false, true>();
    if (e == cudaSuccess) e = set_scan_attributes<G, true, false, true>();
    if (e == cudaSuccess) e = set_scan_attributes<G, false, true, true>();
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(uint64_t(1) << dev);
  }
  if (n_workers <= 0 || n_units <= 0) return cudaSuccess;
  const uint32_t* smax = P->d_status + 1;
  P->launches += 2;
  cudaError_t e = launch_pdl(frag_kernel<G>, dim3((unsigned)n_units), dim3(256), 0, s, (const __nv_bfloat16*)q,
                             (int)hq, scale_log2, d_units, smax, (UnitFrag*)d_frags, d_gpools);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((n_workers + kWarps - 1) / kWarps);
  // pools with INT3 or FP4 pages take the variant that reads them (grouped
  // decodes take no such pool)
  const bool i3 = P->cfg.n_int3_pages > 0 || P->cfg.n_fp4_pages > 0;
  auto* kernel = d_gpools ? (groups_extra ? decode_mma_kernel<G, false, true, true>
                                          : decode_mma_kernel<G, false, true, false>)
                 : i3     ? (P->hdead.empty() ? decode_mma_kernel<G, false, false, true>
                                              : decode_mma_kernel<G, true, false, true>)
                          : (P->hdead.empty() ? decode_mma_kernel<G, false, false, false>
                                              : decode_mma_kernel<G, true, false, false>);
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), (size_t)kScanSmem, s, (const uint8_t*)P->d_pool,
                    P->int4_offset, (int64_t)P->cfg.n_int2_pages, P->cfg.num_kv_heads, P->cfg.max_pages_per_request,
                    (const Entry*)P->d_table, (const UnitFrag*)d_frags, d_splits, d_wsplit, n_workers,
                    (const int32_t*)P->d_ntab, (const uint32_t*)P->d_hdead, d_part, smax, P->d_status,
                    P->first_wait_spins < 0 ? kSpinLimit : (uint32_t)P->first_wait_spins, d_gpools, P->int3_offset,
                    (int64_t)(P->cfg.n_int2_pages + P->cfg.n_int4_pages), P->fp4_offset,
                    (int64_t)(P->cfg.n_int2_pages + P->cfg.n_int4_pages + P->cfg.n_int3_pages));
}

template <int G>
int mma_occupancy() {
  int n = 0;
  if (set_scan_attributes<G, false, false, false>() != cudaSuccess) return 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<G, false, false, false>, kThreads,
                                                    kScanSmem) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

}  // namespace

size_t decode_mma_frag_bytes() { return sizeof(UnitFrag); }

cudaError_t launch_decode_mma(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units, int n_units,
                              const Split* d_splits, const int32_t* d_wsplit, int n_workers, void* d_frags,
                              float* d_part, float* out, cudaStream_t s, const GroupPool* d_gpools,
                              int32_t total_kv_heads, bool groups_extra) {
  cudaError_t e;
  const int g = hq / (total_kv_heads > 0 ? total_kv_heads : P->cfg.num_kv_heads);
#define KVQ_MMA_CASE(gg)                                                                                          \
  case gg:                                                                                                        \
    e = launch_mma_g<gg>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_wsplit, n_workers, d_frags, d_part, s, \
                         d_gpools, groups_extra);                                                                 \
    break;
  switch (g) {
    KVQ_MMA_CASE(1)
    KVQ_MMA_CASE(2)
    KVQ_MMA_CASE(3)
    KVQ_MMA_CASE(4)
    KVQ_MMA_CASE(5)
    KVQ_MMA_CASE(6)
    KVQ_MMA_CASE(7)
    KVQ_MMA_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef KVQ_MMA_CASE
  if (e != cudaSuccess) return e;
  if ((e = launch_fp_pending(P, q, hq, scale_log2, d_units, d_part, s)) != cudaSuccess) return e;
  if (P->merge_event && (e = cudaEventRecord(P->merge_event, s)) != cudaSuccess) return e;
  return launch_merge(P, g, d_units, n_units, d_part, hq, out, s);
}

int decode_mma_workers_per_sm(int g) {
  switch (g) {
    case 1: return kWarps * mma_occupancy<1>();
    case 2: return kWarps * mma_occupancy<2>();
    case 3: return kWarps * mma_occupancy<3>();
    case 4: return kWarps * mma_occupancy<4>();
    case 5: return kWarps * mma_occupancy<5>();
    case 6: return kWarps * mma_occupancy<6>();
    case 7: return kWarps * mma_occupancy<7>();
    default: return kWarps * mma_occupancy<8>();
  }
}

}  // namespace kvq

