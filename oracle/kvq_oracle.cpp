/*
 * kvq_oracle.cpp -- plain, slow CPU oracle for decode attention over a paged,
 * mixed INT2/INT3/INT4/FP4 quantized KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path (no headers, helpers, tables or constants); the only thing the
 * two sides share is the seeded input generator in kvsynth/.
 *
 * What it computes, and the passage each step follows (pages are cited by
 * title and section):
 *   - greedy INT2/INT4 bit allocation by rho_k = (D_k(2) - D_k(4)) / (2 N_k)
 *       [TriAxialKV, key design 2: attention-output-distortion calibration and
 *        greedy bit-width allocation]
 *   - asymmetric group quantization, G = 32: INT4 K and V per token, INT2 K per
 *     channel (scale/zero shared across 32 tokens), INT2 V per token; residual
 *     tokens that cannot fill a 32-token INT2 group stay INT4
 *       [TriAxialKV, key design 3: custom mixed-precision cache layout and
 *        residual fallback]
 *   - one pool holding INT2 and INT4 pages, precision decided by page id;
 *     INT2 pages reordered ahead of INT4 pages in each request's table; new
 *     tokens written as INT4 at the tail
 *       [TriAxialKV, key design 4: unified address space dual pool and the
 *        fused Flash-Decoding operator]
 *   - evicted slots read as a sentinel dead slot (logit -1e4, V = 0) without
 *     moving surviving pages
 *       [IntentKV, method 2: layout-preserving eviction, sentinel dead slot]
 *   - softmax attention in fp64, and a split + log-sum-exp merge variant
 *       [HyQuant, background "FlashAttention and online softmax" (m, l, acc;
 *        O = acc / l) and Algorithm 3 split-K ReduceSoftmax]
 *   - full-precision segments: each key position belongs to exactly one of
 *     the quantized set, the vertical-line set or the window of its head; the
 *     vertical-line, staging and window tokens are kept in bf16 and scanned
 *     after the quantized prefix with the same softmax state; the quantized
 *     copy of a position held in full precision for one head is excluded for
 *     that head only
 *       [HyQuant, core method (K = K_VL u K_Win u K_Q, mutually exclusive),
 *        Algorithm 3 (decode: quantized prefix, vertical lines, staging
 *        buffer, window) and Algorithm 4 (FREEZE)]
 *
 * Readings of points the pages leave open (each restated where it is used):
 *   R1 scale and zero are stored as IEEE binary16 (round to nearest even).
 *   R2 per-token groups are 32 consecutive channels of one token and head.
 *   R3 quantization: mn, mx exact; s32 = (mx - mn) / (2^b - 1) in fp32; s, z =
 *      half(s32), half(mn); code = clamp(rint_even((x - z) / s), 0, 2^b - 1) in
 *      fp32, code = 0 when s == 0; dequantization x^ = fmaf(code, s, z).
 *   R4 INT2-tagged tokens wait in an INT4 "staging" page of their request; when
 *      it holds 32 tokens it is requantized to INT2 from its INT4-dequantized
 *      values, the staging page is freed and the INT2 page is appended to the
 *      request's table.  Ids freed during one append call become reusable
 *      after the call.  All 32 stored slots take part in the requantization;
 *      the live mask is carried over unchanged.
 *   R5 a page id is taken as the lowest free id of its class (INT2 ids
 *      [0, n2), INT4 ids [n2, n2 + n4); with INT3 pages (R11) INT3 ids
 *      [n2 + n4, n2 + n4 + n3) follow them).
 *   R6 the dead slot's logit is -1e4 after scaling and its V is 0; slots never
 *      written are not tokens and are skipped.
 *   R7 the greedy scan skips a tag that does not fit the budget and continues;
 *      the budget test is exact integer arithmetic with B = num / den.
 *   R8 a request's full-precision tokens form one ordered list per kv head
 *      (the caller decides which are vertical-line, staging or window
 *      tokens; every head holds the same count, its own rows); they follow
 *      the quantized tokens in the token sequence; their logit is
 *      scale * q . k and their value v, both read from bf16.  Dropping
 *      tokens keeps the order of the rest.
 *   R9 a slot excluded for one head reads, for that head, as the sentinel
 *      dead slot of R6.
 *   R11 INT3 pages.  The pages name three-bit integers only as a further width
 *      the two-way INT2/INT4 choice could gain.  Read as a third width beside
 *      them: K and V per token in groups of 32 channels exactly as INT4 (R2,
 *      R3 with b = 3: codes 0..7, scale (max - min) / 7), on pages of their
 *      own class (ids [n2 + n4, n2 + n4 + n3), after the INT4 ids); a
 *      request's INT3 tokens fill its own INT3 tail page in arrival order, as
 *      INT4 tokens fill the INT4 tail; the phase-1 reorder sorts each table
 *      stably by width (INT2, INT3, INT4 entries, each in table order); the
 *      greedy allocation stays the pages' INT2/INT4 one (R7), and INT3 widths
 *      come from the caller
 *       [TriAxialKV, limitations and outlook: INT3 as a further width].
 *   R12 FP4 pages.  The pages name non-uniform floating formats as a further
 *      option and compare against a uniform FP4 cache.  Read as a fourth page
 *      class holding E2M1 values (sign, 2 exponent bits with bias 1, 1
 *      mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; code = sign << 3 |
 *      exponent << 1 | mantissa), K and V per token in groups of 32 channels,
 *      symmetric with the scale of the HyQuant background, s = max|x| / c_B
 *      with c_B = 6 the format's largest value (fp32 division, stored as
 *      binary16 as R1), no zero point; a value is coded as the E2M1 value
 *      nearest to x / s (fp32 division), ties to the even mantissa, magnitudes
 *      above 6 saturating to 6, zero coded +0; s = 0 codes every value 0;
 *      dequantization x^ = s * value (exact in fp32).  Ids after the INT3 ids;
 *      a request's FP4 tokens fill its own FP4 tail page; the reorder puts FP4
 *      entries after INT4 entries; FP4 widths come from the caller
 *       [TriAxialKV, limitations and outlook: non-uniform FP formats;
 *        comparison with a uniform FP4 cache; HyQuant, background on
 *        low-bit quantization: s = max|X| / c_B].
 *   R13 bit allocation over three widths (the limitations section: the
 *      two-way INT2/INT4 choice is what INT3 would widen).  Read as the same
 *      greedy over one-bit steps: every tag starts at 2 bits and has a
 *      2 -> 3 step and a 3 -> 4 step, each costing N_k bit-tokens and saving
 *      D_k(2) - D_k(3) and D_k(3) - D_k(4); the available step with the most
 *      distortion saved per bit-token, (saving) / N_k in fp64, is taken next
 *      (a 3 -> 4 step becomes available once its 2 -> 3 step is taken; ties:
 *      the lower tag); a step that does not fit the budget (R7's exact
 *      integer test) is dropped and the scan continues.  With one 2 -> 4 step
 *      per tag (saving D(2) - D(4) over 2 N_k bit-tokens) this is key design
 *      2's rule
 *       [TriAxialKV, key design 2; limitations and outlook].
 *   R10 a full page none of whose 32 slots is live for any kv head may leave
 *      its request's table: the other entries keep their order and their
 *      pages do not move, its id returns to the free set, and the positions
 *      it held read as dropped.  Head groups that keep different amounts of
 *      context are pools of their own over their kv heads, fed the same
 *      tokens; a group drops the pages its budget no longer covers
 *       [Tangram, method steps 6-7: head groups with different retained
 *        lengths, each holding only its own pages; IntentKV, method 2].
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <set>
#include <string>
#include <unordered_map>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ORC_OK = 0, ORC_INVALID = 1, ORC_OOM = 2, ORC_RANGE = 3, ORC_STATE = 6 };
constexpr int kFP4 = 0xF4;     // the width value of FP4 (E2M1) tokens and pages (R12)
constexpr int kD = 128;        // head dim
constexpr int kP = 32;         // tokens per page
constexpr int kG = 32;         // group size

// ---------------------------------------------------------------------------
// IEEE 754 binary16 <-> binary32, written from the format's definition:
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals below
// 2^-14 with spacing 2^-24.  Rounding is to nearest, ties to even.
// ---------------------------------------------------------------------------
uint16_t f32_to_f16(float f) {
  uint32_t x;
  std::memcpy(&x, &f, 4);
  const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  const uint32_t ef = (x >> 23) & 0xFFu;
  const uint32_t frac = x & 0x7FFFFFu;
  if (ef == 0xFFu) return (uint16_t)(sign | 0x7C00u | (frac ? (0x200u | (frac >> 13)) : 0u));
  if (ef == 0 && frac == 0) return sign;
  // value = sig * 2^(e - 23) with sig a 24-bit integer (implicit bit included)
  int e;
  uint32_t sig;
  if (ef == 0) { e = -126; sig = frac; } else { e = (int)ef - 127; sig = frac | 0x800000u; }
  if (e > 15) return (uint16_t)(sign | 0x7C00u);
  int drop;            // fraction bits of sig that do not fit
  uint32_t hexp;       // biased half exponent before rounding (0 = subnormal)
  if (e >= -14) { drop = 13; hexp = (uint32_t)(e + 15); }
  else { drop = 13 + (-14 - e); hexp = 0; }
  if (drop > 24) return sign;                      // below half of the smallest subnormal
  uint32_t q = sig >> drop;
  const uint32_t rem = sig & ((1u << drop) - 1u);
  const uint32_t half = 1u << (drop - 1);
  if (rem > half || (rem == half && (q & 1u))) ++q;
  uint32_t bits;
  if (hexp == 0) bits = q;                          // may carry into the smallest normal
  else bits = (hexp << 10) + q - 0x400u;            // q in [0x400, 0x800]; carry bumps exponent
  if (bits >= 0x7C00u) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | bits);
}

float f16_to_f32(uint16_t h) {
  const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  const uint32_t e = (h >> 10) & 0x1Fu;
  const uint32_t m = h & 0x3FFu;
  float v;
  if (e == 0) v = std::ldexp((float)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = std::ldexp((float)(m | 0x400u), (int)e - 25);
  uint32_t b;
  std::memcpy(&b, &v, 4);
  b |= sign;
  std::memcpy(&v, &b, 4);
  return v;
}

float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

bool in_range(float x) { return std::isfinite(x) && std::fabs(x) <= 65504.0f; }

// ---------------------------------------------------------------------------
// Asymmetric group quantization (TriAxialKV, key design 3; reading R3).
// x[i * stride], i < n; writes codes[i * cstride].
// ---------------------------------------------------------------------------
void quant_group(const float* x, int n, int stride, int bits, uint8_t* codes, int cstride,
                 uint16_t* s_out, uint16_t* z_out) {
  float mn = x[0], mx = x[0];
  for (int i = 1; i < n; ++i) {
    const float v = x[(size_t)i * stride];
    mn = std::min(mn, v);
    mx = std::max(mx, v);
  }
  const int qmax = (1 << bits) - 1;
  volatile float range = mx - mn;                   // one fp32 rounding
  const float s32 = range / (float)qmax;            // one fp32 rounding
  const uint16_t sh = f32_to_f16(s32);
  const uint16_t zh = f32_to_f16(mn);
  const float sf = f16_to_f32(sh), zf = f16_to_f32(zh);
  for (int i = 0; i < n; ++i) {
    int c = 0;
    if ((sh & 0x7FFFu) != 0) {
      volatile float d = x[(size_t)i * stride] - zf;
      const float u = d / sf;
      const float r = std::nearbyint(u);            // default rounding mode: ties to even
      c = r < 0.0f ? 0 : (r > (float)qmax ? qmax : (int)r);
    }
    codes[(size_t)i * cstride] = (uint8_t)c;
  }
  *s_out = sh;
  *z_out = zh;
}

inline float dequant(uint8_t code, uint16_t s, uint16_t z) {
  return std::fma((float)code, f16_to_f32(s), f16_to_f32(z));
}

// ---------------------------------------------------------------------------
// FP4 (E2M1) group quantization (reading R12).
// ---------------------------------------------------------------------------
// magnitude of E2M1 code bits (exponent << 1 | mantissa): exponent 0 holds
// 0 and the subnormal 0.5, exponent e > 0 holds (1 + mantissa / 2) * 2^(e-1)
double e2m1_magnitude(int m) {
  const int e = m >> 1, f = m & 1;
  return e == 0 ? 0.5 * f : (1.0 + 0.5 * f) * std::ldexp(1.0, e - 1);
}
double e2m1_value(uint8_t code) { return (code & 8 ? -1.0 : 1.0) * e2m1_magnitude(code & 7); }

void fp4_group(const float* x, int n, int stride, uint8_t* codes, int cstride, uint16_t* s_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(x[(size_t)i * stride]));
  volatile float s32 = amax / 6.0f;                 // one fp32 rounding
  const uint16_t sh = f32_to_f16(s32);
  const float sf = f16_to_f32(sh);
  for (int i = 0; i < n; ++i) {
    uint8_t c = 0;
    if ((sh & 0x7FFFu) != 0) {
      const float u = x[(size_t)i * stride] / sf;   // one fp32 rounding
      const double a = std::fabs((double)u);
      int best = 0;                                 // nearest magnitude, ties to the even mantissa
      for (int m = 1; m < 8; ++m) {
        const double d = std::fabs(a - e2m1_magnitude(m)), db = std::fabs(a - e2m1_magnitude(best));
        if (d < db || (d == db && (m & 1) == 0)) best = m;
      }
      c = (uint8_t)(best == 0 ? 0 : ((u < 0.0f ? 8 : 0) | best));
    }
    codes[(size_t)i * cstride] = c;
  }
  *s_out = sh;
}

inline float dequant_fp4(uint8_t code, uint16_t s) { return (float)(e2m1_value(code) * (double)f16_to_f32(s)); }

// ---------------------------------------------------------------------------
// Pool model.
// Canonical content of one (page, kv-head) block:
//   kc[slot][ch], vc[slot][ch]      codes, one byte each
//   km[256]: INT4 page -> [slot][group]{s, z};  INT2 page -> [ch]{s, z}
//   vm[256]: [slot][group]{s, z}  (V is per token at both widths)
// ---------------------------------------------------------------------------
struct HeadBlock {
  uint8_t kc[kP * kD];
  uint8_t vc[kP * kD];
  uint16_t km[256];
  uint16_t vm[256];
};

struct Page {
  int32_t id = -1;
  int bits = 4;                   // 2, 3, 4 or kFP4 (the id's class)
  int fill = 0;
  uint32_t live = 0;
  std::vector<uint32_t> hdead;    // per kv head: slots excluded for that head only (R9)
  bool content = false;
  int64_t pos[kP];
  std::vector<HeadBlock> heads;
};

struct Req {
  bool open = false;
  std::vector<int32_t> table;
  int32_t tail4 = -1, tail3 = -1, tailf = -1, staging = -1;
  std::vector<uint32_t> loc;      // token position -> page_id << 5 | slot
  int64_t n_fp = 0;               // full-precision tokens (R8)
  std::vector<uint16_t> fpk, fpv; // their bf16 bits [n_fp][n_sel][128]
};

struct Pool {
  int hkv = 0;
  std::vector<int> sel;           // kv heads whose content is kept
  int64_t n2 = 0, n3 = 0, n4 = 0, nf = 0;
  int max_req = 0, max_pages = 0;
  std::set<int32_t> free2, free3, free4, freef;
  std::unordered_map<int32_t, Page> pages;
  std::vector<Req> reqs;
};

}  // namespace

namespace {

int32_t take_lowest(std::set<int32_t>& s) {
  const int32_t id = *s.begin();
  s.erase(s.begin());
  return id;
}

Page& new_page(Pool* P, int bits, bool content) {
  const int32_t id =
      take_lowest(bits == 2 ? P->free2 : (bits == 3 ? P->free3 : (bits == kFP4 ? P->freef : P->free4)));
  Page& pg = P->pages[id];
  pg = Page();
  pg.id = id;
  pg.bits = bits;
  pg.hdead.assign((size_t)P->hkv, 0u);
  pg.content = content;
  if (content) {
    pg.heads.resize(P->sel.size());
    for (auto& hb : pg.heads) std::memset(&hb, 0, sizeof(HeadBlock));
  }
  return pg;
}

// Per-token quantization of one token into `slot` at the page's width, 4 or 3
// (key design 3; R11), or FP4 (R12: scale in the s entry, zero entry 0).
void write_token(const Pool* P, Page& pg, int slot, const uint16_t* k, const uint16_t* v) {
  const int b = pg.bits;
  float xk[kD], xv[kD];
  for (size_t j = 0; j < P->sel.size(); ++j) {
    HeadBlock& hb = pg.heads[j];
    for (int c = 0; c < kD; ++c) {
      xk[c] = bf16_to_f32(k[j * kD + c]);
      xv[c] = bf16_to_f32(v[j * kD + c]);
    }
    for (int gr = 0; gr < kD / kG; ++gr) {
      if (b == kFP4) {
        fp4_group(xk + gr * kG, kG, 1, hb.kc + slot * kD + gr * kG, 1, &hb.km[(slot * 4 + gr) * 2]);
        fp4_group(xv + gr * kG, kG, 1, hb.vc + slot * kD + gr * kG, 1, &hb.vm[(slot * 4 + gr) * 2]);
        hb.km[(slot * 4 + gr) * 2 + 1] = 0;
        hb.vm[(slot * 4 + gr) * 2 + 1] = 0;
        continue;
      }
      quant_group(xk + gr * kG, kG, 1, b, hb.kc + slot * kD + gr * kG, 1,
                  &hb.km[(slot * 4 + gr) * 2], &hb.km[(slot * 4 + gr) * 2 + 1]);
      quant_group(xv + gr * kG, kG, 1, b, hb.vc + slot * kD + gr * kG, 1,
                  &hb.vm[(slot * 4 + gr) * 2], &hb.vm[(slot * 4 + gr) * 2 + 1]);
    }
  }
}

// Requantize a full INT4 staging page into an INT2 page (key design 3; R4).
void repack_to_int2(const Pool* P, const Page& src, Page& dst) {
  dst.fill = kP;
  dst.live = src.live;
  dst.hdead = src.hdead;
  std::memcpy(dst.pos, src.pos, sizeof(src.pos));
  if (!src.content) return;
  static thread_local float xk[kP * kD], xv[kP * kD];
  for (size_t j = 0; j < P->sel.size(); ++j) {
    const HeadBlock& a = src.heads[j];
    HeadBlock& b = dst.heads[j];
    for (int t = 0; t < kP; ++t)
      for (int c = 0; c < kD; ++c) {
        const int gr = c / kG;
        xk[t * kD + c] = dequant(a.kc[t * kD + c], a.km[(t * 4 + gr) * 2], a.km[(t * 4 + gr) * 2 + 1]);
        xv[t * kD + c] = dequant(a.vc[t * kD + c], a.vm[(t * 4 + gr) * 2], a.vm[(t * 4 + gr) * 2 + 1]);
      }
    // K: per channel, the group is the page's 32 tokens.
    for (int c = 0; c < kD; ++c)
      quant_group(xk + c, kP, kD, 2, b.kc + c, kD, &b.km[c * 2], &b.km[c * 2 + 1]);
    // V: per token, 32 consecutive channels.
    for (int t = 0; t < kP; ++t)
      for (int gr = 0; gr < kD / kG; ++gr)
        quant_group(xv + t * kD + gr * kG, kG, 1, 2, b.vc + t * kD + gr * kG, 1,
                    &b.vm[(t * 4 + gr) * 2], &b.vm[(t * 4 + gr) * 2 + 1]);
  }
}

constexpr uint32_t kDropped = 0xFFFFFFFFu;   // loc entry of a position whose page was dropped

void free_id(Pool* P, int32_t id) {
  P->pages.erase(id);
  if (id < P->n2) P->free2.insert(id);
  else if (id < P->n2 + P->n4) P->free4.insert(id);
  else if (id < P->n2 + P->n4 + P->n3) P->free3.insert(id);
  else P->freef.insert(id);
}

}  // namespace

extern "C" {

// ---- scalar helpers exposed for pins ---------------------------------------
void orc_f32_to_f16(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16(x[i]);
}
void orc_f16_to_f32(const uint16_t* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_to_f32(x[i]);
}
// One FP4 group of n values (R12): codes and the binary16 scale.
int orc_fp4_group(const float* x, int n, uint16_t* s, uint8_t* codes) {
  if (n <= 0) return ORC_INVALID;
  for (int i = 0; i < n; ++i) if (!in_range(x[i])) return ORC_RANGE;
  fp4_group(x, n, 1, codes, 1, s);
  return ORC_OK;
}
double orc_e2m1_value(int code) { return e2m1_value((uint8_t)code); }

// One group of n values at `bits` (2, 3 or 4).
int orc_quant_group(const float* x, int n, int bits, uint16_t* s, uint16_t* z, uint8_t* codes) {
  if (n <= 0 || bits < 2 || bits > 4) return ORC_INVALID;
  for (int i = 0; i < n; ++i) if (!in_range(x[i])) return ORC_RANGE;
  quant_group(x, n, 1, bits, codes, 1, s, z);
  return ORC_OK;
}
float orc_dequant(uint8_t code, uint16_t s, uint16_t z) { return dequant(code, s, z); }

// ---- greedy bit allocation (TriAxialKV key design 2; reading R7) -----------
// bits_out[k] in {2, 4}.  Budget: sum_k N_k b_k <= (B_num / B_den) sum_k N_k.
int orc_alloc_bits(const int64_t* N, const double* D2, const double* D4, int n_tags,
                   int64_t B_num, int64_t B_den, uint8_t* bits_out) {
  if (n_tags <= 0 || B_den <= 0 || B_num < 0) return ORC_INVALID;
  int64_t total = 0;
  for (int k = 0; k < n_tags; ++k) {
    if (N[k] < 0) return ORC_INVALID;
    total += N[k];
    bits_out[k] = 2;
  }
  std::vector<std::pair<double, int>> order;   // (rho, tag)
  for (int k = 0; k < n_tags; ++k)
    if (N[k] > 0) order.push_back({(D2[k] - D4[k]) / (2.0 * (double)N[k]), k});
  std::stable_sort(order.begin(), order.end(), [](const std::pair<double, int>& a,
                                                  const std::pair<double, int>& b) {
    if (a.first != b.first) return a.first > b.first;  // descending rho
    return a.second < b.second;                         // ties: ascending tag id
  });
  int64_t used = 2 * total;
  for (const auto& e : order) {
    const int64_t extra = 2 * N[e.second];
    if ((used + extra) * B_den <= B_num * total) {
      bits_out[e.second] = 4;
      used += extra;
    }
  }
  return ORC_OK;
}

// Greedy allocation over three widths (R13): bits_out[k] in {2, 3, 4}.
int orc_alloc_bits3(const int64_t* N, const double* D2, const double* D3, const double* D4, int n_tags,
                    int64_t B_num, int64_t B_den, uint8_t* bits_out) {
  if (n_tags <= 0 || B_den <= 0 || B_num < 0) return ORC_INVALID;
  int64_t total = 0;
  for (int k = 0; k < n_tags; ++k) {
    if (N[k] < 0) return ORC_INVALID;
    total += N[k];
    bits_out[k] = 2;
  }
  // open[k]: the width tag k's next step starts from (2 or 3), 0 when it has none
  std::vector<int> open(n_tags, 0);
  for (int k = 0; k < n_tags; ++k) open[k] = N[k] > 0 ? 2 : 0;
  int64_t used = 2 * total;
  for (;;) {
    int best = -1;
    double best_rho = 0.0;
    for (int k = 0; k < n_tags; ++k) {
      if (!open[k]) continue;
      const double saving = open[k] == 2 ? D2[k] - D3[k] : D3[k] - D4[k];
      const double rho = saving / (double)N[k];
      if (best < 0 || rho > best_rho) { best = k; best_rho = rho; }   // ties keep the lower tag
    }
    if (best < 0) break;
    if ((used + N[best]) * B_den <= B_num * total) {
      used += N[best];
      bits_out[best] = (uint8_t)(open[best] + 1);
      open[best] = open[best] == 2 ? 3 : 0;
    } else {
      open[best] = 0;                                 // dropped: and so is its 3 -> 4 step
    }
  }
  return ORC_OK;
}

// ---- pool --------------------------------------------------------------------
// sel_heads: kv heads whose codes are materialized (n_sel of them); page ids,
// tables, fills and live masks are modelled for every head regardless.
void* orc_pool_new(int hkv, int64_t n2, int64_t n3, int64_t nf, int64_t n4, int max_req, int max_pages,
                   const int* sel_heads, int n_sel) {
  if (hkv <= 0 || n2 < 0 || n3 < 0 || nf < 0 || n4 < 0 || max_req <= 0 || max_pages <= 0) return nullptr;
  Pool* P = new Pool();
  P->hkv = hkv;
  P->n2 = n2;
  P->n3 = n3;
  P->nf = nf;
  P->n4 = n4;
  P->max_req = max_req;
  P->max_pages = max_pages;
  for (int i = 0; i < n_sel; ++i) P->sel.push_back(sel_heads[i]);
  for (int64_t i = 0; i < n2; ++i) P->free2.insert((int32_t)i);
  for (int64_t i = 0; i < n4; ++i) P->free4.insert((int32_t)(n2 + i));
  for (int64_t i = 0; i < n3; ++i) P->free3.insert((int32_t)(n2 + n4 + i));
  for (int64_t i = 0; i < nf; ++i) P->freef.insert((int32_t)(n2 + n4 + n3 + i));
  P->reqs.resize(max_req);
  return P;
}

void orc_pool_free(void* h) { delete (Pool*)h; }

int orc_request_open(void* h, int32_t* id_out) {
  Pool* P = (Pool*)h;
  for (int r = 0; r < P->max_req; ++r)
    if (!P->reqs[r].open) {
      P->reqs[r] = Req();
      P->reqs[r].open = true;
      *id_out = r;
      return ORC_OK;
    }
  return ORC_OOM;
}

int orc_request_close(void* h, int32_t id) {
  Pool* P = (Pool*)h;
  if (id < 0 || id >= P->max_req || !P->reqs[id].open) return ORC_INVALID;
  for (int32_t pid : P->reqs[id].table) free_id(P, pid);
  P->reqs[id] = Req();
  return ORC_OK;
}

// Append n tokens in arrival order (TriAxialKV key designs 3-4; readings R4, R5, R11).
// k, v: bf16 bits [n][n_sel][128] for the selected heads, or both NULL to model
// page ids and tables only.  Returns ORC_INVALID / ORC_RANGE / ORC_OOM with no
// change to the pool.
int orc_append(void* h, const uint16_t* k, const uint16_t* v, const int32_t* req,
               const uint8_t* bits, int64_t n) {
  Pool* P = (Pool*)h;
  const bool content = (k != nullptr && v != nullptr);
  const size_t nsel = P->sel.size();
  for (int64_t t = 0; t < n; ++t) {
    if (req[t] < 0 || req[t] >= P->max_req || !P->reqs[req[t]].open) return ORC_INVALID;
    if ((bits[t] < 2 || bits[t] > 4) && bits[t] != kFP4) return ORC_INVALID;
  }
  if (content)
    for (int64_t i = 0; i < n * (int64_t)nsel * kD; ++i)
      if (!in_range(bf16_to_f32(k[i])) || !in_range(bf16_to_f32(v[i]))) return ORC_RANGE;
  // Dry run: count the pages this call takes and the table growth.
  struct Sim {
    bool tail = false; int tailfill = 0; bool tail3 = false; int tail3fill = 0; bool tailf = false; int tailffill = 0;
    bool stag = false; int stagfill = 0; int64_t tablen = 0;
  };
  std::unordered_map<int32_t, Sim> sim;
  int64_t need4 = 0, need3 = 0, needf = 0, need2 = 0;
  for (int64_t t = 0; t < n; ++t) {
    auto it = sim.find(req[t]);
    if (it == sim.end()) {
      const Req& R = P->reqs[req[t]];
      Sim s;
      if (R.tail4 >= 0) { s.tail = true; s.tailfill = P->pages.at(R.tail4).fill; }
      if (R.tail3 >= 0) { s.tail3 = true; s.tail3fill = P->pages.at(R.tail3).fill; }
      if (R.tailf >= 0) { s.tailf = true; s.tailffill = P->pages.at(R.tailf).fill; }
      if (R.staging >= 0) { s.stag = true; s.stagfill = P->pages.at(R.staging).fill; }
      s.tablen = (int64_t)R.table.size();
      it = sim.emplace(req[t], s).first;
    }
    Sim& s = it->second;
    if (bits[t] == 4) {
      if (!s.tail || s.tailfill == kP) { ++need4; ++s.tablen; s.tail = true; s.tailfill = 0; }
      ++s.tailfill;
    } else if (bits[t] == 3) {
      if (!s.tail3 || s.tail3fill == kP) { ++need3; ++s.tablen; s.tail3 = true; s.tail3fill = 0; }
      ++s.tail3fill;
    } else if (bits[t] == kFP4) {
      if (!s.tailf || s.tailffill == kP) { ++needf; ++s.tablen; s.tailf = true; s.tailffill = 0; }
      ++s.tailffill;
    } else {
      if (!s.stag) { ++need4; ++s.tablen; s.stag = true; s.stagfill = 0; }
      if (++s.stagfill == kP) { ++need2; s.stag = false; }
    }
    if (s.tablen > P->max_pages) return ORC_OOM;
  }
  if (need4 > (int64_t)P->free4.size() || need3 > (int64_t)P->free3.size() || needf > (int64_t)P->freef.size() ||
      need2 > (int64_t)P->free2.size())
    return ORC_OOM;

  std::vector<int32_t> deferred;
  for (int64_t t = 0; t < n; ++t) {
    Req& R = P->reqs[req[t]];
    const int64_t pos = (int64_t)R.loc.size();
    const uint16_t* kt = content ? k + (size_t)t * nsel * kD : nullptr;
    const uint16_t* vt = content ? v + (size_t)t * nsel * kD : nullptr;
    // INT4 and INT2 tokens go to INT4 pages (the tail, the staging page); INT3
    // and FP4 tokens to their own tails
    int32_t& cur = bits[t] == 4 ? R.tail4 : (bits[t] == 3 ? R.tail3 : (bits[t] == kFP4 ? R.tailf : R.staging));
    if (cur < 0 || P->pages.at(cur).fill == kP) {
      Page& pg = new_page(P, bits[t] == 2 ? 4 : bits[t], content);
      cur = pg.id;
      R.table.push_back(pg.id);
    }
    Page& pg = P->pages.at(cur);
    const int slot = pg.fill++;
    pg.live |= 1u << slot;
    pg.pos[slot] = pos;
    if (pg.content && content) write_token(P, pg, slot, kt, vt);
    else if (pg.content) { pg.content = false; pg.heads.clear(); }
    R.loc.push_back(((uint32_t)pg.id << 5) | (uint32_t)slot);
    if (bits[t] == 2 && pg.fill == kP) {
      Page& np = new_page(P, 2, pg.content);
      repack_to_int2(P, pg, np);
      for (int s = 0; s < kP; ++s) R.loc[np.pos[s]] = ((uint32_t)np.id << 5) | (uint32_t)s;
      R.table.erase(std::find(R.table.begin(), R.table.end(), pg.id));
      R.table.push_back(np.id);
      deferred.push_back(pg.id);
      R.staging = -1;
    }
  }
  for (int32_t id : deferred) free_id(P, id);
  return ORC_OK;
}

// INT2-first stable reorder of each listed request's table (TriAxialKV key
// design 4, phase 1); with INT3 or FP4 pages the table is sorted stably by
// width: INT2, INT3, INT4, FP4 (R11, R12).
int orc_reorder(void* h, const int32_t* req, int n) {
  Pool* P = (Pool*)h;
  for (int i = 0; i < n; ++i)
    if (req[i] < 0 || req[i] >= P->max_req || !P->reqs[req[i]].open) return ORC_INVALID;
  for (int i = 0; i < n; ++i) {
    auto& tb = P->reqs[req[i]].table;
    std::stable_sort(tb.begin(), tb.end(),
                     [P](int32_t a, int32_t b) { return P->pages.at(a).bits < P->pages.at(b).bits; });   // kFP4 > 4
  }
  return ORC_OK;
}

// Evict token positions (IntentKV, layout-preserving eviction): clear live bits only.
int orc_evict(void* h, const int32_t* req, const int64_t* pos, int64_t n) {
  Pool* P = (Pool*)h;
  for (int64_t i = 0; i < n; ++i) {
    if (req[i] < 0 || req[i] >= P->max_req || !P->reqs[req[i]].open) return ORC_INVALID;
    if (pos[i] < 0 || pos[i] >= (int64_t)P->reqs[req[i]].loc.size()) return ORC_INVALID;
  }
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t l = P->reqs[req[i]].loc[pos[i]];
    if (l == kDropped) continue;                    // its page was dropped: already dead
    P->pages.at((int32_t)(l >> 5)).live &= ~(1u << (l & 31u));
  }
  return ORC_OK;
}

// Drop dead pages (R10).  For each listed request, every full page (32 slots
// written) none of whose slots is live for any kv head (evicted, or excluded
// for every head) leaves the table; the other entries keep their order and
// their pages stay where they are (IntentKV method 2: surviving pages do not
// move).  The dropped ids return to the free sets, and the positions they
// held read as dropped (evicting them again changes nothing).
int orc_drop_dead_pages(void* h, const int32_t* req, int n) {
  Pool* P = (Pool*)h;
  for (int i = 0; i < n; ++i)
    if (req[i] < 0 || req[i] >= P->max_req || !P->reqs[req[i]].open) return ORC_INVALID;
  for (int i = 0; i < n; ++i) {
    Req& R = P->reqs[req[i]];
    std::vector<int32_t> keep;
    for (int32_t id : R.table) {
      const Page& pg = P->pages.at(id);
      bool dead = pg.fill == kP;
      for (int hh = 0; hh < P->hkv && dead; ++hh) dead = (pg.live & ~pg.hdead[(size_t)hh]) == 0u;
      if (!dead) {
        keep.push_back(id);
        continue;
      }
      for (int s = 0; s < kP; ++s) R.loc[(size_t)pg.pos[s]] = kDropped;
      if (R.tail4 == id) R.tail4 = -1;
      if (R.tail3 == id) R.tail3 = -1;
      if (R.tailf == id) R.tailf = -1;
      if (R.staging == id) R.staging = -1;
      free_id(P, id);
    }
    R.table = keep;
  }
  return ORC_OK;
}

// Exclude token positions for one kv head each (HyQuant: a vertical-line
// token of a head leaves that head's quantized set; R9).
int orc_evict_head(void* h, const int32_t* req, const int64_t* pos, const int32_t* kvh, int64_t n) {
  Pool* P = (Pool*)h;
  for (int64_t i = 0; i < n; ++i) {
    if (req[i] < 0 || req[i] >= P->max_req || !P->reqs[req[i]].open) return ORC_INVALID;
    if (pos[i] < 0 || pos[i] >= (int64_t)P->reqs[req[i]].loc.size()) return ORC_INVALID;
    if (kvh[i] < 0 || kvh[i] >= P->hkv) return ORC_INVALID;
  }
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t l = P->reqs[req[i]].loc[pos[i]];
    if (l == kDropped) continue;                    // its page was dropped: already dead for every head
    P->pages.at((int32_t)(l >> 5)).hdead[(size_t)kvh[i]] |= 1u << (l & 31u);
  }
  return ORC_OK;
}

// Append n full-precision tokens to a request's list (R8).  k, v: bf16 bits
// [n][n_sel][128], the rows of the selected heads.
int orc_fp_append(void* h, int32_t id, const uint16_t* k, const uint16_t* v, int64_t n) {
  Pool* P = (Pool*)h;
  if (id < 0 || id >= P->max_req || !P->reqs[id].open || n < 0 || (n > 0 && (!k || !v))) return ORC_INVALID;
  Req& R = P->reqs[id];
  const size_t m = (size_t)n * P->sel.size() * kD;
  R.fpk.insert(R.fpk.end(), k, k + m);
  R.fpv.insert(R.fpv.end(), v, v + m);
  R.n_fp += n;
  return ORC_OK;
}

// Remove full-precision tokens [first, first + n) of a request's list; the
// rest keep their order (R8).
int orc_fp_drop(void* h, int32_t id, int64_t first, int64_t n) {
  Pool* P = (Pool*)h;
  if (id < 0 || id >= P->max_req || !P->reqs[id].open) return ORC_INVALID;
  Req& R = P->reqs[id];
  if (first < 0 || n < 0 || first + n > R.n_fp) return ORC_INVALID;
  const size_t row = P->sel.size() * kD;
  R.fpk.erase(R.fpk.begin() + (ptrdiff_t)(first * row), R.fpk.begin() + (ptrdiff_t)((first + n) * row));
  R.fpv.erase(R.fpv.begin() + (ptrdiff_t)(first * row), R.fpv.begin() + (ptrdiff_t)((first + n) * row));
  R.n_fp -= n;
  return ORC_OK;
}

int orc_request_info(void* h, int32_t id, int32_t* n_pages, int64_t* n_tok) {
  Pool* P = (Pool*)h;
  if (id < 0 || id >= P->max_req || !P->reqs[id].open) return ORC_INVALID;
  *n_pages = (int32_t)P->reqs[id].table.size();
  *n_tok = (int64_t)P->reqs[id].loc.size();
  return ORC_OK;
}

// Canonical export of one request, pages in table order.  Content arrays are
// [n_pages][n_sel][32][128] (codes) and [n_pages][n_sel][256] (meta); pass NULL
// to skip them.
int orc_export(void* h, int32_t id, int32_t* ids, uint8_t* is_int2, uint8_t* fill, uint32_t* live,
               uint8_t* kc, uint8_t* vc, uint16_t* km, uint16_t* vm) {
  Pool* P = (Pool*)h;
  if (id < 0 || id >= P->max_req || !P->reqs[id].open) return ORC_INVALID;
  const auto& tb = P->reqs[id].table;
  const size_t nsel = P->sel.size();
  for (size_t i = 0; i < tb.size(); ++i) {
    const Page& pg = P->pages.at(tb[i]);
    ids[i] = pg.id;
    is_int2[i] = pg.bits == 2 ? 1 : 0;
    fill[i] = (uint8_t)pg.fill;
    live[i] = pg.live;
    if (kc) {
      if (!pg.content) return ORC_STATE;
      for (size_t j = 0; j < nsel; ++j) {
        const HeadBlock& hb = pg.heads[j];
        std::memcpy(kc + (i * nsel + j) * kP * kD, hb.kc, kP * kD);
        std::memcpy(vc + (i * nsel + j) * kP * kD, hb.vc, kP * kD);
        std::memcpy(km + (i * nsel + j) * 256, hb.km, 512);
        std::memcpy(vm + (i * nsel + j) * 256, hb.vm, 512);
      }
    }
  }
  return ORC_OK;
}

// Decode attention in fp64 for the listed (batch row, q head) pairs.
// q: bf16 bits [B][Hq][128]; kv head of q head hq is hq / (Hq / Hkv).
// n_splits <= 1: one softmax pass.  n_splits > 1: the token sequence (table
// order, slot order, then the full-precision list) is cut into n_splits
// contiguous chunks; each chunk keeps
// (m, l, acc) and the chunks are merged by log-sum-exp (HyQuant, online
// softmax and Algorithm 3 ReduceSoftmax).  A request with no tokens gives 0.
// out: [n_pairs][128].
int orc_decode(void* h, const uint16_t* q, const int32_t* req, int B, int Hq, float scale,
               const int32_t* pairs, int n_pairs, int n_splits, double* out, int n_threads) {
  Pool* P = (Pool*)h;
  if (Hq <= 0 || Hq % P->hkv != 0) return ORC_INVALID;
  const int g = Hq / P->hkv;
  for (int i = 0; i < n_pairs; ++i) {
    const int b = pairs[2 * i], hq = pairs[2 * i + 1];
    if (b < 0 || b >= B || hq < 0 || hq >= Hq) return ORC_INVALID;
    const int r = req[b];
    if (r < 0 || r >= P->max_req || !P->reqs[r].open) return ORC_INVALID;
    if (std::find(P->sel.begin(), P->sel.end(), hq / g) == P->sel.end()) return ORC_INVALID;
    for (int32_t pid : P->reqs[r].table) if (!P->pages.at(pid).content) return ORC_STATE;
  }
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int i = 0; i < n_pairs; ++i) {
    const int b = pairs[2 * i], hq = pairs[2 * i + 1];
    const Req& R = P->reqs[req[b]];
    const int kv = hq / g;
    const size_t j = (size_t)(std::find(P->sel.begin(), P->sel.end(), kv) - P->sel.begin());
    double qd[kD];
    for (int c = 0; c < kD; ++c) qd[c] = (double)bf16_to_f32(q[((size_t)b * Hq + hq) * kD + c]);
    // Token list: the quantized tokens in table order, then the
    // full-precision tokens in list order (R8).  Per token: logit, source of
    // V (page block and slot, or a bf16 row), live.
    std::vector<double> logit;
    std::vector<std::pair<const HeadBlock*, int>> src;
    std::vector<const uint16_t*> fprow;
    std::vector<bool> alive, vfp4;   // vfp4: V of an FP4 page (R12)
    for (int32_t pid : R.table) {
      const Page& pg = P->pages.at(pid);
      const HeadBlock& hb = pg.heads[j];
      const uint32_t live = pg.live & ~pg.hdead[(size_t)kv];   // R9
      for (int s = 0; s < pg.fill; ++s) {
        const bool lv = (live >> s) & 1u;
        double l = -1e4;                                   // sentinel dead slot (R6)
        if (lv) {
          double acc = 0.0;
          for (int c = 0; c < kD; ++c) {
            const int mi = pg.bits == 2 ? c * 2 : (s * 4 + c / kG) * 2;
            const float kh = pg.bits == kFP4 ? dequant_fp4(hb.kc[s * kD + c], hb.km[mi])
                                             : dequant(hb.kc[s * kD + c], hb.km[mi], hb.km[mi + 1]);
            acc += qd[c] * (double)kh;
          }
          l = (double)scale * acc;
        }
        logit.push_back(l);
        src.push_back({&hb, s});
        fprow.push_back(nullptr);
        alive.push_back(lv);
        vfp4.push_back(pg.bits == kFP4);
      }
    }
    const size_t nsel = P->sel.size();
    for (int64_t t = 0; t < R.n_fp; ++t) {
      const uint16_t* kr = R.fpk.data() + ((size_t)t * nsel + j) * kD;
      double acc = 0.0;
      for (int c = 0; c < kD; ++c) acc += qd[c] * (double)bf16_to_f32(kr[c]);
      logit.push_back((double)scale * acc);
      src.push_back({nullptr, 0});
      fprow.push_back(R.fpv.data() + ((size_t)t * nsel + j) * kD);
      alive.push_back(true);
      vfp4.push_back(false);
    }
    double* o = out + (size_t)i * kD;
    for (int c = 0; c < kD; ++c) o[c] = 0.0;
    const int64_t T = (int64_t)logit.size();
    if (T == 0) continue;
    const int S = n_splits <= 1 ? 1 : n_splits;
    std::vector<double> ms, ls, accs;
    for (int sp = 0; sp < S; ++sp) {
      const int64_t a = T * sp / S, e = T * (sp + 1) / S;
      if (a == e) continue;
      double m = -INFINITY;
      for (int64_t t = a; t < e; ++t) m = std::max(m, logit[t]);
      double l = 0.0, acc[kD] = {0.0};
      for (int64_t t = a; t < e; ++t) {
        const double w = std::exp(logit[t] - m);
        l += w;
        if (!alive[t]) continue;                           // V = 0 at the dead slot
        if (fprow[t]) {
          for (int c = 0; c < kD; ++c) acc[c] += w * (double)bf16_to_f32(fprow[t][c]);
          continue;
        }
        const HeadBlock& hb = *src[t].first;
        const int s = src[t].second;
        const bool f4 = vfp4[t];
        for (int c = 0; c < kD; ++c) {
          const int mi = (s * 4 + c / kG) * 2;
          acc[c] += w * (double)(f4 ? dequant_fp4(hb.vc[s * kD + c], hb.vm[mi])
                                    : dequant(hb.vc[s * kD + c], hb.vm[mi], hb.vm[mi + 1]));
        }
      }
      ms.push_back(m);
      ls.push_back(l);
      accs.insert(accs.end(), acc, acc + kD);
    }
    double M = -INFINITY;
    for (double m : ms) M = std::max(M, m);
    double L = 0.0;
    for (size_t k2 = 0; k2 < ms.size(); ++k2) {
      const double f = std::exp(ms[k2] - M);
      L += ls[k2] * f;
      for (int c = 0; c < kD; ++c) o[c] += accs[k2 * kD + c] * f;
    }
    for (int c = 0; c < kD; ++c) o[c] /= L;
  }
  return ORC_OK;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
