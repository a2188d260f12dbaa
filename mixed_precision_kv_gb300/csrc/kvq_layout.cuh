// Physical byte layout of one (page, kv head) block.  Private to the library:
// kv_export_request() converts it to the canonical (slot, channel) form.
//
// The layout is chosen for the tensor-core decode kernel's fragment ownership
// (mma.m16n8k16, lane = 4*r + i): every lane reads its codes with 16-byte
// shared-memory loads that hit 8 distinct 16-byte bank groups per quarter
// warp, and one 32-bit code word unpacks into whole A-fragment registers with
// a shift and a mask each: a field at bits p..p+w-1 of both 16-bit halves is
// the binary16 subnormal code * 2^(p-24) (p >= 4, so the field's top bit is at
// bit 7 or above).
//
// INT4 block (5120 B)
//   [   0, 2048) K codes: slot t row at 64*t; row = 4 chunks (i) x 4 groups
//                (gr) x 4 bytes; channel c = 32*gr + 8*i + n sits in nibble n
//                (bits 4n..4n+3) of word (i, gr).
//   [2048, 4096) V codes, channel-major: word (channel c, slot chunk j) holds
//                slots 8j..8j+7 in nibbles 0..7.  With c = 16m + 8e + r
//                (m < 8, e < 2, r < 8) it sits at 16-byte chunk
//                32*(m>>1) + 4*r + j, word 2*(m&1) + e inside the chunk, so the
//                16 channels of one tensor-core M tile (16m .. 16m+15) stay in
//                one 32-channel group.
//   [4096, 4608) K scale/zero: [slot][group] half2 {scale, zero}.
//   [4608, 5120) V scale/zero: scales [group][32] half then zeros [group][32]
//                half, slot order inside each 8-slot chunk j permuted so that
//                position 2k holds slot 8j+k and 2k+1 holds slot 8j+k+4.
// INT2 block (3072 B)
//   [   0, 1024) K codes: slot t row at 32*t; channel c at byte c>>2, bits
//                2*(c&3).
//   [1024, 2048) V codes, channel-major: word (r, m, i) holds channels
//                16m+r (bytes 0, 2) and 16m+r+8 (bytes 1, 3) for slot chunk i:
//                byte 0/1 hold slots 8i..8i+3, bytes 2/3 slots 8i+4..8i+7,
//                slot 8i+k at bits 2k of its byte, except that channel
//                16m+r keeps slot 8i in byte 2 and slot 8i+4 in byte 0 (a
//                byte rotation of the word then lines both up with channel
//                16m+r+8).  The word sits at 16-byte chunk 32*(m>>2) + 4*r + i,
//                word m&3 inside the chunk.
//   [2048, 2560) K scales: 128 halves in pair order, then zeros in the same
//                order.  Pair p = (i*2 + wi)*8 + j holds the channels that
//                A-register j of code word (chunk i, word wi) carries: low half
//                = channel 4*(8i + 4wi + (j>>2)) + (j&3), high half = that + 8;
//                pair j = 0 has the two halves the other way round.
//   [2560, 3072) V scale/zero: as in the INT4 block.
// INT3 block (4096 B): the INT4 block's code words with each 4-bit field cut
// into a 2-bit plane (the code's low bits) and a 1-bit plane (bit 2), so
// that one shift + mask of each plane puts both parts of a code at bits
// 6..8 of a 16-bit half, the same A-register fields as INT4 (at bit 6).
//   [   0, 1536) K codes: slot t row at 48*t.  Low plane at 8*i (chunk i):
//                word h (groups 2h, 2h+1) holds the low bits of channel
//                c = 32*gr + 8*i + n at bit 8*(gr&1) + 2*(n&3) + 16*(n>>2).
//                High plane at 32 + 4*i: bit 2 of channel c at bit
//                4*gr + (n&3) + 16*(n>>2).
//   [1536, 3072) V codes, channel-major: INT4 V chunk X = 32*(m>>1) + 4*r + j
//                (channels c = 16m + 8e + r, slots 8j..8j+7, INT4 word
//                w = 2*(m&1) + e) becomes a low-plane uint2 at 1536 + 8*X, word
//                m&1 holding slot 8j+k of channel e at bit
//                8*e + 2*(k&3) + 16*(k>>2), and a high-plane word at
//                2560 + 4*X with bit 4*w + (k&3) + 16*(k>>2).
//   [3072, 3584) K scale/zero: as in the INT4 block ([slot][group] {s, z}).
//   [3584, 4096) V scale/zero: as in the INT4 block.
// FP4 block (4608 B): E2M1 codes (sign << 3 | exponent << 1 | mantissa) in
// the INT4 block's code words, but with the two channels (K) or slots (V)
// that one mma A register pairs sharing a byte, so that one e2m1x2 -> f16x2
// conversion yields the register: byte n of a word holds element n (low
// nibble) and element n + 4 (high nibble).  Symmetric groups: scales only.
//   [   0, 2048) K codes: slot t row at 64*t, chunk i at 16*i, word gr holds
//                channel 32*gr + 8*i + n in byte n & 3, nibble n >> 2.
//   [2048, 4096) V codes: INT4 V chunk X and word w as in the INT4 block,
//                slot 8j + k in byte k & 3, nibble k >> 2.
//   [4096, 4352) K scales: [slot][group] half.
//   [4352, 4608) V scales: [group][32] half in the INT4 V scale order.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define KVQ_HD __host__ __device__ __forceinline__
#else
#define KVQ_HD inline
#endif

namespace kvq {

constexpr int kHeadDim = 128;
constexpr int kPage = 32;
constexpr int kGroup = 32;
constexpr int kInt4Block = 5120;
constexpr int kInt2Block = 3072;
constexpr int kInt3Block = 4096;
constexpr int kFp4Block = 4608;

// INT4 block offsets
constexpr int kI4KCodes = 0, kI4VCodes = 2048, kI4KMeta = 4096, kI4VMeta = 4608;
// INT2 block offsets
constexpr int kI2KCodes = 0, kI2VCodes = 1024, kI2KMeta = 2048, kI2VMeta = 2560;
// INT3 block offsets (kI3VHigh: the V high plane)
constexpr int kI3KCodes = 0, kI3VCodes = 1536, kI3VHigh = 2560, kI3KMeta = 3072, kI3VMeta = 3584;
// FP4 block offsets
constexpr int kF4KCodes = 0, kF4VCodes = 2048, kF4KScale = 4096, kF4VScale = 4352;

// ---- INT4 K codes: byte offset and nibble of (slot, channel)
KVQ_HD int i4k_byte(int t, int c) {
  const int gr = c >> 5, i = (c >> 3) & 3, n = c & 7;
  return kI4KCodes + 64 * t + 16 * i + 4 * gr + (n >> 1);
}
KVQ_HD int i4k_shift(int c) { return 4 * (c & 1); }

// ---- INT4 V codes
KVQ_HD int i4v_byte(int t, int c) {
  const int j = t >> 3, n = t & 7;
  const int m = c >> 4, e = (c >> 3) & 1, r = c & 7;
  return kI4VCodes + 16 * (32 * (m >> 1) + 4 * r + j) + 4 * (2 * (m & 1) + e) + (n >> 1);
}
KVQ_HD int i4v_shift(int t) { return 4 * (t & 1); }

// ---- INT2 K codes
KVQ_HD int i2k_byte(int t, int c) { return kI2KCodes + 32 * t + (c >> 2); }
KVQ_HD int i2k_shift(int c) { return 2 * (c & 3); }

// ---- INT2 V codes
KVQ_HD int i2v_byte(int t, int c) {
  const int m = c >> 4, e = (c >> 3) & 1, r = c & 7;
  const int i = t >> 3, k = t & 7;
  const int half = (k >> 2) ^ ((e == 0 && (k & 3) == 0) ? 1 : 0);
  return kI2VCodes + 16 * (32 * (m >> 2) + 4 * r + i) + 4 * (m & 3) + e + 2 * half;
}
KVQ_HD int i2v_shift(int t) { return 2 * (t & 3); }

// ---- INT2 K scale/zero: half index (0..127) of channel c in the pair order
KVQ_HD int i2k_meta_index(int c) {
  const int i = c >> 5, wi = (c >> 4) & 1, b = (c >> 2) & 3, pos = c & 3;
  const int j = (b & 1) * 4 + pos;      // bytes 0,2 -> regs 0..3; bytes 1,3 -> regs 4..7
  const int hi = (b >> 1) ^ (j == 0 ? 1 : 0);   // bytes 2,3 are the high half (swapped for j = 0)
  return 2 * ((i * 2 + wi) * 8 + j) + hi;
}

// ---- INT3 K codes: byte and bit of the low 2 bits / of bit 2 of (slot, channel)
KVQ_HD int i3k_lo_byte(int t, int c) {
  const int gr = c >> 5, i = (c >> 3) & 3, n = c & 7;
  return kI3KCodes + 48 * t + 8 * i + 4 * (gr >> 1) + (gr & 1) + 2 * (n >> 2);
}
KVQ_HD int i3k_lo_shift(int c) { return 2 * (c & 3); }
KVQ_HD int i3k_hi_byte(int t, int c) {
  const int gr = c >> 5, i = (c >> 3) & 3, n = c & 7;
  return kI3KCodes + 48 * t + 32 + 4 * i + (gr >> 1) + 2 * (n >> 2);
}
KVQ_HD int i3k_hi_shift(int c) { return 4 * ((c >> 5) & 1) + (c & 3); }

// ---- INT3 V codes
KVQ_HD int i3v_chunk(int t, int c) {
  const int m = c >> 4, r = c & 7;
  return 32 * (m >> 1) + 4 * r + (t >> 3);
}
KVQ_HD int i3v_lo_byte(int t, int c) {
  const int m = c >> 4, e = (c >> 3) & 1, k = t & 7;
  return kI3VCodes + 8 * i3v_chunk(t, c) + 4 * (m & 1) + e + 2 * (k >> 2);
}
KVQ_HD int i3v_lo_shift(int t) { return 2 * (t & 3); }
KVQ_HD int i3v_hi_byte(int t, int c) {
  const int m = c >> 4, e = (c >> 3) & 1, k = t & 7;
  const int w = 2 * (m & 1) + e;
  return kI3VHigh + 4 * i3v_chunk(t, c) + (w >> 1) + 2 * (k >> 2);
}
KVQ_HD int i3v_hi_shift(int t, int c) {
  const int m = c >> 4, e = (c >> 3) & 1;
  return 4 * ((2 * (m & 1) + e) & 1) + (t & 3);
}

// ---- FP4 K / V codes: byte and nibble shift of (slot, channel)
KVQ_HD int f4k_byte(int t, int c) {
  const int gr = c >> 5, i = (c >> 3) & 3, n = c & 7;
  return kF4KCodes + 64 * t + 16 * i + 4 * gr + (n & 3);
}
KVQ_HD int f4k_shift(int c) { return 4 * ((c >> 2) & 1); }
KVQ_HD int f4v_byte(int t, int c) {
  const int j = t >> 3, k = t & 7;
  const int m = c >> 4, e = (c >> 3) & 1, r = c & 7;
  return kF4VCodes + 16 * (32 * (m >> 1) + 4 * r + j) + 4 * (2 * (m & 1) + e) + (k & 3);
}
KVQ_HD int f4v_shift(int t) { return 4 * ((t >> 2) & 1); }
// E2M1 value of a code (exponent 0: 0 or the subnormal 0.5)
KVQ_HD float e2m1_value(uint32_t code) {
  const uint32_t e = (code >> 1) & 3u, f = code & 1u;
  const float mag = e == 0 ? 0.5f * (float)f : (1.0f + 0.5f * (float)f) * (float)(1u << (e - 1));
  return (code & 8u) ? -mag : mag;
}

// ---- V scale/zero (every width): half index (0..127) of (slot, group)
KVQ_HD int v_meta_index(int t, int gr) {
  const int j = t >> 3, k = t & 7;
  const int pos = (k < 4) ? 2 * k : 2 * (k - 4) + 1;
  return 32 * gr + 8 * j + pos;
}

}  // namespace kvq
