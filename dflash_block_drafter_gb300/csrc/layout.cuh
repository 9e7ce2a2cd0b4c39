// The library's "fragment-native" streaming layout of a backbone matrix and
// the in-register decoders that turn it into mma.sync m16n8k16 A fragments.
//
// Why: the draft pass multiplies at most 8 activation rows per sequence by
// each weight matrix, so every matrix is streamed from HBM exactly once per
// pass and the kernels are bandwidth bound.  The layout makes every streamed
// byte land, with one 16-byte shared-memory load per lane, in the registers
// of the lane whose MMA fragment needs it, and makes each CTA's share of a
// matrix one contiguous byte range (one bulk copy per unit).
//
// Geometry.  A matrix W [N, K] (N % 64 == 0, K % 256 == 0) is cut into
// groups of 64 rows; a group is 4 m-tiles of 16 rows.  K is cut into 32-wide
// blocks (the GGUF block size).  Inside a 32-block, lane (r = lane/4,
// c = lane%4) of the warp that owns an m-tile takes the 8 consecutive inputs
// 8c .. 8c+7 of rows r and r+8.  The MMA's 16-wide K slots are mapped onto
// those physical inputs identically for A (weights) and B (activations):
//     k-step s (0, 1), slot 2c+j -> 8c + 4s + j,  slot 2c+8+j -> 8c + 4s + 2 + j
// so the product over slots equals the product over the block's 32 inputs.
//
// A "unit" (CB blocks x 64 rows) is the streaming granule; units are stored
// group-major: unit (g, j) at byte (g * UPG + j) * UNIT, UPG = K / (32 CB).
// Inside a unit, sub-chunks of SUBB blocks x one m-tile are stored at
// (sc * 4 + mtile) * CHUNK:
//   BF16 (CB 4, SUBB 1, CHUNK 1024): [lane][8 x bf16 of row r] (512 B) then
//        [lane][8 x bf16 of row r+8] (512 B).
//   Q8_0 (CB 8, SUBB 1, CHUNK 544): [lane][8 codes row r | 8 codes row r+8]
//        (codes biased by +128, u8) then 8 x (d[r], d[r+8]) FP16.
//   Q4_0 (CB 8, SUBB 2, CHUNK 576): [lane][4 words]: (row r, block A),
//        (row r, block B), (row r+8, A), (row r+8, B); a word holds the 8
//        nibble codes e0..e7 in the order e0 e2 e4 e6 e1 e3 e5 e7 (low
//        nibble first) so that (w >> 4j) & 0x000F000F selects (e2j, e2j+1);
//        then 8 x (dA[r], dA[r+8], dB[r], dB[r+8]) FP16.
//   Q5_0 (CB 8, SUBB 2, CHUNK 704): the Q4_0 nibbles of the low four bits,
//        then [lane][u32 fifth bits]: for (half h, block b) at offset
//        o = (2h + b) * 4 bit o + j is e2j's and bit o + 16 + j is e2j+1's,
//        then the scales as Q4_0.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace dflash {

template <int WT>
struct Fmt;

template <>
struct Fmt<WT_BF16> {
  static constexpr int CB = 4, SUBB = 1, CHUNK = 1024, STAGES = 9;
  static constexpr int UNIT = (CB / SUBB) * 4 * CHUNK;  // 16384
  static constexpr bool kF16 = false;                   // activations bf16
};
template <>
struct Fmt<WT_Q8_0> {
  static constexpr int CB = 8, SUBB = 1, CHUNK = 544, STAGES = 8;
  static constexpr int UNIT = (CB / SUBB) * 4 * CHUNK;  // 17408
  static constexpr bool kF16 = true;
};
template <>
struct Fmt<WT_Q4_0> {
  static constexpr int CB = 8, SUBB = 2, CHUNK = 576, STAGES = 13;
  static constexpr int UNIT = (CB / SUBB) * 4 * CHUNK;  // 9216
  static constexpr bool kF16 = true;
};
template <>
struct Fmt<WT_Q5_0> {
  static constexpr int CB = 8, SUBB = 2, CHUNK = 704, STAGES = 11;
  static constexpr int UNIT = (CB / SUBB) * 4 * CHUNK;  // 11264
  static constexpr bool kF16 = true;
};
// Borrowed row-major BF16 LM head: a unit is 64 rows x 128 inputs staged by
// two 64x64 TMA boxes with the 128-byte swizzle.
template <>
struct Fmt<WT_HEAD> {
  static constexpr int CB = 4, SUBB = 1, CHUNK = 0, STAGES = 8;
  static constexpr int UNIT = 64 * 128 * 2;  // 16384
  static constexpr bool kF16 = false;
};

inline size_t packed_bytes(int wtype, int n, int k) {
  switch (wtype) {
    case WT_BF16: return size_t(n / 64) * (k / (32 * Fmt<WT_BF16>::CB)) * Fmt<WT_BF16>::UNIT;
    case WT_Q8_0: return size_t(n / 64) * (k / (32 * Fmt<WT_Q8_0>::CB)) * Fmt<WT_Q8_0>::UNIT;
    case WT_Q4_0: return size_t(n / 64) * (k / (32 * Fmt<WT_Q4_0>::CB)) * Fmt<WT_Q4_0>::UNIT;
    case WT_Q5_0: return size_t(n / 64) * (k / (32 * Fmt<WT_Q5_0>::CB)) * Fmt<WT_Q5_0>::UNIT;
  }
  return 0;
}

// Streamed activations ("chunked" layout).  A GEMV that streams X copies,
// with each weight unit, the unit's KU input columns of all R activation rows
// as one contiguous chunk per plane.  Element (row r, column k, plane p):
//   ((j * planes + p) * R + r) * (KU + 32) + (k - j * KU),   j = k / KU
// in 16-bit elements; rows are padded by 32 elements so that the consumer's
// 16-byte lane loads of neighbouring rows fall in different banks.  BF16
// activations have two planes (hi, lo = x - hi), FP16 ones a single plane.
__host__ __device__ __forceinline__ size_t xchunk_index(int k, int r, int p, int R, int KU, int planes) {
  const int j = k / KU;
  return ((static_cast<size_t>(j) * planes + p) * R + r) * (KU + 32) + (k - j * KU);
}
inline size_t xchunk_elems(int K, int R, int KU, int planes) {
  return static_cast<size_t>(K / KU) * planes * R * (KU + 32);
}

// Row of the 64-row group that mma row m (0..15) of m-tile w computes.  The
// fragment-native formats are in natural order; the swizzled LM-head boxes
// use an interleaved order that keeps the 16-byte lane loads free of bank
// conflicts (rows read by neighbouring lanes differ in bit 2 of their swizzle
// phase).
template <int WT>
__device__ __forceinline__ int frag_row(int w, int m) {
  if constexpr (WT == WT_HEAD) {
    const int lo = m & 7;
    const int sig = ((lo & 1) << 2) | (lo >> 1);
    return w * 16 + (m & 8) + sig;
  } else {
    return w * 16 + m;
  }
}

// ---------------------------------------------------------------- decoders
// Every quantised code is a small integer, exact in FP16 and in BF16.  The
// decoders produce pairs in the activation type the MMA is fed with: FP16
// (layer GEMVs of quantised models) or BF16 (the fusion projection, whose
// inputs are the target's BF16 taps).
//
// 4 signed 8-bit codes (biased +128) -> pairs (e0,e1) and (e2,e3), exact.
template <bool F16>
__device__ __forceinline__ uint32_t q8_pair(uint32_t word, uint32_t sel) {
  const uint32_t h = hsub2_u32(prmt(word, 0x64646464u, sel), 0x64806480u);
  if constexpr (F16) {
    return h;
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    return pack_bf16x2(f.x, f.y);
  }
}
// The four nibble pairs of a Q4 word -> FP16 (e - 8) pairs, exact: pairs 0
// and 2 as 0x6400 | n = 1024 + n minus 1032; pairs 1 and 3 taken in place
// (bits 4..7 / 20..23) as 0x6400 | 16 n = 1024 + 16 n, times 1/16 minus 72
// in one fused multiply-add (every intermediate is an exact FP16 integer).
__device__ __forceinline__ void q4_word_f16(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  const uint32_t w8 = w >> 8;
  p0 = hsub2_u32((w & 0x000F000Fu) | 0x64006400u, 0x64086408u);
  p1 = hfma2_u32((w & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD480D480u);
  p2 = hsub2_u32((w8 & 0x000F000Fu) | 0x64006400u, 0x64086408u);
  p3 = hfma2_u32((w8 & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD480D480u);
}

// Nibble pair j of a Q4 word -> (e2j - 8, e2j+1 - 8), exact.  0x6400 | n is
// the FP16 1024 + n; 0x4300 | n is the BF16 128 + n (n < 128).
template <bool F16>
__device__ __forceinline__ uint32_t q4_pair(uint32_t word, int j) {
  const uint32_t n = (word >> (4 * j)) & 0x000F000Fu;
  if constexpr (F16) return hsub2_u32(n | 0x64006400u, 0x64086408u);
  else return hsub2_bf16_u32(n | 0x43004300u, 0x43084308u);
}
// Nibble pair j of a Q5 word plus its fifth bits -> (q - 16), exact.
template <bool F16>
__device__ __forceinline__ uint32_t q5_pair(uint32_t word, uint32_t hb, int j, int off) {
  const uint32_t n = ((word >> (4 * j)) & 0x000F000Fu) | (((hb >> (j + off)) & 0x00010001u) << 4);
  if constexpr (F16) return hsub2_u32(n | 0x64006400u, 0x64106410u);
  else return hsub2_bf16_u32(n | 0x43004300u, 0x43104310u);
}

// A fragments of one 32-block for both k-steps, plus the per-row scales
// (1.0 for BF16).  a[s][0..3] are the four A registers of k-step s.
struct BlockFrag {
  uint32_t a[2][4];
  float d_r, d_r8;
};

// Decode 32-block `bl` (0..CB-1) of the unit at shared address `ubase` for
// m-tile w.  Lane layout per the header comment.
template <int WT, bool F16 = Fmt<WT>::kF16>
__device__ __forceinline__ BlockFrag decode_block(uint32_t ubase, int w, int lane, int bl) {
  BlockFrag f;
  if constexpr (WT == WT_BF16) {
    const uint32_t base = ubase + (bl * 4 + w) * Fmt<WT_BF16>::CHUNK;
    const uint4 wa = lds128(base + lane * 16);
    const uint4 wb = lds128(base + 512 + lane * 16);
    f.a[0][0] = wa.x; f.a[0][1] = wb.x; f.a[0][2] = wa.y; f.a[0][3] = wb.y;
    f.a[1][0] = wa.z; f.a[1][1] = wb.z; f.a[1][2] = wa.w; f.a[1][3] = wb.w;
    f.d_r = f.d_r8 = 1.f;
  } else if constexpr (WT == WT_HEAD) {
    // two 64x64 boxes of 128-byte rows; chunk q of row R sits at q ^ (R & 7)
    const uint32_t box = ubase + (bl >> 1) * 8192;
    const int r = lane >> 2, c = lane & 3;
    const int q = (bl & 1) * 4 + c;
    const int ra = frag_row<WT_HEAD>(w, r);
    const int rb = frag_row<WT_HEAD>(w, r + 8);
    const uint4 wa = lds128(box + ra * 128 + ((q ^ (ra & 7)) << 4));
    const uint4 wb = lds128(box + rb * 128 + ((q ^ (rb & 7)) << 4));
    f.a[0][0] = wa.x; f.a[0][1] = wb.x; f.a[0][2] = wa.y; f.a[0][3] = wb.y;
    f.a[1][0] = wa.z; f.a[1][1] = wb.z; f.a[1][2] = wa.w; f.a[1][3] = wb.w;
    f.d_r = f.d_r8 = 1.f;
  } else if constexpr (WT == WT_Q8_0) {
    const uint32_t base = ubase + (bl * 4 + w) * Fmt<WT_Q8_0>::CHUNK;
    const uint4 q = lds128(base + lane * 16);
    const uint32_t sc = lds32(base + 512 + (lane >> 2) * 4);
    f.a[0][0] = q8_pair<F16>(q.x, 0x4140); f.a[0][1] = q8_pair<F16>(q.z, 0x4140);
    f.a[0][2] = q8_pair<F16>(q.x, 0x4342); f.a[0][3] = q8_pair<F16>(q.z, 0x4342);
    f.a[1][0] = q8_pair<F16>(q.y, 0x4140); f.a[1][1] = q8_pair<F16>(q.w, 0x4140);
    f.a[1][2] = q8_pair<F16>(q.y, 0x4342); f.a[1][3] = q8_pair<F16>(q.w, 0x4342);
    const __half2 d = *reinterpret_cast<const __half2*>(&sc);
    f.d_r = __low2float(d);
    f.d_r8 = __high2float(d);
  } else {  // Q4_0 / Q5_0: two blocks per sub-chunk
    constexpr int CHUNK = Fmt<WT>::CHUNK;
    const int pair = bl >> 1, b = bl & 1;
    const uint32_t base = ubase + (pair * 4 + w) * CHUNK;
    const uint4 q = lds128(base + lane * 16);
    const uint32_t wr = b ? q.y : q.x;
    const uint32_t wr8 = b ? q.w : q.z;
    constexpr int SC_OFF = (WT == WT_Q4_0) ? 512 : 640;
    const uint2 sc = lds64(base + SC_OFF + (lane >> 2) * 8);
    const uint32_t scb = b ? sc.y : sc.x;
    const __half2 d = *reinterpret_cast<const __half2*>(&scb);
    f.d_r = __low2float(d);
    f.d_r8 = __high2float(d);
    if constexpr (WT == WT_Q4_0 && F16) {
      q4_word_f16(wr, f.a[0][0], f.a[0][2], f.a[1][0], f.a[1][2]);
      q4_word_f16(wr8, f.a[0][1], f.a[0][3], f.a[1][1], f.a[1][3]);
    } else if constexpr (WT == WT_Q4_0) {
      f.a[0][0] = q4_pair<F16>(wr, 0); f.a[0][1] = q4_pair<F16>(wr8, 0);
      f.a[0][2] = q4_pair<F16>(wr, 1); f.a[0][3] = q4_pair<F16>(wr8, 1);
      f.a[1][0] = q4_pair<F16>(wr, 2); f.a[1][1] = q4_pair<F16>(wr8, 2);
      f.a[1][2] = q4_pair<F16>(wr, 3); f.a[1][3] = q4_pair<F16>(wr8, 3);
    } else {
      const uint32_t hb = lds32(base + 512 + lane * 4);
      const int o_r = b * 4, o_r8 = 8 + b * 4;
      f.a[0][0] = q5_pair<F16>(wr, hb, 0, o_r); f.a[0][1] = q5_pair<F16>(wr8, hb, 0, o_r8);
      f.a[0][2] = q5_pair<F16>(wr, hb, 1, o_r); f.a[0][3] = q5_pair<F16>(wr8, hb, 1, o_r8);
      f.a[1][0] = q5_pair<F16>(wr, hb, 2, o_r); f.a[1][1] = q5_pair<F16>(wr8, hb, 2, o_r8);
      f.a[1][2] = q5_pair<F16>(wr, hb, 3, o_r); f.a[1][3] = q5_pair<F16>(wr8, hb, 3, o_r8);
    }
  }
  return f;
}

// Both 32-blocks of sub-chunk `pair` of a Q4_0 / Q5_0 unit (blocks 2 pair and
// 2 pair + 1), with one load of the shared codes and scales.
template <int WT, bool F16 = Fmt<WT>::kF16>
__device__ __forceinline__ void decode_pair(uint32_t ubase, int w, int lane, int pair, BlockFrag& f0,
                                            BlockFrag& f1) {
  static_assert(WT == WT_Q4_0 || WT == WT_Q5_0, "two blocks per sub-chunk");
  constexpr int CHUNK = Fmt<WT>::CHUNK;
  const uint32_t base = ubase + (pair * 4 + w) * CHUNK;
  const uint4 q = lds128(base + lane * 16);
  constexpr int SC_OFF = (WT == WT_Q4_0) ? 512 : 640;
  const uint2 sc = lds64(base + SC_OFF + (lane >> 2) * 8);
  uint32_t hb = 0;
  if constexpr (WT == WT_Q5_0) hb = lds32(base + 512 + lane * 4);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    BlockFrag& f = b ? f1 : f0;
    const uint32_t wr = b ? q.y : q.x;
    const uint32_t wr8 = b ? q.w : q.z;
    const uint32_t scb = b ? sc.y : sc.x;
    const __half2 d = *reinterpret_cast<const __half2*>(&scb);
    f.d_r = __low2float(d);
    f.d_r8 = __high2float(d);
    if constexpr (WT == WT_Q4_0 && F16) {
      q4_word_f16(wr, f.a[0][0], f.a[0][2], f.a[1][0], f.a[1][2]);
      q4_word_f16(wr8, f.a[0][1], f.a[0][3], f.a[1][1], f.a[1][3]);
    } else if constexpr (WT == WT_Q4_0) {
      f.a[0][0] = q4_pair<F16>(wr, 0); f.a[0][1] = q4_pair<F16>(wr8, 0);
      f.a[0][2] = q4_pair<F16>(wr, 1); f.a[0][3] = q4_pair<F16>(wr8, 1);
      f.a[1][0] = q4_pair<F16>(wr, 2); f.a[1][1] = q4_pair<F16>(wr8, 2);
      f.a[1][2] = q4_pair<F16>(wr, 3); f.a[1][3] = q4_pair<F16>(wr8, 3);
    } else {
      const int o_r = b * 4, o_r8 = 8 + b * 4;
      f.a[0][0] = q5_pair<F16>(wr, hb, 0, o_r); f.a[0][1] = q5_pair<F16>(wr8, hb, 0, o_r8);
      f.a[0][2] = q5_pair<F16>(wr, hb, 1, o_r); f.a[0][3] = q5_pair<F16>(wr8, hb, 1, o_r8);
      f.a[1][0] = q5_pair<F16>(wr, hb, 2, o_r); f.a[1][1] = q5_pair<F16>(wr8, hb, 2, o_r8);
      f.a[1][2] = q5_pair<F16>(wr, hb, 3, o_r); f.a[1][3] = q5_pair<F16>(wr8, hb, 3, o_r8);
    }
  }
}

}  // namespace dflash
