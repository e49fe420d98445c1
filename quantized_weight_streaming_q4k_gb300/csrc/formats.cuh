// formats.cuh -- per-lane decoders for the three GGUF block formats.
//
// Block layouts (infer-compute README, §Design Principles "GGUF-compatible" and
// §Shaders Q4_0 / Q4_K / Q6_K rows; the public GGUF layouts):
//   Q4_K 144 B / 256 w : f16 d, f16 dmin, 12 B packed 6-bit scales+mins, 128 B nibbles
//                        w = d*sc[s]*q - dmin*m[s]     (eight 32-weight sub-blocks)
//   Q6_K 210 B / 256 w : 128 B low nibbles, 64 B 2-bit highs, 16 int8 scales, f16 d
//                        w = d*sc[i/16]*(q-32)
//   Q4_0  18 B /  32 w : f16 d, 16 B nibbles;  w = d*(q-8)
//   Q8_0  34 B /  32 w : f16 d, 32 int8 codes;  w = d*q   (8-bit path)
//
// Lane unit.  Every lane owns a fixed group of 64 (Q6_K: 32) columns of the
// row ("unit") and keeps the matching activations in registers for the whole
// phase (x-stationary).  The weight bytes of one row stream through shared memory;
// for each row the lane decodes its unit and returns a partial dot product.
//
// Decode without int->float conversion.  A 4- or 6-bit field masked in place
// inside a 32-bit word, with every other bit zero, is a valid subnormal
// float: q * 2^(pos - 149) where pos is the field's bit position (pos <= 16,
// so the field stays below the exponent bits).  The activation for that weight
// is stored pre-scaled as x * 2^(kE - pos), so the FMA product is exactly
// q * x * 2^(kE - 149) = q * x * 2^-60, accumulated in f32.  One LOP per weight
// replaces shift + convert; the 2^60 and the sub-block scales are applied once
// per sub-block.  Fields whose bit position would reach the exponent are
// shifted down by 8 or 12 first.  Pre-scaling by a power of two is exact for
// |x| in [2^-66, 2^38]; outside that range products lose bits or overflow.
#pragma once

#include <cstdint>

#include "device_common.cuh"

namespace qws {

constexpr int kE = 89;                 // x' = x * 2^(kE - pos)

// columns per lane unit of each format
__host__ __device__ constexpr int unit_weights(int) { return 64; }

__device__ __forceinline__ float bits(uint32_t v) { return __uint_as_float(v); }

// ---------------------------------------------------------------------------
// Nibble positions inside one 32-bit word of four bytes (b = byte 0..3).
// Low nibble of byte b:  b=0 bits 0-3, b=1 bits 8-11, b=2 bits 16-19 (direct);
//                        b=3 bits 24-27 -> (w >> 12) bits 12-15.
// High nibble of byte b: b=0 bits 4-7, b=1 bits 12-15 (direct);
//                        b=2 bits 20-23 -> (w >> 12) bits 8-11;
//                        b=3 bits 28-31 -> (w >> 12) bits 16-19.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int pos_lo(int b) { return b == 0 ? 0 : b == 1 ? 8 : b == 2 ? 16 : 12; }
__host__ __device__ constexpr int pos_hi(int b) { return b == 0 ? 4 : b == 1 ? 12 : b == 2 ? 8 : 16; }

// lo[0..3] += low nibbles of bytes 0..3 times xl[0..3]; same for the high
// nibbles with xh.  Two accumulator pairs per nibble class (packed FMA).
__device__ __forceinline__ void nibble_word(uint32_t w, const float* xl, const float* xh,
                                            float& l0, float& l1, float& h0, float& h1) {
  const uint32_t s = w >> 12;
  fma2(l0, l1, bits(w & 0xFu), bits(w & 0xF00u), xl[0], xl[1]);
  fma2(l0, l1, bits(w & 0xF0000u), bits(s & 0xF000u), xl[2], xl[3]);
  fma2(h0, h1, bits(w & 0xF0u), bits(w & 0xF000u), xh[0], xh[1]);
  fma2(h0, h1, bits(s & 0xF00u), bits(s & 0xF0000u), xh[2], xh[3]);
}

// ---------------------------------------------------------------------------
// Byte split: both nibbles of a byte from one mask and two FP operations.
// A byte b = lo + 16 hi masked in place at bit p (p <= 16; the top byte is
// shifted down to p = 0 first) is the float B = b * 2^(p-149).  Multiplying
// by 2^(-p-4) with round-toward-zero lands on the subnormal grid 2^-149 and
// drops the low nibble: H = hi * 2^-149 exactly; then L = B - 16 * 2^p * H =
// lo * 2^(p-149) exactly (an FMA whose result is representable).  So H takes
// activations pre-scaled by 2^kE and L by 2^(kE - p), and both products are
// q * x * 2^-60 as for the in-place masks.  One integer operation per two
// weights instead of two: the work moves to the FMA pipe, which the in-place
// decode leaves mostly idle.  (mul.rz / fma on f32 keep subnormals: no .ftz.)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mul2_rz(float& d0, float& d1, float a0, float a1, float b0,
                                        float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rz.f32x2 rc, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Bit position of byte b (0..3) of a word in the byte split: bytes 0..2 in
// place, byte 3 shifted down to 0.
__host__ __device__ constexpr int split_pos(int b) { return b == 3 ? 0 : 8 * b; }

// lo[0..3] += low nibbles of bytes 0..3 times xl[0..3], hi likewise with xh;
// xl[b] pre-scaled by 2^(kE - split_pos(b)), xh by 2^kE.
__device__ __forceinline__ void nibble_word_split(uint32_t w, const float* xl, const float* xh,
                                                  float& l0, float& l1, float& h0, float& h1) {
  const float B0 = bits(w & 0xFFu), B3 = bits(w >> 24);          // p = 0, 0
  const float B1 = bits(w & 0xFF00u), B2 = bits(w & 0xFF0000u);  // p = 8, 16
  float H0, H3, H1, H2;
  mul2_rz(H0, H3, B0, B3, exp2i(-4), exp2i(-4));
  mul2_rz(H1, H2, B1, B2, exp2i(-12), exp2i(-20));
  float L0 = B0, L3 = B3, L1 = B1, L2 = B2;
  fma2(L0, L3, H0, H3, -16.f, -16.f);
  fma2(L1, L2, H1, H2, -4096.f, -1048576.f);
  fma2(l0, l1, L0, L3, xl[0], xl[3]);
  fma2(l0, l1, L1, L2, xl[1], xl[2]);
  fma2(h0, h1, H0, H3, xh[0], xh[3]);
  fma2(h0, h1, H1, H2, xh[1], xh[2]);
}

// The same byte split with scalar operations (immediate operands, no
// register pairs to build): for the Q4_K chunk, where the measured mix of
// scalar and packed FP instructions decodes faster than the packed split
// (the Q4_0 and Q6_K decoders keep the packed form, faster there).
__device__ __forceinline__ void nibble_word_split_scalar(uint32_t w, const float* xl,
                                                         const float* xh, float& l0, float& l1,
                                                         float& h0, float& h1) {
  const float B0 = bits(w & 0xFFu), B3 = bits(w >> 24);          // p = 0, 0
  const float B1 = bits(w & 0xFF00u), B2 = bits(w & 0xFF0000u);  // p = 8, 16
  const float H0 = __fmul_rz(B0, exp2i(-4)), H3 = __fmul_rz(B3, exp2i(-4));
  const float H1 = __fmul_rz(B1, exp2i(-12)), H2 = __fmul_rz(B2, exp2i(-20));
  const float L0 = fmaf(H0, -16.f, B0), L3 = fmaf(H3, -16.f, B3);
  const float L1 = fmaf(H1, -4096.f, B1), L2 = fmaf(H2, -1048576.f, B2);
  fma2(l0, l1, L0, L3, xl[0], xl[3]);
  fma2(l0, l1, L1, L2, xl[1], xl[2]);
  fma2(h0, h1, H0, H3, xh[0], xh[3]);
  fma2(h0, h1, H1, H2, xh[1], xh[2]);
}

// Which of the eight words of a 32-byte Q4_K chunk take the byte split (bit
// k set: word k), the rest the in-place masks.  Measured with the scalar
// split (same box, two passes): none 84.3 us for the 262144 x 2560 matvec
// and 1032 us for the 34-layer chain, 0x11 84.1 / 1035, 0x33 84.8 / 1042,
// 0x55 86.0 / 1039, 0x77 85.7 / 1044, all 85.3 / 1043: the in-place masks
// take the fewest instructions (1.6 per weight against 2.0), and the chain
// is bound by instruction issue.
constexpr unsigned kQ4kSplitWords = 0x00u;

__host__ __device__ constexpr bool q4k_word_split(int k) { return (kQ4kSplitWords >> k) & 1u; }

// Words 2i and 2i + 1 of a chunk decoded as a pair (kPair; both in place):
// one byte permute brings the top bytes of both down to bytes 0 and 1 of a
// third word, and every nibble is then masked in place (one instruction per
// word pair fewer than a shift per word).  Measured on the 262144 x 2560
// Q4_K matvec (same box, two passes): 81.0 -> 79.45 us, the fused FFN 23.75
// -> 23.58 us; the 34-layer chain (its own register budget) 982 -> 994 us,
// so the chain keeps one shift per word.  Positions: bytes 0..2 of
// each word at bits 8b (low nibble) and 8b + 4 (high; bits 20-23 too: with
// q >= 8 the top bit lands on the exponent's lowest bit and the value is
// still q * 2^(20-149)); byte 3 of the even word at bits 0 / 4 of the
// permuted word, of the odd word at bits 8 / 12.
template <bool kPair>
__host__ __device__ constexpr bool q4k_pair_inplace(int k) {
  return kPair && !q4k_word_split(k & ~1) && !q4k_word_split(k | 1);
}
__host__ __device__ constexpr int pair_pos_lo(int k, int b) { return b < 3 ? 8 * b : 8 * (k & 1); }
__host__ __device__ constexpr int pair_pos_hi(int k, int b) {
  return b < 3 ? 8 * b + 4 : 8 * (k & 1) + 4;
}

// Pre-scale exponents of the activations of chunk byte l (0..31): xa for the
// low nibble (sub-block 2c), xb for the high nibble (sub-block 2c+1).
template <bool kPair>
__host__ __device__ constexpr int q4k_xa_exp(int l) {
  return q4k_word_split(l >> 2)             ? kE - split_pos(l & 3)
         : q4k_pair_inplace<kPair>(l >> 2) ? kE - pair_pos_lo(l >> 2, l & 3)
                                            : kE - pos_lo(l & 3);
}
template <bool kPair>
__host__ __device__ constexpr int q4k_xb_exp(int l) {
  return q4k_word_split(l >> 2)             ? kE
         : q4k_pair_inplace<kPair>(l >> 2) ? kE - pair_pos_hi(l >> 2, l & 3)
                                            : kE - pos_hi(l & 3);
}

// Exponents of the activation pre-scale for byte b of a full nibble word,
// decoded in place (kSplit false) or by the byte split.
template <bool kSplit>
__host__ __device__ constexpr int lo_exp(int b) {
  return kSplit ? kE - split_pos(b) : kE - pos_lo(b);
}
template <bool kSplit>
__host__ __device__ constexpr int hi_exp(int b) {
  return kSplit ? kE : kE - pos_hi(b);
}

template <bool kSplit>
__device__ __forceinline__ void nib_word(uint32_t w, const float* xl, const float* xh, float& l0,
                                         float& l1, float& h0, float& h1) {
  if constexpr (kSplit)
    nibble_word_split(w, xl, xh, l0, l1, h0, h1);
  else
    nibble_word(w, xl, xh, l0, l1, h0, h1);
}

template <int k>
__device__ __forceinline__ void q4k_word(uint32_t w, const float* xa, const float* xb, float& a0,
                                         float& a1, float& b0, float& b1) {
  if constexpr (q4k_word_split(k))
    nibble_word_split_scalar(w, xa + 4 * k, xb + 4 * k, a0, a1, b0, b1);
  else
    nibble_word(w, xa + 4 * k, xb + 4 * k, a0, a1, b0, b1);
}

// Words k (even) and k + 1 of the chunk (positions: pair_pos_lo / _hi when
// kPair, else one word at a time).
template <bool kPair, int k>
__device__ __forceinline__ void q4k_word_pair(uint32_t w0, uint32_t w1, const float* xa,
                                              const float* xb, float& a0, float& a1, float& b0,
                                              float& b1) {
  static_assert((k & 1) == 0, "pairs start on an even word");
  if constexpr (!q4k_pair_inplace<kPair>(k)) {
    q4k_word<k>(w0, xa, xb, a0, a1, b0, b1);
    q4k_word<k + 1>(w1, xa, xb, a0, a1, b0, b1);
  } else {
    const uint32_t t = __byte_perm(w0, w1, 0x0073u);   // [w0 byte 3, w1 byte 3, ...]
    const float* la = xa + 4 * k;
    const float* ha = xb + 4 * k;
    fma2(a0, a1, bits(w0 & 0xFu), bits(w0 & 0xF00u), la[0], la[1]);
    fma2(a0, a1, bits(w0 & 0xF0000u), bits(t & 0xFu), la[2], la[3]);
    fma2(b0, b1, bits(w0 & 0xF0u), bits(w0 & 0xF000u), ha[0], ha[1]);
    fma2(b0, b1, bits(w0 & 0xF00000u), bits(t & 0xF0u), ha[2], ha[3]);
    fma2(a0, a1, bits(w1 & 0xFu), bits(w1 & 0xF00u), la[4], la[5]);
    fma2(a0, a1, bits(w1 & 0xF0000u), bits(t & 0xF00u), la[6], la[7]);
    fma2(b0, b1, bits(w1 & 0xF0u), bits(w1 & 0xF000u), ha[4], ha[5]);
    fma2(b0, b1, bits(w1 & 0xF00000u), bits(t & 0xF000u), ha[6], ha[7]);
  }
}

// ---------------------------------------------------------------------------
// Q4_K.  Unit u -> super-block kb = u/4, chunk c = u%4: the 32 qs bytes
// qs[32c .. 32c+31] (weights 64c+l of sub-block 2c in the low nibbles and
// 64c+32+l of sub-block 2c+1 in the high nibbles) plus the block header.
// ---------------------------------------------------------------------------
// Scale / min selection of one Q4_K chunk, fixed per lane unit (chunk c of
// the block: sub-blocks 2c and 2c + 1).  With j = 2 (c & 1):
//   P = bytes [y_j, y_j+1, z_j, z_j+1] of the header words hd.y (scale bytes
//       0..3) and hd.z (4..7); Q = [w_j, w_j+1, w_j, w_j+1] of hd.w (8..11)
//       for c >= 2, zero for c < 2;
//   R = ((P >> sh) & mask) | (Q's low nibbles in bytes 0, 1 and high nibbles
//       in bytes 2, 3) = [scale_a, scale_b, min_a, min_b]:
//   c < 2 : sh = 0, mask 0x3F3F3F3F (the 6-bit fields themselves);
//   c >= 2: sh = 2, mask 0x30303030 (bits 6, 7 of y / z as bits 4, 5 on top
//           of w's nibble) -- the GGUF packing of sub-blocks 4..7.
struct Q4kSel {
  uint32_t selP, selQ, sh, mask;
  __device__ __forceinline__ void set(int c) {
    const uint32_t j = 2u * static_cast<uint32_t>(c & 1);
    selP = j | (j + 1) << 4 | (4 + j) << 8 | (5 + j) << 12;
    selQ = c >= 2 ? (j | (j + 1) << 4 | j << 8 | (j + 1) << 12) : 0x4444u;
    sh = c >= 2 ? 2u : 0u;
    mask = c >= 2 ? 0x30303030u : 0x3F3F3F3Fu;
  }
};

__device__ __forceinline__ uint32_t q4k_scale_bytes(const uint4 hd, uint32_t selP, uint32_t selQ,
                                                    uint32_t sh, uint32_t mask) {
  const uint32_t P = __byte_perm(hd.y, hd.z, selP);
  const uint32_t Q = __byte_perm(hd.w, 0u, selQ);
  const uint32_t N = ((Q & 0x0000FFFFu) | ((Q >> 4) & 0xFFFF0000u)) & 0x0F0F0F0Fu;
  return ((P >> sh) & mask) | N;
}

// byte k of r as an exact float: under the exponent of 2^23, minus 2^23
__device__ __forceinline__ float byte_to_float(uint32_t r, uint32_t k) {
  return __uint_as_float(__byte_perm(r, 0x4B000000u, 0x7650u | k)) - 8388608.0f;
}

// Dot product of one Q4_K chunk (32 bytes: 32 low nibbles of sub-block 2c,
// 32 high nibbles of sub-block 2c+1) with the pre-scaled activations xa / xb
// (q4k_xa_exp / q4k_xb_exp of the same kPair); hd is the block header, the
// selection constants come from Q4kSel::set(c).
template <bool kPair>
__device__ __forceinline__ float q4k_chunk_dot(const uint4 hd, const uint4 q0, const uint4 q1,
                                               const float* xa, const float* xb, float sxa,
                                               float sxb, uint32_t selP, uint32_t selQ,
                                               uint32_t sh, uint32_t mask) {
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
  q4k_word_pair<kPair, 0>(q0.x, q0.y, xa, xb, a0, a1, b0, b1);
  q4k_word_pair<kPair, 2>(q0.z, q0.w, xa, xb, a0, a1, b0, b1);
  q4k_word_pair<kPair, 4>(q1.x, q1.y, xa, xb, a0, a1, b0, b1);
  q4k_word_pair<kPair, 6>(q1.z, q1.w, xa, xb, a0, a1, b0, b1);
  const uint32_t R = q4k_scale_bytes(hd, selP, selQ, sh, mask);
  const float sca = byte_to_float(R, 0), scb = byte_to_float(R, 1);
  const float mna = byte_to_float(R, 2), mnb = byte_to_float(R, 3);
  const float d = half_bits_to_float(hd.x) * exp2i(60);
  const float dmin = half_bits_to_float(hd.x >> 16);
  const float qx = fmaf(sca, a0 + a1, scb * (b0 + b1));
  const float mx = fmaf(mna, sxa, mnb * sxb);
  return fmaf(d, qx, -dmin * mx);
}

struct UnitQ4K {
  static constexpr int kFmt = 12;
  static constexpr int kUnitW = 64;
  static constexpr bool kMixed = false;
  static constexpr bool kDirect = false;  // activations staged through shared memory
  static constexpr int kBlockW = 256;
  static constexpr int kBlockBytes = 144;
  float xa[32];   // sub-block 2c,   column 64c + l,      pre-scaled
  float xb[32];   // sub-block 2c+1, column 64c + 32 + l, pre-scaled
  float sxa, sxb; // plain sums of x over the two sub-blocks
  uint32_t off;   // byte offset of the block header within the row
  uint32_t qoff;  // byte offset of the chunk within the block
  Q4kSel sel;     // scale / min selection of the unit's chunk

  // Unit u covers columns 64u .. 64u + 63; unit-local index l = col % 64.
  __device__ __forceinline__ static void unit_of(int64_t col, int& u, int& l) {
    u = static_cast<int>(col >> 6);
    l = static_cast<int>(col & 63);
  }

  // xu(l): activation of unit-local column l (0..63).
  template <class XU>
  __device__ __forceinline__ void setup(int u, const XU& xu) {
    const int kb = u >> 2, c = u & 3;
    off = static_cast<uint32_t>(kb) * kBlockBytes;
    qoff = 16u + 32u * c;
    sel.set(c);
    float sa = 0.f, sb = 0.f;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
      const float va = xu(l), vb = xu(32 + l);
      sa += va;
      sb += vb;
      xa[l] = va * exp2i(q4k_xa_exp<true>(l));
      xb[l] = vb * exp2i(q4k_xb_exp<true>(l));
    }
    sxa = sa;
    sxb = sb;
  }

  // Bytes of one row this unit reads: the block header and its 32-byte chunk.
  struct Frag {
    uint4 hd, q0, q1;
  };

  __device__ __forceinline__ void load(const uint8_t* rp, Frag& f) const {
    const uint8_t* bp = rp + off;
    f.hd = *reinterpret_cast<const uint4*>(bp);
    f.q0 = *reinterpret_cast<const uint4*>(bp + qoff);
    f.q1 = *reinterpret_cast<const uint4*>(bp + qoff + 16);
  }

  // Partial dot product of this unit with one row (its bytes in f).
  __device__ __forceinline__ float compute(const Frag& f) const {
    return q4k_chunk_dot<true>(f.hd, f.q0, f.q1, xa, xb, sxa, sxb, sel.selP, sel.selQ, sel.sh,
                               sel.mask);
  }

  __device__ __forceinline__ float row(const uint8_t* rp) const {
    Frag f;
    load(rp, f);
    return compute(f);
  }
};

// ---------------------------------------------------------------------------
// Q6_K.  Unit u -> super-block kb = u/4, half h = (u/2)%2, column group
// m = u%2: weights 128h + 32a + 16m + i for a = 0..3, i = 0..15 (64 weights).
// Bytes: ql[64h+16m ..+16] (a=0 low nibbles, a=2 high), ql[64h+32+16m ..+16]
// (a=1, a=3), qh[32h+16m ..+16] (2-bit fields a=0..3 at bits 0,2,4,6); the
// scale of column group a is sc[(128h + 32a + 16m) / 16] = sc[8h + 2a + m]:
// the unit's four scales share one 8-byte window, and one d serves all 64.
// Blocks are 210 B, so a block starts on a 2-byte boundary: the lane loads
// aligned words and funnel-shifts them.  The aligned pointer is p minus its
// misalignment (pointer arithmetic, not an integer round trip), so that a
// pointer into shared memory stays one the compiler can load with LDS.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t misalign4(const uint8_t* p) {
  return static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p)) & 3u;
}

// One Q6_K block's runs share the block's misalignment (every run offset
// is a multiple of 4 bytes): the row's aligned base and funnel shift are
// formed once, and each run loads aligned words at a word offset from it.
struct Q6kRow {
  const uint32_t* base;   // block start rounded down to 4 bytes
  uint32_t s;             // 8 * (block start & 3)
  __device__ __forceinline__ explicit Q6kRow(const uint8_t* bp) {
    const uint32_t m = misalign4(bp);
    base = reinterpret_cast<const uint32_t*>(bp - m);
    s = m * 8u;
  }
  // 16 bytes at byte offset o (a multiple of 4) of the block
  __device__ __forceinline__ void run16(uint32_t o, uint32_t (&w)[4]) const {
    const uint32_t* q = base + (o >> 2);
    uint32_t r[5];
#pragma unroll
    for (int k = 0; k < 5; ++k) r[k] = q[k];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = __funnelshift_r(r[k], r[k + 1], s);
  }
  __device__ __forceinline__ void run8(uint32_t o, uint32_t& w0, uint32_t& w1) const {
    const uint32_t* q = base + (o >> 2);
    const uint32_t r0 = q[0], r1 = q[1], r2 = q[2];
    w0 = __funnelshift_r(r0, r1, s);
    w1 = __funnelshift_r(r1, r2, s);
  }
  // the f16 d at byte 208
  __device__ __forceinline__ uint32_t dbits() const { return base[52] >> s; }
};

// Register slot of column j (0..3) of the 4-column group gi = 4a + t inside
// the unit's 64-float activation array (slot 16a + 4t + q6k_slot(gi, j)).
// The packed FMAs take columns (0, 2) and (1, 3) of a group as register
// pairs.  In the plain order (kQ4Pairs false) slot = j.  A decoder that also
// runs Q4_K on the same array (UnitChain) stores the columns so that these
// pairs fall on the slots the Q4_K decode pairs: slots (0, 3) / (1, 2) for
// the groups of byte-split words, (0, 1) / (2, 3) for the in-place ones.  One
// pairing for both formats lets the compiler keep every activation pair in
// place instead of copying registers into pairs for one of them.
// Q6_K fields: the 16-bit-pair split (true) or masks in place (false).
// Same instruction count per word (7); measured 120.7 against 125.4 us for
// the 262144 x 2560 matvec (same box, two passes), the chain unchanged.
constexpr bool kQ6kSplit = true;
// bit position of byte b's field for the in-place masks
__host__ __device__ constexpr int q6k_pos(int b) { return b == 0 ? 0 : b == 1 ? 8 : 16; }
__host__ __device__ constexpr int q6k_x_exp(int b) { return kQ6kSplit ? kE : kE - q6k_pos(b); }

template <bool kQ4Pairs>
__host__ __device__ constexpr int q6k_slot(int gi, int j) {
  return !kQ4Pairs ? j
         : q4k_word_split(gi & 7) ? (j == 2 ? 3 : j == 3 ? 2 : j)
                                  : (j == 1 ? 2 : j == 2 ? 1 : j);
}

// Dot product of one 64-column Q6_K unit (16 bytes of each of the two ql runs,
// 16 bytes of qh, the 8 scale bytes of the half) with activations pre-scaled
// by 2^kE, column 16a + 4t + j in slot 16a + 4t + q6k_slot(4a + t, j);
// sx32[a] carries the -32 offset.
template <bool kQ4Pairs = false>
__device__ __forceinline__ float q6k_unit_dot(const uint32_t (&A)[4], const uint32_t (&B)[4],
                                              const uint32_t (&Q)[4], uint32_t S0, uint32_t S1,
                                              uint32_t dbits, const float* x, const float* sx32,
                                              uint32_t sshift) {
  const float d = half_bits_to_float(dbits) * exp2i(60);
  float p[4][2];
#pragma unroll
  for (int a = 0; a < 4; ++a) p[a][0] = p[a][1] = 0.f;
  constexpr uint32_t M = 0x0F0F0F0Fu;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t wa = A[t], wb = B[t], hh = Q[t];
    // 6-bit quants of four consecutive columns, one per byte (bits 6,7 of
    // each byte are don't-care; the extraction masks drop them)
    const uint32_t v0 = (wa & M) | ((hh << 4) & ~M);
    const uint32_t v1 = (wb & M) | ((hh << 2) & ~M);
    const uint32_t v2 = ((wa >> 4) & M) | (hh & ~M);
    const uint32_t v3 = ((wb >> 4) & M) | ((hh >> 2) & ~M);
    const uint32_t vv[4] = {v0, v1, v2, v3};
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const uint32_t v = vv[a];
      float L0, L1, H0, H1;   // the fields of bytes 0, 2 and 1, 3
      if constexpr (kQ6kSplit) {
        // two 6-bit fields per 16-bit half (bits 0-5 and 8-13 after the
        // mask), split like the nibbles of a byte: H = upper field, L = lower
        // field, both on the 2^-149 grid (activations pre-scaled by 2^kE)
        const float P0 = bits(v & 0x3F3Fu), P1 = bits((v >> 16) & 0x3F3Fu);
        mul2_rz(H0, H1, P0, P1, exp2i(-8), exp2i(-8));
        L0 = P0;
        L1 = P1;
        fma2(L0, L1, H0, H1, -256.f, -256.f);
      } else {
        // each field masked in place at bit q6k_pos(b) (byte 3 shifted down
        // to 16), activations pre-scaled by 2^(kE - q6k_pos(b))
        L0 = bits(v & 0x3Fu);
        H0 = bits(v & 0x3F00u);
        L1 = bits(v & 0x3F0000u);
        H1 = bits((v >> 8) & 0x3F0000u);
      }
      const float* xr = x + 16 * a + 4 * t;
      const int gi = 4 * a + t;
      fma2(p[a][0], p[a][1], L0, L1, xr[q6k_slot<kQ4Pairs>(gi, 0)],
           xr[q6k_slot<kQ4Pairs>(gi, 2)]);
      fma2(p[a][0], p[a][1], H0, H1, xr[q6k_slot<kQ4Pairs>(gi, 1)],
           xr[q6k_slot<kQ4Pairs>(gi, 3)]);
    }
  }
  // scale of group a: byte 2a + m of the 8 scale bytes of half h
  float acc = 0.f;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const uint32_t wsc = a < 2 ? S0 : S1;
    const uint32_t shift = 16u * (a & 1) + sshift;
    const int sc = static_cast<int>(static_cast<int8_t>((wsc >> shift) & 0xFFu));
    acc = fmaf(static_cast<float>(sc), (p[a][0] + p[a][1]) - sx32[a], acc);
  }
  return d * acc;
}

// Column 256kb + 128h + 32a + 16m + i belongs to Q6_K unit 4kb + 2h + m with
// unit-local index l = 16a + i.
__device__ __forceinline__ void q6k_unit_of(int64_t col, int& u, int& l) {
  const int kb = static_cast<int>(col >> 8), r = static_cast<int>(col & 255);
  const int h = r >> 7, a = (r >> 5) & 3, m = (r >> 4) & 1, i = r & 15;
  u = 4 * kb + 2 * h + m;
  l = 16 * a + i;
}

// Set-up shared by the Q6_K lane units: byte offsets of the unit's runs and
// the pre-scaled activations.
struct Q6kUnitGeom {
  uint32_t off, oA, oB, oQ, oS, sshift;
  __device__ __forceinline__ void set(int u) {
    const int kb = u >> 2, h = (u >> 1) & 1, m = u & 1;
    off = static_cast<uint32_t>(kb) * 210u;
    oA = 64u * h + 16u * m;
    oB = 64u * h + 32u + 16u * m;
    oQ = 128u + 32u * h + 16u * m;
    oS = 192u + 8u * h;            // the 8 scales of half h
    sshift = 8u * static_cast<uint32_t>(m);
  }
};

template <bool kQ4Pairs = false, class XU>
__device__ __forceinline__ void q6k_setup_x(const XU& xu, float* x, float* sx32) {
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float v = xu(16 * a + i);
      s += v;
      x[16 * a + (i & ~3) + q6k_slot<kQ4Pairs>(4 * a + (i >> 2), i & 3)] =
          v * exp2i(q6k_x_exp(i & 3));
    }
    sx32[a] = s * exp2i(5 - 60);
  }
}

struct UnitQ6K {
  static constexpr int kFmt = 14;
  static constexpr int kUnitW = 64;
  static constexpr bool kMixed = false;
  static constexpr bool kDirect = false;  // activations staged through shared memory
  static constexpr int kBlockW = 256;
  static constexpr int kBlockBytes = 210;
  float x[64];      // [16a + i], pre-scaled by 2^kE
  float sx32[4];    // 32 * sum_i x[a][i] * 2^-60 (the -32 offset, in product units)
  Q6kUnitGeom g;

  __device__ __forceinline__ static void unit_of(int64_t col, int& u, int& l) {
    q6k_unit_of(col, u, l);
  }

  template <class XU>
  __device__ __forceinline__ void setup(int u, const XU& xu) {
    g.set(u);
    q6k_setup_x(xu, x, sx32);
  }

  struct Frag {
    uint32_t A[4], B[4], Q[4], S0, S1;
    uint32_t dbits;
  };

  __device__ __forceinline__ void load(const uint8_t* rp, Frag& f) const {
    const Q6kRow br(rp + g.off);
    br.run16(g.oA, f.A);
    br.run16(g.oB, f.B);
    br.run16(g.oQ, f.Q);
    br.run8(g.oS, f.S0, f.S1);
    f.dbits = br.dbits();
  }

  __device__ __forceinline__ float compute(const Frag& f) const {
    return q6k_unit_dot(f.A, f.B, f.Q, f.S0, f.S1, f.dbits, x, sx32, g.sshift);
  }

  __device__ __forceinline__ float row(const uint8_t* rp) const {
    Frag f;
    load(rp, f);
    return compute(f);
  }
};

// ---------------------------------------------------------------------------
// Q4_0.  Unit u -> blocks 2u and 2u+1 (36 bytes at row offset 36u, 4-byte
// aligned when the row length is a multiple of 16 bytes).  Words w0..w8:
//   w0 = d0 | qs0[0..1] << 16,  w1..w3 = qs0[2..13],  w4 = qs0[14..15] | d1 << 16,
//   w5..w8 = qs1[0..15].
// Block 0 weight j is the low nibble of qs0[j], weight 16+j the high nibble.
// ---------------------------------------------------------------------------
// Full nibble words of a Q4_0 unit that take the byte split (the rest are
// decoded in place): w1..w3 of block 0 (index 0..2), w5..w8 of block 1 (0..3).
// None: measured 76.8 us for the 262144 x 2560 lm_head against 77.6 with
// words 0 and 2 of each block split and 79.1 with every word split (same
// box, two passes); as for Q4_K, the in-place masks issue fewest.
__host__ __device__ constexpr bool q40_split0(int k) { return k < 0; }
__host__ __device__ constexpr bool q40_split1(int k) { return k < 0; }

struct UnitQ40 {
  static constexpr int kFmt = 2;
  static constexpr int kUnitW = 64;
  static constexpr bool kMixed = false;
  static constexpr bool kDirect = false;  // activations staged through shared memory
  static constexpr int kBlockW = 32;
  static constexpr int kBlockBytes = 18;
  float e0[4];               // qs0[0..1] via w0 >> 12: lo0 hi0 lo1 hi1 (pos 4, 8, 12, 16)
  float xl0[12], xh0[12];    // qs0[2..13]: low / high nibble columns 2+k / 18+k
  float g0[4];               // qs0[14..15] via w4: lo14 hi14 lo15 hi15 (pos 0, 4, 8, 12)
  float xl1[16], xh1[16];    // qs1[0..15]
  float s8_0, s8_1;          // 8 * sum(x) * 2^-60 per block
  uint32_t off;

  // Unit u covers columns 64u .. 64u + 63 (blocks 2u, 2u+1).
  __device__ __forceinline__ static void unit_of(int64_t col, int& u, int& l) {
    u = static_cast<int>(col >> 6);
    l = static_cast<int>(col & 63);
  }

  template <class XU>
  __device__ __forceinline__ void setup(int u, const XU& xu) {
    off = 36u * static_cast<uint32_t>(u);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) s0 += xu(c);
#pragma unroll
    for (int c = 32; c < 64; ++c) s1 += xu(c);
    s8_0 = s0 * exp2i(3 - 60);
    s8_1 = s1 * exp2i(3 - 60);
    e0[0] = xu(0) * exp2i(kE - 4);
    e0[1] = xu(16) * exp2i(kE - 8);
    e0[2] = xu(1) * exp2i(kE - 12);
    e0[3] = xu(17) * exp2i(kE - 16);
#pragma unroll
    for (int k = 0; k < 12; ++k) {
      const bool sp = q40_split0(k >> 2);
      xl0[k] = xu(2 + k) * exp2i(sp ? lo_exp<true>(k & 3) : lo_exp<false>(k & 3));
      xh0[k] = xu(18 + k) * exp2i(sp ? hi_exp<true>(k & 3) : hi_exp<false>(k & 3));
    }
    g0[0] = xu(14) * exp2i(kE - 0);
    g0[1] = xu(30) * exp2i(kE - 4);
    g0[2] = xu(15) * exp2i(kE - 8);
    g0[3] = xu(31) * exp2i(kE - 12);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const bool sp = q40_split1(k >> 2);
      xl1[k] = xu(32 + k) * exp2i(sp ? lo_exp<true>(k & 3) : lo_exp<false>(k & 3));
      xh1[k] = xu(48 + k) * exp2i(sp ? hi_exp<true>(k & 3) : hi_exp<false>(k & 3));
    }
  }

  struct Frag {
    uint32_t w[9];
  };

  __device__ __forceinline__ void load(const uint8_t* rp, Frag& f) const {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(rp + off);
#pragma unroll
    for (int i = 0; i < 9; ++i) f.w[i] = q[i];
  }

  __device__ __forceinline__ float compute(const Frag& f) const {
    const uint32_t w0 = f.w[0], w1 = f.w[1], w2 = f.w[2], w3 = f.w[3], w4 = f.w[4];
    const uint32_t w5 = f.w[5], w6 = f.w[6], w7 = f.w[7], w8 = f.w[8];
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    const uint32_t s = w0 >> 12;
    fma2(a0, a1, bits(s & 0xF0u), bits(s & 0xF00u), e0[0], e0[1]);
    fma2(a0, a1, bits(s & 0xF000u), bits(s & 0xF0000u), e0[2], e0[3]);
    nib_word<q40_split0(0)>(w1, xl0 + 0, xh0 + 0, a0, a1, b0, b1);
    nib_word<q40_split0(1)>(w2, xl0 + 4, xh0 + 4, a0, a1, b0, b1);
    nib_word<q40_split0(2)>(w3, xl0 + 8, xh0 + 8, a0, a1, b0, b1);
    fma2(b0, b1, bits(w4 & 0xFu), bits(w4 & 0xF0u), g0[0], g0[1]);
    fma2(b0, b1, bits(w4 & 0xF00u), bits(w4 & 0xF000u), g0[2], g0[3]);
    float c0 = 0.f, c1 = 0.f, e0a = 0.f, e1a = 0.f;
    nib_word<q40_split1(0)>(w5, xl1 + 0, xh1 + 0, c0, c1, e0a, e1a);
    nib_word<q40_split1(1)>(w6, xl1 + 4, xh1 + 4, c0, c1, e0a, e1a);
    nib_word<q40_split1(2)>(w7, xl1 + 8, xh1 + 8, c0, c1, e0a, e1a);
    nib_word<q40_split1(3)>(w8, xl1 + 12, xh1 + 12, c0, c1, e0a, e1a);
    const float d0 = half_bits_to_float(w0) * exp2i(60);
    const float d1 = half_bits_to_float(w4 >> 16) * exp2i(60);
    const float p0 = ((a0 + a1) + (b0 + b1)) - s8_0;
    const float p1 = ((c0 + c1) + (e0a + e1a)) - s8_1;
    return fmaf(d0, p0, d1 * p1);
  }

  __device__ __forceinline__ float row(const uint8_t* rp) const {
    Frag f;
    load(rp, f);
    return compute(f);
  }
};

// ---------------------------------------------------------------------------
// Units over Q8_0 activations (the 8-bit path: infer-compute README §Shaders
// row "Q8" and §Architecture "Q4_0 through legacy Q8 path").  The activation
// vector arrives already quantized, as Q8_0 blocks (34 B / 32 values: f16 d,
// then 32 int8 codes), so a block's product is an exact integer sum of code
// products times the two scales.  The integer sums run on dp4a (four 8-bit
// products and their sum per instruction), which needs no decode to float.
//
// Unit u covers columns 64u .. 64u + 63: activation blocks 2u and 2u + 1,
// 68 bytes at offset 68u of the vector (4-byte aligned when hidden % 64 == 0).
// As 17 words:  x0 = dx0 | a0[0..1] << 16,  x1..x7 = a0[2..29],
//               x8 = a0[30..31] | dx1 << 16, x9..x16 = a1[0..31].
// The lanes read these 68 bytes straight from global memory once per phase
// (kDirect): nothing is staged through shared memory.
// ---------------------------------------------------------------------------

// sum of the four byte products of a (unsigned) and b (signed), plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

__device__ __forceinline__ void load_q8_unit_words(const uint8_t* xq, int u, uint32_t (&x)[17]) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(xq + 68 * static_cast<int64_t>(u));
#pragma unroll
  for (int i = 0; i < 17; ++i) x[i] = p[i];
}

// Q4_0 weights x Q8_0 activations.  The Q4_0 unit is 36 bytes at 36u (words
// w0..w8, as for UnitQ40): w0 = dw0 | qs0[0..1] << 16, w1..w3 = qs0[2..13],
// w4 = qs0[14..15] | dw1 << 16, w5..w8 = qs1[0..15].  Weight j of a block is
// the low nibble of qs[j], weight 16 + j the high nibble, value q - 8.
// The activation words are re-packed once so that byte k of lo0[i] / hi0[i]
// is the activation of the low / high nibble in byte k of weight word i
// (zero against the scale bytes of w0 and w4):
//   lo0 = {x0 & 0xFFFF0000, x1, x2, x3, x4 & 0xFFFF}    a0[0..15]
//   hi0 = {x4 & 0xFFFF0000, x5, x6, x7, x8 & 0xFFFF}    a0[16..31]
//   lo1 = x9..x12 (a1[0..15]),  hi1 = x13..x16 (a1[16..31]).
// Low nibbles are masked in place (0x0F0F0F0F); high nibbles are masked in
// place too (0xF0F0F0F0: 16 q per byte, unsigned), so that sum is 16x and is
// shifted down once.  sum_j (q_j - 8) a_j = sum q a - 8 sum a, with 8 sum a
// precomputed per block.
struct UnitQ40xQ8 {
  static constexpr int kFmt = 2;
  static constexpr int kUnitW = 64;
  static constexpr bool kMixed = false;
  static constexpr bool kDirect = true;
  uint32_t lo0[5], hi0[5], lo1[4], hi1[4];
  float dx0, dx1;
  int c0, c1;        // 8 * sum of the block's activation codes
  uint32_t off;

  __device__ __forceinline__ static void unit_of(int64_t col, int& u, int& l) {
    u = static_cast<int>(col >> 6);
    l = static_cast<int>(col & 63);
  }

  __device__ __forceinline__ void setup(int u, const uint8_t* xq) {
    uint32_t x[17];
    load_q8_unit_words(xq, u, x);
    lo0[0] = x[0] & 0xFFFF0000u;
    hi0[0] = x[4] & 0xFFFF0000u;
#pragma unroll
    for (int i = 1; i < 4; ++i) {
      lo0[i] = x[i];
      hi0[i] = x[4 + i];
    }
    lo0[4] = x[4] & 0xFFFFu;
    hi0[4] = x[8] & 0xFFFFu;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo1[i] = x[9 + i];
      hi1[i] = x[13 + i];
    }
    dx0 = half_bits_to_float(x[0]);
    dx1 = half_bits_to_float(x[8] >> 16);
    int s0 = 0, s1 = 0;
#pragma unroll
    for (int i = 0; i < 5; ++i) s0 = dp4a_ss(hi0[i], 0x01010101u, dp4a_ss(lo0[i], 0x01010101u, s0));
#pragma unroll
    for (int i = 0; i < 4; ++i) s1 = dp4a_ss(hi1[i], 0x01010101u, dp4a_ss(lo1[i], 0x01010101u, s1));
    c0 = 8 * s0;
    c1 = 8 * s1;
    off = 36u * static_cast<uint32_t>(u);
  }

  struct Frag {
    uint32_t w[9];
  };

  __device__ __forceinline__ void load(const uint8_t* rp, Frag& f) const {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(rp + off);
#pragma unroll
    for (int i = 0; i < 9; ++i) f.w[i] = q[i];
  }

  __device__ __forceinline__ float compute(const Frag& f) const {
    int l0 = 0, h0 = 0, l1 = 0, h1 = 0;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      l0 = dp4a_ss(f.w[i] & 0x0F0F0F0Fu, lo0[i], l0);
      h0 = dp4a_us(f.w[i] & 0xF0F0F0F0u, hi0[i], h0);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      l1 = dp4a_ss(f.w[5 + i] & 0x0F0F0F0Fu, lo1[i], l1);
      h1 = dp4a_us(f.w[5 + i] & 0xF0F0F0F0u, hi1[i], h1);
    }
    const int i0 = l0 + (h0 >> 4) - c0;
    const int i1 = l1 + (h1 >> 4) - c1;
    // f16 x f16 products are exact in f32
    const float s0 = half_bits_to_float(f.w[0]) * dx0;
    const float s1 = half_bits_to_float(f.w[4] >> 16) * dx1;
    return fmaf(s0, static_cast<float>(i0), s1 * static_cast<float>(i1));
  }

  __device__ __forceinline__ float row(const uint8_t* rp) const {
    Frag f;
    load(rp, f);
    return compute(f);
  }
};

// Q8_0 weights x Q8_0 activations: the weight unit (68 bytes at 68u) has the
// same word layout as the activation unit, so word i of one pairs with word i
// of the other; the activation's scale bytes are zeroed (x0 low half, x8 high
// half) so the weight's scale bytes multiply 0.
struct UnitQ80xQ8 {
  static constexpr int kFmt = 8;
  static constexpr int kUnitW = 64;
  static constexpr bool kMixed = false;
  static constexpr bool kDirect = true;
  uint32_t a[17];
  float dx0, dx1;
  uint32_t off;

  __device__ __forceinline__ static void unit_of(int64_t col, int& u, int& l) {
    u = static_cast<int>(col >> 6);
    l = static_cast<int>(col & 63);
  }

  __device__ __forceinline__ void setup(int u, const uint8_t* xq) {
    load_q8_unit_words(xq, u, a);
    dx0 = half_bits_to_float(a[0]);
    dx1 = half_bits_to_float(a[8] >> 16);
    a[0] &= 0xFFFF0000u;
    a[8] &= 0xFFFFu;
    off = 68u * static_cast<uint32_t>(u);
  }

  struct Frag {
    uint32_t w[17];
  };

  __device__ __forceinline__ void load(const uint8_t* rp, Frag& f) const {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(rp + off);
#pragma unroll
    for (int i = 0; i < 17; ++i) f.w[i] = q[i];
  }

  __device__ __forceinline__ float compute(const Frag& f) const {
    int i0 = 0, i1 = 0;
#pragma unroll
    for (int i = 0; i < 9; ++i) i0 = dp4a_ss(f.w[i], a[i], i0);
#pragma unroll
    for (int i = 9; i < 17; ++i) i1 = dp4a_ss(f.w[i], a[i], i1);
    const float s0 = half_bits_to_float(f.w[0]) * dx0;
    const float s1 = half_bits_to_float(f.w[8] >> 16) * dx1;
    return fmaf(s0, static_cast<float>(i0), s1 * static_cast<float>(i1));
  }

  __device__ __forceinline__ float row(const uint8_t* rp) const {
    Frag f;
    load(rp, f);
    return compute(f);
  }
};

// ---------------------------------------------------------------------------
// Decoder for a kernel that streams both Q4_K (64-column units) and Q6_K
// (32-column units) phases: one 64-float activation array serves either
// format, so both decode loops share one register allocation.
// ---------------------------------------------------------------------------
struct UnitChain {
  static constexpr bool kMixed = true;
  static constexpr bool kDirect = false;
  bool q6;         // set from the phase's format before setup()
  float x[64];     // Q4_K: xa = x[0..31], xb = x[32..63]; Q6_K: x[16a + i]
  float s[4];      // Q4_K: sxa, sxb; Q6_K: sx32[0..3]
  // Q6_K: block offset, the four operand offsets and the scale shift;
  // Q4_K: off, o1 = chunk offset, o2..o4 / sh = the Q4kSel constants
  uint32_t off, o1, o2, o3, o4, sh;

  template <class XU>
  __device__ __forceinline__ void setup_q4k(int u, const XU& xu) {
    const int kb = u >> 2, c = u & 3;
    off = static_cast<uint32_t>(kb) * 144u;
    o1 = 16u + 32u * c;
    Q4kSel sel;
    sel.set(c);
    o2 = sel.selP;
    o3 = sel.selQ;
    o4 = sel.mask;
    sh = sel.sh;
    float sa = 0.f, sb = 0.f;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
      const float va = xu(l), vb = xu(32 + l);
      sa += va;
      sb += vb;
      x[l] = va * exp2i(q4k_xa_exp<false>(l));
      x[32 + l] = vb * exp2i(q4k_xb_exp<false>(l));
    }
    s[0] = sa;
    s[1] = sb;
  }

  template <class XU>
  __device__ __forceinline__ void setup_q6k(int u, const XU& xu) {
    Q6kUnitGeom g;
    g.set(u);
    off = g.off;
    o1 = g.oA;
    o2 = g.oB;
    o3 = g.oQ;
    o4 = g.oS;
    sh = g.sshift;
    q6k_setup_x<true>(xu, x, s);
  }

  template <class XU>
  __device__ __forceinline__ void setup(int u, const XU& xu) {
    if (q6)
      setup_q6k(u, xu);
    else
      setup_q4k(u, xu);
  }

  __device__ __forceinline__ float row(const uint8_t* rp) const {
    return q6 ? row_q6k(rp) : row_q4k(rp);
  }

  // two rows, one format branch: the two decode chains interleave
  __device__ __forceinline__ void row2(const uint8_t* r0, const uint8_t* r1, float& y0,
                                       float& y1) const {
    if (q6) {
      y0 = row_q6k(r0);
      y1 = row_q6k(r1);
    } else {
      y0 = row_q4k(r0);
      y1 = row_q4k(r1);
    }
  }

  __device__ __forceinline__ float row_q4k(const uint8_t* rp) const {
    const uint8_t* bp = rp + off;
    const uint4 hd = *reinterpret_cast<const uint4*>(bp);
    const uint4 q0 = *reinterpret_cast<const uint4*>(bp + o1);
    const uint4 q1 = *reinterpret_cast<const uint4*>(bp + o1 + 16);
    return q4k_chunk_dot<false>(hd, q0, q1, x, x + 32, s[0], s[1], o2, o3, sh, o4);
  }

  __device__ __forceinline__ float row_q6k(const uint8_t* rp) const {
    const Q6kRow br(rp + off);
    uint32_t A[4], B[4], Q[4], S0, S1;
    br.run16(o1, A);
    br.run16(o2, B);
    br.run16(o3, Q);
    br.run8(o4, S0, S1);
    return q6k_unit_dot<true>(A, B, Q, S0, S1, br.dbits(), x, s, sh);
  }
};

}  // namespace qws
