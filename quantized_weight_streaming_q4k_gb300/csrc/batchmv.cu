// batchmv.cu -- Q4_0 / Q4_K matvec for 2..8 activation vectors that decodes
// every weight once for all vectors (the 262144-row lm_head at batch 8).
//
// The lane-unit engine decodes a weight once per vector (each lane holds one
// vector's activations), which at batch 8 makes the stream ALU-bound.  Here a
// 32-column Q4_0 block times the 8 vectors is a small matrix product done
// with mma.sync (m16n8k16, f16 inputs, f32 accumulation) and kept exact:
//
//   * A = the block's codes q - 8 (integers in [-8, 7], exact in f16), built
//     in registers straight from the packed nibbles (a nibble pair masked
//     under the f16 exponent of 1024 gives 1024 + q; subtracting 1032 gives
//     q - 8 exactly), rows of a 16-row tile;
//   * B = the activations, scaled per vector by a power of two 2^s (exact) so
//     that max |x| lies in [2^13, 2^14), and split into f16 hi + lo parts
//     (hi = f16(x'), lo = f16(x' - hi)), so hi + lo carries x' to 2^-22
//     relative; two MMAs (hi, lo) per 16 columns;
//   * each block's 16 x 8 result starts from zero (exact products summed
//     over 32 columns), is multiplied by the block's scale d per row and
//     added to an f32 running sum in registers; the sums are scaled back by
//     2^-s at the end.
//   * Q4_K: the same per 32-column sub-block with A = the codes q (0..15),
//     scale a = d * sc and the min term b = dmin * m times the sub-block's
//     sum of x' (summed once per launch): acc += a C - b S.
//
// CTA: one copy warp streams 16-row tiles (1-D TMA bulk copies) into a
// shared-memory ring; 16 consumer warps each take a sixteenth of the blocks
// of a tile (a column slice) and the 16 slice sums of each output are added
// in a fixed order.  The activations live in shared memory for the whole launch.
// Every wait is bounded.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "launch.h"

namespace qws {

__device__ unsigned g_err_batchmv;

constexpr int kBmRows = 16;                     // rows per tile (MMA M)
// consumer warps = column slices, per format.  Measured for the 262144 x
// 2560 lm_head at batch 8 (same box, us for 16 / 20 warps): Q4_K 206.1 /
// 199.5 (20: two sub-block pairs per slice, none alone), Q4_0 150.0 / 156.9,
// Q8_0 activations 145.0 / 152.8; 8 warps: Q4_K 263.8.
__host__ __device__ constexpr int bm_warps(int fmt) { return fmt == 12 ? 20 : 16; }
__host__ __device__ constexpr int bm_threads(int fmt) { return 32 + bm_warps(fmt) * 32; }
constexpr int kBmMaxB = 8;                      // MMA N
constexpr int kBmStages = 4;                    // at most; fewer when the rows are wide
constexpr int64_t kBmMaxK = 3072;

// kFmt: 2 Q4_0 / 12 Q4_K weights with f32 activations x; 102 Q4_0 / 108
// Q8_0 weights with Q8_0 activations xq (integer codes exact in f16, no split)
struct BmParams {
  const uint8_t* W;     // rows x K in the weight format
  const float* x;       // [B][K] (f32 activations)
  const uint8_t* xq;    // [B][K / 32 * 34] (Q8_0 activations)
  float* y;             // [B][rows]
  int64_t rows, K;
  int B;
  int n_tiles;          // ceil(rows / 16)
  int stages;           // ring depth, 2..kBmStages
  uint32_t row_bytes;   // K / 32 * 18 = K / 256 * 144
  uint32_t xs_stride;   // f16 elements per staged activation row: K + 8
};

__host__ __device__ constexpr size_t bm_xs_bytes(int64_t K) {
  return static_cast<size_t>(2 * kBmMaxB) * static_cast<size_t>(K + 8) * 2;  // hi and lo
}
// block bytes per 32 weights: Q8_0 34, Q4_0 18, Q4_K 144 / 8 = 18
__host__ __device__ constexpr int64_t bm_block_bytes(int fmt) { return fmt == 108 ? 34 : 18; }
__host__ __device__ constexpr size_t bm_stage_bytes(int64_t K, int fmt) {
  return (static_cast<size_t>(kBmRows) * (K / 32 * bm_block_bytes(fmt)) + 16 + 127) / 128 * 128;
}
__host__ __device__ constexpr size_t bm_fixed_bytes(int64_t K, int fmt) {
  return bm_xs_bytes(K) + 2 * bm_warps(fmt) * kBmRows * kBmMaxB * sizeof(float) +
         kBmMaxB * sizeof(float) + static_cast<size_t>(kBmMaxB) * (K / 32) * sizeof(float) +
         2 * kBmStages * sizeof(uint64_t) + 64;
}
constexpr size_t kBmSmemBudget = 227 * 1024;
// ring depth that fits beside the activations (0 when not even two do)
__host__ __device__ constexpr int bm_stages(int64_t K, int fmt) {
  const size_t f = bm_fixed_bytes(K, fmt), st = bm_stage_bytes(K, fmt);
  const size_t n = f >= kBmSmemBudget ? 0 : (kBmSmemBudget - f) / st;
  return n >= kBmStages ? kBmStages : static_cast<int>(n);
}
__host__ __device__ constexpr size_t bm_smem_bytes(int64_t K, int fmt) {
  return bm_fixed_bytes(K, fmt) + bm_stages(K, fmt) * bm_stage_bytes(K, fmt);
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (lo, hi) nibble pairs of the two bytes of u (byte 0 -> low half) as f16x2
// of q - 8.  One byte permute spreads the two bytes to bytes 0 and 2; a low
// nibble masked in place under the f16 exponent of 1024 gives 1024 + q (one
// three-input logic op), a high nibble under the exponent of 64 gives
// 64 + q (its mantissa step is 1/16); subtracting 1032 or 72 gives q - 8
// exactly.
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t spread16(uint32_t u) { return __byte_perm(u, 0u, 0x4140u); }
__device__ __forceinline__ uint32_t codes_lo(uint32_t u) {
  return f16x2_sub((spread16(u) & 0x000F000Fu) | 0x64006400u, 0x64086408u);
}
__device__ __forceinline__ uint32_t codes_hi(uint32_t u) {
  return f16x2_sub((spread16(u) & 0x00F000F0u) | 0x54005400u, 0x54805480u);
}
// two int8 codes (byte 0 -> low half) as f16x2: offset to 0..255 under the
// f16 exponent of 1024, then 1152 subtracted (exact)
__device__ __forceinline__ uint32_t s8codes(uint32_t u) {
  return f16x2_sub((spread16(u) ^ 0x00800080u) | 0x64006400u, 0x64806480u);
}
// Q4_K codes q (no offset): the low or the high nibble pair as f16x2 of q
__device__ __forceinline__ uint32_t kcodes(uint32_t u, bool high) {
  const uint32_t t = spread16(u);
  return high ? f16x2_sub((t & 0x00F000F0u) | 0x54005400u, 0x54005400u)
              : f16x2_sub((t & 0x000F000Fu) | 0x64006400u, 0x64006400u);
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}

// A fragments of one 32-column block of Q4_0 / Q8_0 weights for rows g
// (pa) and g + 8 (pb): a0 = columns 0..15, a1 = 16..31, as exact f16 codes
template <int kFmt>
__device__ __forceinline__ void q8_block_codes(const uint8_t* pa, const uint8_t* pb, int tq,
                                               uint32_t (&a0)[4], uint32_t (&a1)[4]) {
  if constexpr (kFmt == 102) {
    const uint32_t u0 = ld_u16(pa + 2 + 2 * tq), u1 = ld_u16(pb + 2 + 2 * tq);
    const uint32_t u2 = ld_u16(pa + 10 + 2 * tq), u3 = ld_u16(pb + 10 + 2 * tq);
    a0[0] = codes_lo(u0); a0[1] = codes_lo(u1); a0[2] = codes_lo(u2); a0[3] = codes_lo(u3);
    a1[0] = codes_hi(u0); a1[1] = codes_hi(u1); a1[2] = codes_hi(u2); a1[3] = codes_hi(u3);
  } else {
    a0[0] = s8codes(ld_u16(pa + 2 + 2 * tq));
    a0[1] = s8codes(ld_u16(pb + 2 + 2 * tq));
    a0[2] = s8codes(ld_u16(pa + 10 + 2 * tq));
    a0[3] = s8codes(ld_u16(pb + 10 + 2 * tq));
    a1[0] = s8codes(ld_u16(pa + 18 + 2 * tq));
    a1[1] = s8codes(ld_u16(pb + 18 + 2 * tq));
    a1[2] = s8codes(ld_u16(pa + 26 + 2 * tq));
    a1[3] = s8codes(ld_u16(pb + 26 + 2 * tq));
  }
}

// acc += (dw dx) C for one block's integer product C: rows g (da) and g + 8
// (db), vectors 2 tq and 2 tq + 1 (dx)
__device__ __forceinline__ void q8_block_scale(float (&acc)[4], const float (&c)[4], float da,
                                               float db, float2 dx) {
  acc[0] = fmaf(da * dx.x, c[0], acc[0]);
  acc[1] = fmaf(da * dx.y, c[1], acc[1]);
  acc[2] = fmaf(db * dx.x, c[2], acc[2]);
  acc[3] = fmaf(db * dx.y, c[3], acc[3]);
}

// Scales and mins of the aligned sub-block pair (2c, 2c + 1) of one block,
// from its 16-byte header (d, dmin, the 12 packed scale bytes) in one load:
// a[k] = d * sc(2c + k), b[k] = dmin * m(2c + k), products exact in f32.
__device__ __forceinline__ void q4k_pair_ab(const uint8_t* h, int c, float (&a)[2],
                                            float (&b)[2]) {
  const uint4 hd = *reinterpret_cast<const uint4*>(h);   // block headers are 16-byte aligned
  Q4kSel sel;
  sel.set(c);
  const uint32_t R = q4k_scale_bytes(hd, sel.selP, sel.selQ, sel.sh, sel.mask);
  const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
  a[0] = d * byte_to_float(R, 0);
  a[1] = d * byte_to_float(R, 1);
  b[0] = dmin * byte_to_float(R, 2);
  b[1] = dmin * byte_to_float(R, 3);
}

// a = d * sc(2c + k), b = dmin * m(2c + k) of one sub-block (k = 0, 1)
__device__ __forceinline__ void q4k_sub_ab(const uint8_t* h, int c, int k, float& a, float& b) {
  const uint4 hd = *reinterpret_cast<const uint4*>(h);   // block headers are 16-byte aligned
  Q4kSel sel;
  sel.set(c);
  const uint32_t R = q4k_scale_bytes(hd, sel.selP, sel.selQ, sel.sh, sel.mask);
  a = half_bits_to_float(hd.x) * byte_to_float(R, static_cast<uint32_t>(k));
  b = half_bits_to_float(hd.x >> 16) * byte_to_float(R, static_cast<uint32_t>(2 + k));
}

// acc (rows g, g + 8 x vectors 2tq, 2tq + 1) += a C - b S of Q4_K sub-block bi
__device__ __forceinline__ void q4k_sub(const uint8_t* rg, const uint8_t* rg8, int bi, int tq,
                                        const uint32_t* xh, const uint32_t* xl,
                                        const float* ssum, float (&acc)[4]) {
  const int kb = bi >> 3, j = bi & 7, c = j >> 1;
  const bool high = (j & 1) != 0;
  const uint8_t* ha = rg + kb * 144;
  const uint8_t* hb = rg8 + kb * 144;
  const uint8_t* qa = ha + 16 + 32 * c + 2 * tq;
  const uint8_t* qb = hb + 16 + 32 * c + 2 * tq;
  const uint32_t alo[4] = {kcodes(ld_u16(qa), high), kcodes(ld_u16(qb), high),
                           kcodes(ld_u16(qa + 8), high), kcodes(ld_u16(qb + 8), high)};
  const uint32_t ahi[4] = {kcodes(ld_u16(qa + 16), high), kcodes(ld_u16(qb + 16), high),
                           kcodes(ld_u16(qa + 24), high), kcodes(ld_u16(qb + 24), high)};
  const int w0 = bi * 16 + tq;
  float cc[4] = {0.f, 0.f, 0.f, 0.f};
  mma_16816(cc, alo, xh[w0], xh[w0 + 4]);
  mma_16816(cc, alo, xl[w0], xl[w0 + 4]);
  mma_16816(cc, ahi, xh[w0 + 8], xh[w0 + 12]);
  mma_16816(cc, ahi, xl[w0 + 8], xl[w0 + 12]);
  float aa[2], ba[2], ab[2], bb[2];
  q4k_pair_ab(ha, c, aa, ba);
  q4k_pair_ab(hb, c, ab, bb);
  const bool odd = (j & 1) != 0;
  const float a0 = odd ? aa[1] : aa[0], b0 = odd ? ba[1] : ba[0];
  const float a1 = odd ? ab[1] : ab[0], b1 = odd ? bb[1] : bb[0];
  // ssum [sub-block][vector]: the sums of vectors 2 tq, 2 tq + 1 in one load
  const float2 sv = reinterpret_cast<const float2*>(ssum)[bi * 4 + tq];
  acc[0] = fmaf(a0, cc[0], fmaf(-b0, sv.x, acc[0]));
  acc[1] = fmaf(a0, cc[1], fmaf(-b0, sv.y, acc[1]));
  acc[2] = fmaf(a1, cc[2], fmaf(-b1, sv.x, acc[2]));
  acc[3] = fmaf(a1, cc[3], fmaf(-b1, sv.y, acc[3]));
}

// the aligned pair bi (even), bi + 1: one load of the shared code bytes
__device__ __forceinline__ void q4k_pair(const uint8_t* rg, const uint8_t* rg8, int bi, int tq,
                                         const uint32_t* xh, const uint32_t* xl,
                                         const float* ssum, float (&acc)[4]) {
  const int kb = bi >> 3, j = bi & 7, c = j >> 1;
  const uint8_t* ha = rg + kb * 144;
  const uint8_t* hb = rg8 + kb * 144;
  const uint8_t* qa = ha + 16 + 32 * c + 2 * tq;
  const uint8_t* qb = hb + 16 + 32 * c + 2 * tq;
  const uint32_t u0 = ld_u16(qa), u1 = ld_u16(qb), u2 = ld_u16(qa + 8), u3 = ld_u16(qb + 8);
  const uint32_t u4 = ld_u16(qa + 16), u5 = ld_u16(qb + 16), u6 = ld_u16(qa + 24),
                 u7 = ld_u16(qb + 24);
  const uint32_t l0[4] = {kcodes(u0, false), kcodes(u1, false), kcodes(u2, false),
                          kcodes(u3, false)};
  const uint32_t l1[4] = {kcodes(u4, false), kcodes(u5, false), kcodes(u6, false),
                          kcodes(u7, false)};
  const uint32_t h0[4] = {kcodes(u0, true), kcodes(u1, true), kcodes(u2, true), kcodes(u3, true)};
  const uint32_t h1[4] = {kcodes(u4, true), kcodes(u5, true), kcodes(u6, true), kcodes(u7, true)};
  const int w0 = bi * 16 + tq, w1 = w0 + 16;
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
  mma_16816(c0, l0, xh[w0], xh[w0 + 4]);
  mma_16816(c1, h0, xh[w1], xh[w1 + 4]);
  mma_16816(c0, l0, xl[w0], xl[w0 + 4]);
  mma_16816(c1, h0, xl[w1], xl[w1 + 4]);
  mma_16816(c0, l1, xh[w0 + 8], xh[w0 + 12]);
  mma_16816(c1, h1, xh[w1 + 8], xh[w1 + 12]);
  mma_16816(c0, l1, xl[w0 + 8], xl[w0 + 12]);
  mma_16816(c1, h1, xl[w1 + 8], xl[w1 + 12]);
  // the four threads of an MMA group need the same eight values: thread tq
  // decodes (row g or g + 8 by tq & 1, sub-block 2c + (tq >> 1)) and the
  // group exchanges them by shuffles
  float am, bm;
  q4k_sub_ab((tq & 1) ? hb : ha, c, tq >> 1, am, bm);
  const int q0 = (threadIdx.x & 31) & ~3;   // lane of tq = 0
  const float a0 = __shfl_sync(0xFFFFFFFFu, am, q0), b0 = __shfl_sync(0xFFFFFFFFu, bm, q0);
  const float a1 = __shfl_sync(0xFFFFFFFFu, am, q0 + 1), b1 = __shfl_sync(0xFFFFFFFFu, bm, q0 + 1);
  const float a2 = __shfl_sync(0xFFFFFFFFu, am, q0 + 2), b2 = __shfl_sync(0xFFFFFFFFu, bm, q0 + 2);
  const float a3 = __shfl_sync(0xFFFFFFFFu, am, q0 + 3), b3 = __shfl_sync(0xFFFFFFFFu, bm, q0 + 3);
  const float2 sv = reinterpret_cast<const float2*>(ssum)[bi * 4 + tq];
  const float2 tv = reinterpret_cast<const float2*>(ssum)[(bi + 1) * 4 + tq];
  acc[0] = fmaf(a0, c0[0], fmaf(-b0, sv.x, acc[0]));
  acc[1] = fmaf(a0, c0[1], fmaf(-b0, sv.y, acc[1]));
  acc[2] = fmaf(a1, c0[2], fmaf(-b1, sv.x, acc[2]));
  acc[3] = fmaf(a1, c0[3], fmaf(-b1, sv.y, acc[3]));
  acc[0] = fmaf(a2, c1[0], fmaf(-b2, tv.x, acc[0]));
  acc[1] = fmaf(a2, c1[1], fmaf(-b2, tv.y, acc[1]));
  acc[2] = fmaf(a3, c1[2], fmaf(-b3, tv.x, acc[2]));
  acc[3] = fmaf(a3, c1[3], fmaf(-b3, tv.y, acc[3]));
}

template <int kFmt>   // 2: Q4_0, 12: Q4_K (f32 x); 102: Q4_0, 108: Q8_0 (Q8_0 x)
__global__ void __launch_bounds__(bm_threads(kFmt), 1) batch_q4_matvec_kernel(
    const __grid_constant__ BmParams p) {
  constexpr int kBmWarps = bm_warps(kFmt);
  extern __shared__ __align__(128) uint8_t bm_smem[];
  const int64_t K = p.K;
  __half* xs_hi = reinterpret_cast<__half*>(bm_smem);
  __half* xs_lo = xs_hi + kBmMaxB * p.xs_stride;
  const int S = p.stages;
  uint8_t* ring = bm_smem + bm_xs_bytes(K);
  const size_t stage_bytes = bm_stage_bytes(K, kFmt);
  float* red = reinterpret_cast<float*>(ring + S * stage_bytes);          // [2][8][128]
  float* unscale = red + 2 * kBmWarps * kBmRows * kBmMaxB;                  // [8]
  float* ssum = unscale + kBmMaxB;                                          // [K / 32][8]
  uint64_t* full = reinterpret_cast<uint64_t*>(ssum + kBmMaxB * (K / 32));
  uint64_t* empty = full + kBmStages;

  const int warp = static_cast<int>(threadIdx.x >> 5) - 1;   // -1: the copy warp
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp < 0) {
    // ---- copy warp: tiles cta, cta + grid, ... (weights need nothing from
    // the previous kernel: stream right away)
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int k = 0;
      for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++k) {
        const int s = k % S;
        const uint32_t ph = static_cast<uint32_t>(k / S) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u)) {
          atomicOr(&g_err_batchmv, kErrEmptyWait);
          break;
        }
        const int64_t r0 = static_cast<int64_t>(t) * kBmRows;
        const int64_t nr = min(static_cast<int64_t>(kBmRows), p.rows - r0);
        const uint32_t bytes = static_cast<uint32_t>(nr) * p.row_bytes;   // a multiple of 16
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_copy_g2s(ring + s * stage_bytes, p.W + r0 * p.row_bytes, bytes, &full[s], pol);
      }
      const int first = k > S ? k - S : 0;
      for (int i = first; i < k; ++i)
        if (!mbar_wait(&full[i % S], static_cast<uint32_t>(i / S) & 1u))
          atomicOr(&g_err_batchmv, kErrDrain);
    }
    return;
  }

  // ---- consumers: stage the activations (x comes from the previous kernel)
  pdl_wait();
  const int ct = static_cast<int>(threadIdx.x) - 32;
  if constexpr (kFmt >= 100) {
    // Q8_0 activations: codes to f16 (exact), block scales to f32
    const int64_t nb = K / 32;
    for (int n = warp; n < kBmMaxB; n += kBmWarps) {
      if (lane == 0) unscale[n] = 1.f;
      const uint8_t* xb = p.xq + static_cast<int64_t>(n) * nb * 34;
      for (int64_t i = lane; i < K + 8; i += 32) {
        float v = 0.f;
        if (n < p.B && i < K) v = static_cast<float>(static_cast<int8_t>(xb[(i >> 5) * 34 + 2 + (i & 31)]));
        xs_hi[n * p.xs_stride + i] = __float2half_rn(v);
        xs_lo[n * p.xs_stride + i] = __float2half_rn(0.f);
      }
      // block scales [block][vector]: one float2 per thread and block below
      for (int64_t bk = lane; bk < nb; bk += 32)
        ssum[bk * kBmMaxB + n] = n < p.B ? half_bits_to_float(ld_u16(xb + bk * 34)) : 0.f;
    }
  } else
  for (int n = warp; n < kBmMaxB; n += kBmWarps) {
    // vector n: its power-of-two scale 2^s with max |x| 2^s in [2^13, 2^14)
    float m = 0.f;
    if (n < p.B)
      for (int64_t i = lane; i < K; i += 32) m = fmaxf(m, fabsf(p.x[n * K + i]));
    m = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m)));
    int s = 0;
    if (m > 0.f) {
      const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127;
      s = min(126, max(-126, 13 - e));
    }
    const float sc = exp2i(s);
    if (lane == 0) unscale[n] = exp2i(-s);
    for (int64_t i = lane; i < K + 8; i += 32) {
      float v = 0.f;
      if (n < p.B && i < K) v = p.x[n * K + i] * sc;
      const __half hi = __float2half_rn(v);
      const __half lo = __float2half_rn(v - __half2float(hi));
      xs_hi[n * p.xs_stride + i] = hi;
      xs_lo[n * p.xs_stride + i] = lo;
    }
    if constexpr (kFmt == 12) {
      // sum of x' over each 32-column sub-block, in column order
      for (int64_t bk = lane; bk < K / 32; bk += 32) {
        float t = 0.f;
        if (n < p.B)
          for (int i = 0; i < 32; ++i) t += p.x[n * K + bk * 32 + i] * sc;
        ssum[bk * kBmMaxB + n] = t;                // [sub-block][vector]
      }
    }
  }
  bar_sync(1, kBmWarps * 32);

  const int g = lane >> 2, tq = lane & 3;          // MMA group / thread in group
  const int nblk = static_cast<int>(K / 32);
  // blocks of this warp's slice: an equal share, the first nblk % kBmWarps
  // slices one more
  const int base = nblk / kBmWarps, extra = nblk % kBmWarps;
  const int per = base + (warp < extra ? 1 : 0);
  const int b0 = warp * base + min(warp, extra);
  // activation fragment base of vector g (the B column), f16x2 words
  const uint32_t* xh = reinterpret_cast<const uint32_t*>(xs_hi + g * p.xs_stride);
  const uint32_t* xl = reinterpret_cast<const uint32_t*>(xs_lo + g * p.xs_stride);
  int k = 0;
  for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++k) {
    const int s = k % S;
    const uint32_t ph = static_cast<uint32_t>(k / S) & 1u;
    const bool landed = mbar_wait(&full[s], ph);
    if (!landed) atomicOr(&g_err_batchmv, kErrFullWait);
    const uint8_t* st = ring + s * stage_bytes;
    const uint8_t* rg = st + g * p.row_bytes;          // row g of the tile
    const uint8_t* rg8 = st + (g + 8) * p.row_bytes;   // row g + 8
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (kFmt == 2) {
      // two blocks at a time: two independent MMA chains interleave (an odd
      // slice ends with one block alone)
      int bi = b0;
      for (; landed && bi + 1 < b0 + per; bi += 2) {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        const uint8_t* pa0 = rg + bi * 18;
        const uint8_t* pb0 = rg8 + bi * 18;
        const uint8_t* pa1 = pa0 + 18;
        const uint8_t* pb1 = pb0 + 18;
        // bytes 2tq, 2tq+1 and 2tq+8, 2tq+9 of each row's 16 code bytes;
        // columns 0..15 of a block are the low nibbles, 16..31 the high ones
        const uint32_t u0 = ld_u16(pa0 + 2 + 2 * tq), u1 = ld_u16(pb0 + 2 + 2 * tq);
        const uint32_t u2 = ld_u16(pa0 + 10 + 2 * tq), u3 = ld_u16(pb0 + 10 + 2 * tq);
        const uint32_t v0 = ld_u16(pa1 + 2 + 2 * tq), v1 = ld_u16(pb1 + 2 + 2 * tq);
        const uint32_t v2 = ld_u16(pa1 + 10 + 2 * tq), v3 = ld_u16(pb1 + 10 + 2 * tq);
        const uint32_t alo0[4] = {codes_lo(u0), codes_lo(u1), codes_lo(u2), codes_lo(u3)};
        const uint32_t ahi0[4] = {codes_hi(u0), codes_hi(u1), codes_hi(u2), codes_hi(u3)};
        const uint32_t alo1[4] = {codes_lo(v0), codes_lo(v1), codes_lo(v2), codes_lo(v3)};
        const uint32_t ahi1[4] = {codes_hi(v0), codes_hi(v1), codes_hi(v2), codes_hi(v3)};
        const int w0 = bi * 16 + tq;                      // f16x2 word of column 32 bi + 2 tq
        const int w1 = w0 + 16;                           // block bi + 1
        mma_16816(c0, alo0, xh[w0], xh[w0 + 4]);
        mma_16816(c1, alo1, xh[w1], xh[w1 + 4]);
        mma_16816(c0, alo0, xl[w0], xl[w0 + 4]);
        mma_16816(c1, alo1, xl[w1], xl[w1 + 4]);
        mma_16816(c0, ahi0, xh[w0 + 8], xh[w0 + 12]);
        mma_16816(c1, ahi1, xh[w1 + 8], xh[w1 + 12]);
        mma_16816(c0, ahi0, xl[w0 + 8], xl[w0 + 12]);
        mma_16816(c1, ahi1, xl[w1 + 8], xl[w1 + 12]);
        const float da0 = half_bits_to_float(ld_u16(pa0)), db0 = half_bits_to_float(ld_u16(pb0));
        const float da1 = half_bits_to_float(ld_u16(pa1)), db1 = half_bits_to_float(ld_u16(pb1));
        acc[0] = fmaf(da0, c0[0], acc[0]);
        acc[1] = fmaf(da0, c0[1], acc[1]);
        acc[2] = fmaf(db0, c0[2], acc[2]);
        acc[3] = fmaf(db0, c0[3], acc[3]);
        acc[0] = fmaf(da1, c1[0], acc[0]);
        acc[1] = fmaf(da1, c1[1], acc[1]);
        acc[2] = fmaf(db1, c1[2], acc[2]);
        acc[3] = fmaf(db1, c1[3], acc[3]);
      }
      if (landed && bi < b0 + per) {
        float c0[4] = {0.f, 0.f, 0.f, 0.f};
        const uint8_t* pa0 = rg + bi * 18;
        const uint8_t* pb0 = rg8 + bi * 18;
        const uint32_t u0 = ld_u16(pa0 + 2 + 2 * tq), u1 = ld_u16(pb0 + 2 + 2 * tq);
        const uint32_t u2 = ld_u16(pa0 + 10 + 2 * tq), u3 = ld_u16(pb0 + 10 + 2 * tq);
        const uint32_t alo0[4] = {codes_lo(u0), codes_lo(u1), codes_lo(u2), codes_lo(u3)};
        const uint32_t ahi0[4] = {codes_hi(u0), codes_hi(u1), codes_hi(u2), codes_hi(u3)};
        const int w0 = bi * 16 + tq;
        mma_16816(c0, alo0, xh[w0], xh[w0 + 4]);
        mma_16816(c0, alo0, xl[w0], xl[w0 + 4]);
        mma_16816(c0, ahi0, xh[w0 + 8], xh[w0 + 12]);
        mma_16816(c0, ahi0, xl[w0 + 8], xl[w0 + 12]);
        const float da0 = half_bits_to_float(ld_u16(pa0)), db0 = half_bits_to_float(ld_u16(pb0));
        acc[0] = fmaf(da0, c0[0], acc[0]);
        acc[1] = fmaf(da0, c0[1], acc[1]);
        acc[2] = fmaf(db0, c0[2], acc[2]);
        acc[3] = fmaf(db0, c0[3], acc[3]);
      }
    } else if constexpr (kFmt >= 100) {
      // weights x Q8_0 activations: one MMA per 16 columns (codes exact),
      // then the two block scales: acc += (dw dx) C, dw dx exact in f32; two
      // blocks at a time so that two independent MMA chains interleave
      constexpr int kBB = kFmt == 102 ? 18 : 34;   // weight block bytes
      const float2* dx2 = reinterpret_cast<const float2*>(ssum) + tq;   // [block][4]
      int bi = b0;
      for (; landed && bi + 1 < b0 + per; bi += 2) {
        const uint8_t* pa = rg + bi * kBB;
        const uint8_t* pb = rg8 + bi * kBB;
        uint32_t a0[4], a1[4], e0[4], e1[4];
        q8_block_codes<kFmt>(pa, pb, tq, a0, a1);
        q8_block_codes<kFmt>(pa + kBB, pb + kBB, tq, e0, e1);
        const int w0 = bi * 16 + tq, w1 = w0 + 16;
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(c0, a0, xh[w0], xh[w0 + 4]);
        mma_16816(c1, e0, xh[w1], xh[w1 + 4]);
        mma_16816(c0, a1, xh[w0 + 8], xh[w0 + 12]);
        mma_16816(c1, e1, xh[w1 + 8], xh[w1 + 12]);
        q8_block_scale(acc, c0, half_bits_to_float(ld_u16(pa)), half_bits_to_float(ld_u16(pb)),
                       dx2[bi * 4]);
        q8_block_scale(acc, c1, half_bits_to_float(ld_u16(pa + kBB)),
                       half_bits_to_float(ld_u16(pb + kBB)), dx2[(bi + 1) * 4]);
      }
      if (landed && bi < b0 + per) {
        const uint8_t* pa = rg + bi * kBB;
        const uint8_t* pb = rg8 + bi * kBB;
        uint32_t a0[4], a1[4];
        q8_block_codes<kFmt>(pa, pb, tq, a0, a1);
        const int w0 = bi * 16 + tq;
        float c0[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(c0, a0, xh[w0], xh[w0 + 4]);
        mma_16816(c0, a1, xh[w0 + 8], xh[w0 + 12]);
        q8_block_scale(acc, c0, half_bits_to_float(ld_u16(pa)), half_bits_to_float(ld_u16(pb)),
                       dx2[bi * 4]);
      }
    } else {
      int bi = b0;
      // a sub-block on its own when the slice starts on an odd one
      if (landed && per > 0 && (bi & 1)) {
        q4k_sub(rg, rg8, bi, tq, xh, xl, ssum, acc);
        ++bi;
      }
      // aligned pairs (2c, 2c + 1): the same 32 code bytes, low nibbles for
      // the first, high for the second; two independent MMA chains
      for (; landed && bi + 1 < b0 + per; bi += 2) q4k_pair(rg, rg8, bi, tq, xh, xl, ssum, acc);
      if (landed && bi < b0 + per) q4k_sub(rg, rg8, bi, tq, xh, xl, ssum, acc);
    }
    // slice sums: [row][vector] of this warp, buffer k & 1
    float* rw = red + (static_cast<size_t>(k & 1) * kBmWarps + warp) * (kBmRows * kBmMaxB);
    rw[g * kBmMaxB + 2 * tq] = acc[0];
    rw[g * kBmMaxB + 2 * tq + 1] = acc[1];
    rw[(g + 8) * kBmMaxB + 2 * tq] = acc[2];
    rw[(g + 8) * kBmMaxB + 2 * tq + 1] = acc[3];
    // every slice written and the stage read; a timeout seen by any warp ends
    // all of them here together
    if (bar_sync_or(1, kBmWarps * 32, !landed)) break;
    if (ct == 0) mbar_arrive(&empty[s]);
    if (ct < kBmRows * kBmMaxB) {
      const int row = ct / kBmMaxB, n = ct % kBmMaxB;
      const int64_t r = static_cast<int64_t>(t) * kBmRows + row;
      const float* rb = red + static_cast<size_t>(k & 1) * kBmWarps * (kBmRows * kBmMaxB) + ct;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kBmWarps; ++w) v += rb[w * kBmRows * kBmMaxB];
      if (n < p.B && r < p.rows) p.y[n * p.rows + r] = v * unscale[n];
    }
  }
}

// ------------------------------------------------------------------ host side
bool batch_q4_eligible(int fmt, int64_t K, int B) {
  return (fmt == 2 || fmt == 12 || fmt == 102 || fmt == 108) && B >= 2 && B <= kBmMaxB &&
         K >= 256 && K % 256 == 0 && K <= kBmMaxK && bm_stages(K, fmt) >= 2;
}

template <int kFmt>
static cudaError_t set_smem_attr() {
  // set on every launch (cheap): no per-device cache shared between threads
  return cudaFuncSetAttribute(batch_q4_matvec_kernel<kFmt>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kBmSmemBudget));
}

cudaError_t launch_batch_q4_matvec(int fmt, const uint8_t* W, const float* x, float* y,
                                   int64_t rows, int64_t K, int B, cudaStream_t st,
                                   const uint8_t* xq) {
  BmParams p;
  p.W = W;
  p.x = x;
  p.xq = xq;
  p.y = y;
  p.rows = rows;
  p.K = K;
  p.B = B;
  p.n_tiles = static_cast<int>((rows + kBmRows - 1) / kBmRows);
  p.row_bytes = static_cast<uint32_t>(K / 32 * (fmt == 108 ? 34 : 18));
  p.xs_stride = static_cast<uint32_t>(K + 8);
  p.stages = bm_stages(K, fmt);
  const size_t smem = bm_smem_bytes(K, fmt);
  const cudaError_t ea = fmt == 12    ? set_smem_attr<12>()
                         : fmt == 102 ? set_smem_attr<102>()
                         : fmt == 108 ? set_smem_attr<108>()
                                      : set_smem_attr<2>();
  if (ea != cudaSuccess) return ea;
  const int grid = static_cast<int>(std::min<int64_t>(p.n_tiles, device_sms()));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(bm_threads(fmt));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (fmt) {
    case 12: return cudaLaunchKernelEx(&cfg, batch_q4_matvec_kernel<12>, p);
    case 102: return cudaLaunchKernelEx(&cfg, batch_q4_matvec_kernel<102>, p);
    case 108: return cudaLaunchKernelEx(&cfg, batch_q4_matvec_kernel<108>, p);
    default: return cudaLaunchKernelEx(&cfg, batch_q4_matvec_kernel<2>, p);
  }
}

unsigned read_clear_batchmv_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_batchmv, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_batchmv, &z, sizeof(z));
  return v;
}

}  // namespace qws
