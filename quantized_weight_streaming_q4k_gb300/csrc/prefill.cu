// prefill.cu -- the batch-N (prefill) Q4_K matrix product on the 5th-generation
// tensor cores: Y[n][r] = sum_k W[r][k] * X[n][k] for N token vectors at once
// (infer-compute README §Quick Start / §Shaders, prefill_q4: the seq > 1
// path).  At N >= ~100 the product is compute-bound, so it runs as a GEMM, to
// the same accuracy as the matvecs (|y - y_exact| <= 1e-5 * sum_k |w x|):
// each operand is split into two f16 parts, hi + lo, and three f16 products
// (hi*hi, hi*lo, lo*hi; the lo*lo term is below 2^-22 of the product) are
// accumulated in f32 in tensor memory.
//
//   * X (f32 [N][K]) is scaled per token by a power of two 2^e (max |x| of
//     the token into [2^14, 2^15), exact) and split by a small packing kernel,
//     one warp per token, into hi = f16(x') and lo = f16(x' - hi), written
//     into the workspace already in the shared-memory image the MMA reads:
//     tiles of 256 tokens x 64 columns (32 KB), each a contiguous run in the
//     128-byte-swizzled K-major layout, hi and lo side by side; 2^-e is kept
//     per token for the epilogue.
//   * The weights stay packed in HBM.  One thread copies the tile rows' next
//     super-block (128 rows x 144 bytes) into shared memory with one 2-D tensor
//     copy (TMA); eight decoder warps (two threads per weight row) take their
//     row's 144 bytes into registers (which frees the buffer for the next
//     super-block at once), dequantize w = d*sc*q - dmin*m in f32, scale by
//     2^10 (exact) and split it into f16 hi + lo, stored into the swizzled A
//     tiles.
//   * One thread issues tcgen05.mma (kind::f16, M = 128 rows, N = 256 tokens,
//     K = 16 per instruction, f32 accumulation) with all operands in shared
//     memory: hi*hi into one accumulator, hi*lo and lo*hi into a second (256
//     TMEM columns each); a tcgen05.commit per stage frees that stage when its
//     MMAs have read it.
//   * The decoder warps then read both accumulators back with tcgen05.ld (warp
//     w reads TMEM lanes 32*(w % 4) .. +31 = 32 weight rows, half of the
//     columns), add them, undo the two power-of-two scales and store Y with
//     coalesced 128-byte rows.
//
// Error per output: the splits leave <= 2^-22 of |w| and of |x| each (f16 hi
// keeps 11 bits, lo the next 11), the dropped lo*lo term <= 2^-22 of |w x|, and
// the f32 accumulation in tensor memory adds one rounding per 16-column MMA to
// each accumulator (K / 16 of them): together far inside 1e-5 * sum |w x|.
// Range: the split needs |w| < 64 (2^10 |w| within f16); a decoder that meets
// a larger sub-block scale records kErrPfRange.
//
// Shared-memory layout of one operand tile (K-major, 128-byte swizzle): row i
// (a weight row for A, a token for B) holds 64 f16 = 128 bytes at
// (i / 8) * 1024 + (i % 8) * 128; inside it, 16-byte chunk c (columns
// 8c .. 8c+7) sits at chunk position c ^ (i % 8).  Tiles start on 1024-byte
// boundaries.  Descriptor: start >> 4, leading offset 16 B (unused by this
// layout), stride offset 1024 B between 8-row groups, version 1, swizzle mode
// 128 B.  The k-th 16-column slice of a tile starts 32 * k bytes in.
//
// Every wait is bounded; on a timeout the thread records kErrPrefill* in the
// module's error word and the kernel still frees its tensor memory.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "launch.h"

namespace qws {

__device__ unsigned g_err_prefill;

constexpr int kPfM = 128;                  // weight rows per tile (MMA M, TMEM lanes)
constexpr int kPfN = 256;                  // tokens per tile (MMA N, TMEM columns)
constexpr int kPfK = 64;                   // columns per stage: one 128-byte f16 row
constexpr uint32_t kPfATile = kPfM * kPfK * 2;     // 16 KB
constexpr uint32_t kPfBTile = kPfN * kPfK * 2;     // 32 KB
constexpr uint32_t kPfWBuf = kPfM * 144;           // one Q4_K super-block of every row
constexpr int kPfThreads = 352;            // 3 role warps + 8 decoder warps
constexpr int kPfDecoders = 256;
constexpr float kPfWScale = 1024.0f;       // 2^10: weights into the f16 split's range
static_assert(kPfN == 256, "two accumulators of N = 256 fill the 512 TMEM columns");
// A stage holds A hi, A lo (weight rows) then B hi, B lo (tokens); two stages
// beside the one weight buffer.
struct PfCfg {
  static constexpr uint32_t kStage = 2 * kPfATile + 2 * kPfBTile;   // 96 KB
  static constexpr int kStages = 2;
  static constexpr size_t kSmem = 1024 + kStages * kStage + kPfWBuf + 256;
  static constexpr uint32_t kTmemCols = 512;   // hi*hi accumulator, cross-term accumulator
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// f32 accumulate, f16 A and B, both K-major, N = 256, M = 128.
constexpr uint32_t kPfIdesc = (1u << 4) | (0u << 7) | (0u << 10) |
                              (static_cast<uint32_t>(kPfN >> 3) << 17) |
                              (static_cast<uint32_t>(kPfM >> 4) << 24);

struct PrefillParams {
  CUtensorMap wmap;       // W as a [rows][row_bytes] byte matrix; box 144 x 128
  const uint8_t* W;       // Q4_K, rows x K
  const uint8_t* X16;     // packed f16 tiles [n_tiles_n][KC][hi, lo][32 KB]
  const float* xscale;    // [n_tiles_n * 256] 2^-e per token
  float* Y;               // [N][rows]
  int64_t rows, K, N;
  int KC;                 // K / 64
  int n_tiles_n;
};

// ------------------------------------------------------------ tcgen05 wrappers
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrives on `bar` once every tcgen05.mma this thread issued before has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 2-D tensor copy (TMA) of one box at coordinates (x, y) of `map` into
// shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// two f32 -> packed f16x2 (round to nearest even); lo in bits 0..15
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Shared-memory matrix descriptor of a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// byte offset of 16-byte chunk c of row i inside a swizzled tile
__host__ __device__ constexpr uint32_t sw128_off(uint32_t i, uint32_t c) {
  return (i >> 3) * 1024u + (i & 7u) * 128u + ((c ^ (i & 7u)) << 4);
}

// ------------------------------------------------------------ X packing
// f32 -> f16 hi, and the f32 remainder x - hi (exact) -> f16 lo
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_f16x2(a, b);
  const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  lo = pack_f16x2(a - h.x, b - h.y);
}

// X [N][K] f32 -> per token: 2^e with max |x| 2^e in [2^14, 2^15) (e = 0 for a
// zero token, e clamped to [-126, 126]), then hi / lo f16 tiles of 256 tokens x
// 64 columns in the swizzled image, and xscale = 2^-e.  One CTA of 256 threads
// per token (its maximum by a warp max, then over the 8 warps in shared
// memory); tokens N .. n_tiles_n * 256 - 1 are zero.
__global__ void __launch_bounds__(256) prefill_pack_x_kernel(const float* __restrict__ X,
                                                             uint8_t* __restrict__ X16,
                                                             float* __restrict__ xscale,
                                                             int64_t N, int64_t K,
                                                             int n_tiles_n) {
  __shared__ float wmax[8];
  pdl_launch_dependents();
  pdl_wait();
  const int lane = static_cast<int>(threadIdx.x & 31), warp = static_cast<int>(threadIdx.x >> 5);
  const int64_t tokens = static_cast<int64_t>(n_tiles_n) * kPfN;
  const int KC = static_cast<int>(K / kPfK);
  const int64_t chunks = K / 8;
  for (int64_t tok = blockIdx.x; tok < tokens; tok += gridDim.x) {
    const bool live = tok < N;
    const float* xr = X + tok * K;
    // each thread keeps the 8-column chunks it packs below in registers
    // (K <= 20480: at most 10 chunks of 8 per thread)
    float v[10][8];
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 10; ++j) {
      const int64_t qk = threadIdx.x + static_cast<int64_t>(j) * 256;
      if (live && qk < chunks) {
        const float4* p = reinterpret_cast<const float4*>(xr + qk * 8);
        const float4 a = p[0], b = p[1];
        v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
        v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[j][i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[j][i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    m = wmax[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, wmax[w]);
    __syncthreads();   // wmax is rewritten by the next token
    int e = 0;
    if (m > 0.f) {
      int E;
      frexpf(m, &E);                  // m = f * 2^E, f in [0.5, 1)
      e = min(126, max(-126, 15 - E));
    }
    const float sc = ldexpf(1.0f, e);
    if (threadIdx.x == 0) xscale[tok] = ldexpf(1.0f, -e);
    const int64_t tn = tok / kPfN;
    const uint32_t t = static_cast<uint32_t>(tok - tn * kPfN);
#pragma unroll
    for (int j = 0; j < 10; ++j) {
      const int64_t qk = threadIdx.x + static_cast<int64_t>(j) * 256;
      if (qk < chunks) {
        uint4 hi, lo;
        split_f16x2(v[j][0] * sc, v[j][1] * sc, hi.x, lo.x);
        split_f16x2(v[j][2] * sc, v[j][3] * sc, hi.y, lo.y);
        split_f16x2(v[j][4] * sc, v[j][5] * sc, hi.z, lo.z);
        split_f16x2(v[j][6] * sc, v[j][7] * sc, hi.w, lo.w);
        const int64_t kc = qk / 8;
        const uint32_t c = static_cast<uint32_t>(qk - kc * 8);
        uint8_t* tile = X16 + ((tn * KC + kc) * 2) * static_cast<int64_t>(kPfBTile);
        *reinterpret_cast<uint4*>(tile + sw128_off(t, c)) = hi;
        *reinterpret_cast<uint4*>(tile + kPfBTile + sw128_off(t, c)) = lo;
      }
    }
  }
}

// ------------------------------------------------------------ Q4_K row chunk
// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1), one rounding each (packed FMA)
__device__ __forceinline__ void fma2_to(float& d0, float& d1, float a0, float a1, float b0,
                                        float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Four nibbles (one per byte of n, each 0..15) -> w = a * q + nb (rounded once
// to f32, as fmaf), split into f16 hi (o_hi) and lo (o_lo), two per word.
// Byte k of n is placed under the exponent of 2^23 by one byte permute
// (0x4B0000qq = 2^23 + q, exact); subtracting 2^23 gives q exactly.
__device__ __forceinline__ void nib4_split(uint32_t n, float a, float nb, uint32_t& h0,
                                           uint32_t& h1, uint32_t& l0, uint32_t& l1) {
  const float m0 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7650));
  const float m1 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7651));
  const float m2 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7652));
  const float m3 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7653));
  float q0, q1, q2, q3, w0, w1, w2, w3;
  fma2_to(q0, q1, m0, m1, 1.0f, 1.0f, -8388608.0f, -8388608.0f);
  fma2_to(q2, q3, m2, m3, 1.0f, 1.0f, -8388608.0f, -8388608.0f);
  fma2_to(w0, w1, q0, q1, a, a, nb, nb);
  fma2_to(w2, w3, q2, q3, a, a, nb, nb);
  split_f16x2(w0, w1, h0, l0);
  split_f16x2(w2, w3, h1, l1);
}

// Dequantizes half of the 64-column chunk c (0..3) of one super-block row,
// scaled by 2^10, and stores it as four swizzled 16-byte chunks of the A hi
// tile row and four of the A lo tile row.  hd = the block's first 16 bytes (d,
// dmin, 12 scale bytes), q0/q1 = its qs bytes 32c .. 32c+31.  Column l < 32 is
// the low nibble of qs byte 32c + l (sub-block 2c, half 0), column 32 + l the
// high nibble (sub-block 2c + 1, half 1); w = d*sc*q - dmin*m.  Returns false
// when 2^10 |w| could leave the f16 range (|d sc| * 15 + |dmin m| >= 64).
__device__ __forceinline__ bool q4k_half_split(const uint4 hd, const uint4 q0, const uint4 q1,
                                               int c, int half, uint8_t* tile_hi,
                                               uint8_t* tile_lo, uint32_t row) {
  const bool hi = c >= 2;
  const uint32_t sh = 16u * static_cast<uint32_t>(c & 1) + 8u * static_cast<uint32_t>(half);
  const uint32_t S = hi ? ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u))
                        : (hd.y & 0x3F3F3F3Fu);
  const uint32_t M = hi ? (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u))
                        : (hd.z & 0x3F3F3F3Fu);
  // half 0: sub-block 2c, low nibbles (columns 0..31 of the chunk);
  // half 1: sub-block 2c + 1, high nibbles (columns 32..63)
  const float a = half_bits_to_float(hd.x) * static_cast<float>((S >> sh) & 0xFFu) * kPfWScale;
  const float nb =
      -half_bits_to_float(hd.x >> 16) * static_cast<float>((M >> sh) & 0xFFu) * kPfWScale;
  const bool in_range = fabsf(a) * 15.0f + fabsf(nb) < 65504.0f;
  const uint32_t s0 = 4u * static_cast<uint32_t>(half);
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // 16-byte chunk 4*half + j: columns 8j .. 8j + 7 of this half = nibbles of
    // qs bytes 8j .. 8j + 7 (words 2j, 2j + 1)
    uint4 oh, ol;
    nib4_split((w[2 * j] >> s0) & 0x0F0F0F0Fu, a, nb, oh.x, oh.y, ol.x, ol.y);
    nib4_split((w[2 * j + 1] >> s0) & 0x0F0F0F0Fu, a, nb, oh.z, oh.w, ol.z, ol.w);
    const uint32_t off = sw128_off(row, static_cast<uint32_t>(4 * half + j));
    *reinterpret_cast<uint4*>(tile_hi + off) = oh;
    *reinterpret_cast<uint4*>(tile_lo + off) = ol;
  }
  return in_range;
}

// ------------------------------------------------------------ the GEMM kernel
enum : unsigned {
  kErrPfFull = 16u,      // MMA issuer gave up waiting for a stage
  kErrPfEmpty = 32u,     // a producer gave up waiting for a free stage
  kErrPfDone = 64u,      // the epilogue gave up waiting for the accumulator
  kErrPfW = 128u,        // a wait on the packed-weight buffer gave up
  kErrPfRange = 256u,    // a weight sub-block outside the split's range (|w| >= 64)
};

// Roles (11 warps): warp 0 copies X tiles (B hi and lo), warp 1 issues the
// MMAs and owns the TMEM allocation, warp 2 copies packed weight rows (one
// 144-byte super-block per row per copy, one buffer), warps 3..10 decode (two
// threads per weight row: low-nibble and high-nibble halves) and then run the
// epilogue (warp w reads TMEM lanes 32 * (w % 4) .. + 31, columns of its half
// of the tile).
__global__ void __launch_bounds__(kPfThreads, 1) prefill_q4k_kernel(const __grid_constant__
                                                                    PrefillParams p) {
  constexpr int kStages = PfCfg::kStages;
  constexpr uint32_t kStage = PfCfg::kStage;
  extern __shared__ __align__(1024) uint8_t pf_smem_raw[];
  const uint32_t raw = smem_addr(pf_smem_raw);
  uint8_t* stages = pf_smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* wbuf = stages + kStages * kStage;                      // one super-block buffer
  uint64_t* full = reinterpret_cast<uint64_t*>(wbuf + kPfWBuf);
  uint64_t* empty = full + kStages;
  uint64_t* wfull = empty + kStages;
  uint64_t* wempty = wfull + 1;
  uint64_t* done = wempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int tm = static_cast<int>(blockIdx.x) / p.n_tiles_n;
  const int tn = static_cast<int>(blockIdx.x) - tm * p.n_tiles_n;   // token tile
  const int64_t m0 = static_cast<int64_t>(tm) * kPfM;
  const int KC = p.KC;
  const int KB = KC / 4;
  const int64_t rem = p.rows - m0;
  const int live_rows = static_cast<int>(rem < kPfM ? rem : kPfM);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], kPfDecoders + 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(wfull, 1);
    mbar_init(wempty, kPfDecoders);
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, PfCfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_launch_dependents();
  pdl_wait();   // X16 and xscale are written by the packing kernel just before

  bool ok = true;
  if (warp == 0) {
    // ---- B producer: the hi and lo tiles of one 64-column chunk per stage
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const uint8_t* xb = p.X16 + static_cast<int64_t>(tn) * KC * 2 * kPfBTile;
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kStages;
        const uint32_t ph = static_cast<uint32_t>(kc / kStages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u)) {
          atomicOr(&g_err_prefill, kErrPfEmpty);
          break;
        }
        mbar_arrive_expect_tx(&full[s], 2 * kPfBTile);
        uint8_t* dst = stages + s * kStage + 2 * kPfATile;
        const uint8_t* src = xb + static_cast<int64_t>(kc) * 2 * kPfBTile;
        bulk_copy_g2s(dst, src, kPfBTile, &full[s], pol);
        bulk_copy_g2s(dst + kPfBTile, src + kPfBTile, kPfBTile, &full[s], pol);
      }
    }
  } else if (warp == 2) {
    // ---- W producer: super-block kb of the tile's 128 rows, one 2-D tensor
    // copy (rows past the matrix end are zero-filled and still counted); the
    // decoders take the bytes into registers and free the buffer at once
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(wempty, (static_cast<uint32_t>(kb) & 1u) ^ 1u)) {
          atomicOr(&g_err_prefill, kErrPfW);
          break;
        }
        mbar_arrive_expect_tx(wfull, kPfWBuf);
        tma_load_2d(wbuf, &p.wmap, kb * 144, static_cast<int>(m0), wfull, pol);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: per 16-column slice, hi*hi into accumulator 0, hi*lo
    // and lo*hi into accumulator 1 (256 columns further)
    if (lane == 0) {
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kStages;
        const uint32_t ph = static_cast<uint32_t>(kc / kStages) & 1u;
        if (!mbar_wait(&full[s], ph)) {
          atomicOr(&g_err_prefill, kErrPfFull);
          break;
        }
        tc_fence_after();
        const uint32_t ahi = smem_addr(stages + s * kStage);
        const uint32_t alo = ahi + kPfATile;
        const uint32_t bhi = ahi + 2 * kPfATile;
        const uint32_t blo = bhi + kPfBTile;
#pragma unroll
        for (int k = 0; k < kPfK / 16; ++k) {
          const uint32_t first = (kc | k) != 0 ? 1u : 0u;
          tc_mma_f16(tmem, sw128_desc(ahi + 32u * k), sw128_desc(bhi + 32u * k), kPfIdesc, first);
          tc_mma_f16(tmem + static_cast<uint32_t>(kPfN), sw128_desc(ahi + 32u * k),
                     sw128_desc(blo + 32u * k), kPfIdesc, first);
          tc_mma_f16(tmem + static_cast<uint32_t>(kPfN), sw128_desc(alo + 32u * k),
                     sw128_desc(bhi + 32u * k), kPfIdesc, 1u);
        }
        tc_commit(&empty[s]);
      }
      // the accumulators are final once every MMA above has completed
      tc_commit(done);
    }
  } else {
    // ---- decoders: thread d -> weight row d / 2 of the tile, half d % 2
    const int d = static_cast<int>(threadIdx.x) - 96;
    const uint32_t row = static_cast<uint32_t>(d >> 1);
    const int half = d & 1;
    const bool live = static_cast<int>(row) < live_rows;
    bool in_range = true;
    uint4 hd = make_uint4(0u, 0u, 0u, 0u), qs[8];
    for (int kc = 0; kc < KC; ++kc) {
      const int s = kc % kStages;
      const uint32_t ph = static_cast<uint32_t>(kc / kStages) & 1u;
      const int kb = kc >> 2, c = kc & 3;
      if (c == 0) {
        // the row's super-block: into registers, then the buffer is free
        if (!mbar_wait(wfull, static_cast<uint32_t>(kb) & 1u)) {
          atomicOr(&g_err_prefill, kErrPfW);
          ok = false;
          break;
        }
        const uint8_t* bp = wbuf + row * 144u;
        hd = *reinterpret_cast<const uint4*>(bp);
#pragma unroll
        for (int i = 0; i < 8; ++i) qs[i] = *reinterpret_cast<const uint4*>(bp + 16 + 16 * i);
        mbar_arrive(wempty);
      }
      if (!mbar_wait(&empty[s], ph ^ 1u)) {
        atomicOr(&g_err_prefill, kErrPfEmpty);
        ok = false;
        break;
      }
      uint8_t* tile = stages + s * kStage;
      if (live) {
        // chunk c's 32 qs bytes are registers 2c and 2c + 1
        uint4 q0 = qs[0], q1 = qs[1];
        if (c == 1) { q0 = qs[2]; q1 = qs[3]; }
        if (c == 2) { q0 = qs[4]; q1 = qs[5]; }
        if (c == 3) { q0 = qs[6]; q1 = qs[7]; }
        in_range = q4k_half_split(hd, q0, q1, c, half, tile, tile + kPfATile, row) && in_range;
      } else {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = sw128_off(row, static_cast<uint32_t>(4 * half + j));
          *reinterpret_cast<uint4*>(tile + off) = z;
          *reinterpret_cast<uint4*>(tile + kPfATile + off) = z;
        }
      }
      fence_proxy_async_smem();   // generic-proxy stores -> visible to the MMA
      mbar_arrive(&full[s]);
    }
    if (!in_range) atomicOr(&g_err_prefill, kErrPfRange);
    // ---- epilogue: y = (hi*hi + cross terms) * 2^-10 * 2^-e(token)
    if (!mbar_wait(done, 0u)) {
      atomicOr(&g_err_prefill, kErrPfDone);
      ok = false;
    }
    tc_fence_after();
    if (ok) {
      const int q = warp & 3;
      // warps 3..6 take the first 128 token columns, 7..10 the rest
      constexpr int kCols = kPfN / 2;
      const int colh = (warp - 3) >> 2;
      const int64_t rr = m0 + 32 * q + lane;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16);
      const int64_t n0 = static_cast<int64_t>(tn) * kPfN;
      for (int cc = colh * kCols; cc < (colh + 1) * kCols; cc += 16) {
        uint32_t v0[16], v1[16];
        tc_ld16(tbase + static_cast<uint32_t>(cc), v0);
        tc_ld16(tbase + static_cast<uint32_t>(kPfN + cc), v1);
        tc_wait_ld();
        if (rr < p.rows) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int64_t n = n0 + cc + j;
            if (n < p.N) {
              const float y = __uint_as_float(v0[j]) + __uint_as_float(v1[j]);
              p.Y[n * p.rows + rr] = y * (1.0f / kPfWScale) * p.xscale[n];
            }
          }
        }
      }
    }
  }
  // every MMA has completed before the accumulators are freed: wait (bounded)
  // for the final commit on all paths, including after a timeout
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0 && !mbar_wait(done, 0u)) atomicOr(&g_err_prefill, kErrPfDone);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, PfCfg::kTmemCols);
  }
}

// ------------------------------------------------------------ host side
// Token tiles of 256.  Workspace: per token tile and 64-column chunk the hi and
// lo f16 tiles (2 x 32 KB), then one f32 scale per padded token.
static int64_t token_tiles(int64_t n_tokens) { return (n_tokens + kPfN - 1) / kPfN; }

static size_t prefill_tiles_bytes(int64_t hidden, int64_t n_tokens) {
  return static_cast<size_t>(token_tiles(n_tokens)) * kPfN * static_cast<size_t>(hidden) * 2 * 2;
}

size_t prefill_workspace_bytes(int64_t hidden, int64_t n_tokens) {
  return prefill_tiles_bytes(hidden, n_tokens) +
         static_cast<size_t>(token_tiles(n_tokens)) * kPfN * sizeof(float);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  // a function-local static: initialised once, thread-safe
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

// W viewed as a byte matrix [rows][row_bytes]; boxes of 144 bytes (one
// super-block) x 128 rows.
static bool encode_w_map(CUtensorMap* map, const uint8_t* W, int64_t rows, int64_t K) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 256 * 144),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 256 * 144)};
  const cuuint32_t box[2] = {144u, static_cast<cuuint32_t>(kPfM)};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(W), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class... KArgs, class... Args>
static cudaError_t launch_pdl_pf(void (*kernel)(KArgs...), int grid, int threads, size_t smem,
                                 cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

static cudaError_t launch_prefill_kernel(const PrefillParams& p, int grid, cudaStream_t st) {
  // set on every launch (cheap): no per-device cache shared between threads
  const cudaError_t e = cudaFuncSetAttribute(prefill_q4k_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(PfCfg::kSmem));
  if (e != cudaSuccess) return e;
  return launch_pdl_pf(prefill_q4k_kernel, grid, kPfThreads, PfCfg::kSmem, st, p);
}

cudaError_t launch_prefill_q4k(const uint8_t* W, const float* X, float* Y, int64_t rows,
                               int64_t K, int64_t N, uint8_t* ws, cudaStream_t st) {
  const int n_tiles_n = static_cast<int>(token_tiles(N));
  const int n_tiles_m = static_cast<int>((rows + kPfM - 1) / kPfM);
  float* xscale = reinterpret_cast<float*>(ws + prefill_tiles_bytes(K, N));
  const int64_t tokens = static_cast<int64_t>(n_tiles_n) * kPfN;
  const int64_t pack_blocks = std::min<int64_t>(tokens, 8 * device_sms());
  cudaError_t e = launch_pdl_pf(prefill_pack_x_kernel, static_cast<int>(pack_blocks), 256, 0, st,
                                X, ws, xscale, N, K, n_tiles_n);
  if (e != cudaSuccess) return e;
  PrefillParams p;
  if (!encode_w_map(&p.wmap, W, rows, K)) return cudaErrorInvalidValue;
  p.W = W;
  p.X16 = ws;
  p.xscale = xscale;
  p.Y = Y;
  p.rows = rows;
  p.K = K;
  p.N = N;
  p.KC = static_cast<int>(K / kPfK);
  p.n_tiles_n = n_tiles_n;
  return launch_prefill_kernel(p, n_tiles_m * n_tiles_n, st);
}

unsigned read_clear_prefill_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_prefill, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_prefill, &z, sizeof(z));
  return v;
}

}  // namespace qws
