// batchmv.cu -- Q4_0 matvec for 2..8 activation vectors that decodes every
// weight once for all vectors (the 262144-row lm_head at batch 8).
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
//
// CTA: one copy warp streams 16-row tiles (1-D TMA bulk copies) into a
// shared-memory ring; 8 consumer warps each take one eighth of the blocks of
// a tile (a column slice) and the 8 slice sums of each output are added in a
// fixed order.  The activations live in shared memory for the whole launch.
// Every wait is bounded.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "launch.h"

namespace qws {

__device__ unsigned g_err_batchmv;

constexpr int kBmRows = 16;                     // rows per tile (MMA M)
constexpr int kBmWarps = 8;                     // consumer warps = column slices
constexpr int kBmThreads = 32 + kBmWarps * 32;
constexpr int kBmMaxB = 8;                      // MMA N
constexpr int kBmStages = 4;
constexpr int64_t kBmMaxK = 3072;

struct BmParams {
  const uint8_t* W;     // Q4_0, rows x K
  const float* x;       // [B][K]
  float* y;             // [B][rows]
  int64_t rows, K;
  int B;
  int n_tiles;          // ceil(rows / 16)
  uint32_t row_bytes;   // K / 32 * 18
  uint32_t xs_stride;   // f16 elements per staged activation row: K + 8
};

__host__ __device__ constexpr size_t bm_xs_bytes(int64_t K) {
  return static_cast<size_t>(2 * kBmMaxB) * static_cast<size_t>(K + 8) * 2;  // hi and lo
}
__host__ __device__ constexpr size_t bm_stage_bytes(int64_t K) {
  return (static_cast<size_t>(kBmRows) * (K / 32 * 18) + 16 + 127) / 128 * 128;
}
__host__ __device__ constexpr size_t bm_smem_bytes(int64_t K) {
  return bm_xs_bytes(K) + kBmStages * bm_stage_bytes(K) +
         2 * kBmWarps * kBmRows * kBmMaxB * sizeof(float) +   // slice sums, two buffers
         kBmMaxB * sizeof(float) + 2 * kBmStages * sizeof(uint64_t) + 64;
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
// of q - 8: nibbles placed under the f16 exponent of 1024 (0x6400 | q =
// 1024 + q, exact), then 1032 subtracted (exact).
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t codes_lo(uint32_t u) {
  return f16x2_sub((u & 0x000Fu) | ((u & 0x0F00u) << 8) | 0x64006400u, 0x64086408u);
}
__device__ __forceinline__ uint32_t codes_hi(uint32_t u) {
  return f16x2_sub(((u >> 4) & 0x000Fu) | ((u & 0xF000u) << 4) | 0x64006400u, 0x64086408u);
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}

__global__ void __launch_bounds__(kBmThreads, 1) batch_q40_matvec_kernel(
    const __grid_constant__ BmParams p) {
  extern __shared__ __align__(128) uint8_t bm_smem[];
  const int64_t K = p.K;
  __half* xs_hi = reinterpret_cast<__half*>(bm_smem);
  __half* xs_lo = xs_hi + kBmMaxB * p.xs_stride;
  uint8_t* ring = bm_smem + bm_xs_bytes(K);
  const size_t stage_bytes = bm_stage_bytes(K);
  float* red = reinterpret_cast<float*>(ring + kBmStages * stage_bytes);   // [2][8][128]
  float* unscale = red + 2 * kBmWarps * kBmRows * kBmMaxB;                  // [8]
  uint64_t* full = reinterpret_cast<uint64_t*>(unscale + kBmMaxB);
  uint64_t* empty = full + kBmStages;

  const int warp = static_cast<int>(threadIdx.x >> 5) - 1;   // -1: the copy warp
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBmStages; ++s) {
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
        const int s = k % kBmStages;
        const uint32_t ph = static_cast<uint32_t>(k / kBmStages) & 1u;
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
      const int first = k > kBmStages ? k - kBmStages : 0;
      for (int i = first; i < k; ++i)
        if (!mbar_wait(&full[i % kBmStages], static_cast<uint32_t>(i / kBmStages) & 1u))
          atomicOr(&g_err_batchmv, kErrDrain);
    }
    return;
  }

  // ---- consumers: stage the activations (x comes from the previous kernel)
  pdl_wait();
  const int ct = static_cast<int>(threadIdx.x) - 32;
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
    const int s = k % kBmStages;
    const uint32_t ph = static_cast<uint32_t>(k / kBmStages) & 1u;
    const bool landed = mbar_wait(&full[s], ph);
    if (!landed) atomicOr(&g_err_batchmv, kErrFullWait);
    const uint8_t* st = ring + s * stage_bytes;
    const uint8_t* rg = st + g * p.row_bytes;          // row g of the tile
    const uint8_t* rg8 = st + (g + 8) * p.row_bytes;   // row g + 8
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
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
bool batch_q40_eligible(int64_t K, int B) {
  return B >= 2 && B <= kBmMaxB && K >= 256 && K % 256 == 0 && K <= kBmMaxK;
}

cudaError_t launch_batch_q40_matvec(const uint8_t* W, const float* x, float* y, int64_t rows,
                                    int64_t K, int B, cudaStream_t st) {
  BmParams p;
  p.W = W;
  p.x = x;
  p.y = y;
  p.rows = rows;
  p.K = K;
  p.B = B;
  p.n_tiles = static_cast<int>((rows + kBmRows - 1) / kBmRows);
  p.row_bytes = static_cast<uint32_t>(K / 32 * 18);
  p.xs_stride = static_cast<uint32_t>(K + 8);
  const size_t smem = bm_smem_bytes(K);
  static size_t attr_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && attr_smem[dev] < smem) {
    const cudaError_t e = cudaFuncSetAttribute(batch_q40_matvec_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(bm_smem_bytes(kBmMaxK)));
    if (e != cudaSuccess) return e;
    attr_smem[dev] = bm_smem_bytes(kBmMaxK);
  }
  const int grid = static_cast<int>(std::min<int64_t>(p.n_tiles, device_sms()));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, batch_q40_matvec_kernel, p);
}

unsigned read_clear_batchmv_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_batchmv, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_batchmv, &z, sizeof(z));
  return v;
}

}  // namespace qws
