// prefill.cu -- the batch-N (prefill) Q4_K matrix product on the 5th-generation
// tensor cores: Y[n][r] = sum_k W[r][k] * X[n][k] for N token vectors at once
// (infer-compute README §Quick Start / §Shaders, prefill_q4: the seq > 1
// path).  At N >= ~100 the product is compute-bound, so it runs as a GEMM:
//
//   * X (f32 [N][K]) is first rounded to f16 and written, by a small packing
//     kernel, into the workspace already in the shared-memory image the MMA
//     reads: tiles of 256 tokens x 64 columns (32 KB), each a contiguous run
//     in the 128-byte-swizzled K-major layout.  A tile then moves into shared
//     memory as one 1-D bulk copy (TMA).
//   * The weights stay packed in HBM.  One thread copies the tile rows' next
//     super-block (128 rows x 144 bytes) into shared memory with one 2-D
//     tensor copy (TMA, two buffers); eight decoder warps (two threads per weight row) dequantize
//     w = d*sc*q - dmin*m in f32, round to f16 and store the row's 128 bytes
//     of each 64-column chunk into the swizzled A tile.
//   * One thread issues tcgen05.mma (kind::f16, M = 128 rows, N = 256 tokens,
//     K = 16 per instruction, f32 accumulation) with both operands in shared
//     memory and the accumulator in tensor memory (256 TMEM columns); a
//     tcgen05.commit per stage frees that stage when its MMAs have read it.
//   * The decoder warps then read the accumulator back with tcgen05.ld (warp
//     w reads TMEM lanes 32*(w % 4) .. +31 = 32 weight rows, half of the
//     columns) and store Y with coalesced 128-byte rows.
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
// TMEM columns: a power of two >= 32 that holds the N accumulator columns
constexpr uint32_t kPfTmemCols = kPfN <= 32 ? 32u : kPfN <= 64 ? 64u : kPfN <= 128 ? 128u : 256u;
static_assert(kPfN % 16 == 0 && kPfN <= 256, "MMA N must be a multiple of 16 up to 256");
// A CTA computes kAcc token tiles of 256 against one decoded weight tile
// (kAcc accumulators of 256 TMEM columns side by side), so one decode of the
// weights serves 256 * kAcc tokens.  A stage holds the weight tile and kAcc
// token tiles; as many stages as fit beside the two weight buffers in 227 KB.
template <int kAcc>
struct PfCfg {
  static constexpr uint32_t kStage = kPfATile + kAcc * kPfBTile;
  static constexpr int kStages =
      static_cast<int>((227u * 1024u - 1024u - 2u * kPfWBuf - 256u) / kStage);
  static constexpr size_t kSmem = 1024 + kStages * kStage + 2 * kPfWBuf + 256;
  static constexpr uint32_t kTmemCols = kAcc == 1 ? kPfTmemCols : 512u;
  static_assert(kStages >= 2, "shared memory too small for two stages");
  static_assert(kAcc == 1 || (kAcc == 2 && kPfN == 256), "two accumulators fill the 512 columns");
};

// f32 accumulate, f16 A and B, both K-major, N = 256, M = 128.
constexpr uint32_t kPfIdesc = (1u << 4) | (0u << 7) | (0u << 10) |
                              (static_cast<uint32_t>(kPfN >> 3) << 17) |
                              (static_cast<uint32_t>(kPfM >> 4) << 24);

struct PrefillParams {
  CUtensorMap wmap;       // W as a [rows][row_bytes] byte matrix; box 144 x 128
  const uint8_t* W;       // Q4_K, rows x K
  const uint8_t* X16;     // packed f16 tiles [n_tiles_n][KC][32 KB] (n_tiles_n % kAcc == 0)
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
// X [N][K] f32 -> f16 tiles of 256 tokens x 64 columns in the swizzled image;
// tokens N .. n_tiles_n * 256 - 1 are zero.
__global__ void __launch_bounds__(256) prefill_pack_x_kernel(const float* __restrict__ X,
                                                             uint8_t* __restrict__ X16,
                                                             int64_t N, int64_t K,
                                                             int n_tiles_n) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t chunks = K / 8;
  const int64_t total = static_cast<int64_t>(n_tiles_n) * kPfN * chunks;
  const int KC = static_cast<int>(K / kPfK);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = i / chunks;
    const int64_t qk = i - tok * chunks;
    float v[8];
    if (tok < N) {
      const float4* p = reinterpret_cast<const float4*>(X + tok * K + qk * 8);
      const float4 a = p[0], b = p[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.f;
    }
    uint4 o;
    o.x = pack_f16x2(v[0], v[1]);
    o.y = pack_f16x2(v[2], v[3]);
    o.z = pack_f16x2(v[4], v[5]);
    o.w = pack_f16x2(v[6], v[7]);
    const int64_t tn = tok / kPfN;
    const uint32_t t = static_cast<uint32_t>(tok - tn * kPfN);
    const int64_t kc = qk / 8;
    const uint32_t c = static_cast<uint32_t>(qk - kc * 8);
    uint8_t* tile = X16 + (tn * KC + kc) * static_cast<int64_t>(kPfBTile);
    *reinterpret_cast<uint4*>(tile + sw128_off(t, c)) = o;
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

// Four nibbles (one per byte of n, each 0..15) -> f16(a * q + nb), packed in
// two words.  Byte k of n is placed under the exponent of 2^23 by one byte
// permute (0x4B0000qq = 2^23 + q, exact); subtracting 2^23 gives q exactly, and
// a * q + nb is rounded once to f32 (the same value as fmaf), then to f16.
__device__ __forceinline__ void nib4_to_f16(uint32_t n, float a, float nb, uint32_t& o0,
                                            uint32_t& o1) {
  const float m0 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7650));
  const float m1 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7651));
  const float m2 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7652));
  const float m3 = __uint_as_float(__byte_perm(n, 0x4B000000u, 0x7653));
  float q0, q1, q2, q3, w0, w1, w2, w3;
  fma2_to(q0, q1, m0, m1, 1.0f, 1.0f, -8388608.0f, -8388608.0f);
  fma2_to(q2, q3, m2, m3, 1.0f, 1.0f, -8388608.0f, -8388608.0f);
  fma2_to(w0, w1, q0, q1, a, a, nb, nb);
  fma2_to(w2, w3, q2, q3, a, a, nb, nb);
  o0 = pack_f16x2(w0, w1);
  o1 = pack_f16x2(w2, w3);
}

// Dequantizes half of the 64-column chunk c (0..3) of one super-block row to
// f32 and stores it as four swizzled 16-byte f16 chunks of the A tile row.
// hd = the block's first 16 bytes (d, dmin, 12 scale bytes), q0/q1 = its qs
// bytes 32c .. 32c+31.  Column l < 32 is the low nibble of qs byte 32c + l
// (sub-block 2c, half 0), column 32 + l the high nibble (sub-block 2c + 1,
// half 1); w = d*sc*q - dmin*m.
__device__ __forceinline__ void q4k_half_to_f16(const uint4 hd, const uint4 q0, const uint4 q1,
                                                int c, int half, uint8_t* tile, uint32_t row) {
  const bool hi = c >= 2;
  const uint32_t sh = 16u * static_cast<uint32_t>(c & 1) + 8u * static_cast<uint32_t>(half);
  const uint32_t S = hi ? ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u))
                        : (hd.y & 0x3F3F3F3Fu);
  const uint32_t M = hi ? (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u))
                        : (hd.z & 0x3F3F3F3Fu);
  // half 0: sub-block 2c, low nibbles (columns 0..31 of the chunk);
  // half 1: sub-block 2c + 1, high nibbles (columns 32..63)
  const float a = half_bits_to_float(hd.x) * static_cast<float>((S >> sh) & 0xFFu);
  const float nb = -half_bits_to_float(hd.x >> 16) * static_cast<float>((M >> sh) & 0xFFu);
  const uint32_t s0 = 4u * static_cast<uint32_t>(half);
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // 16-byte chunk 4*half + j: columns 8j .. 8j + 7 of this half = nibbles of
    // qs bytes 8j .. 8j + 7 (words 2j, 2j + 1)
    uint4 o;
    nib4_to_f16((w[2 * j] >> s0) & 0x0F0F0F0Fu, a, nb, o.x, o.y);
    nib4_to_f16((w[2 * j + 1] >> s0) & 0x0F0F0F0Fu, a, nb, o.z, o.w);
    *reinterpret_cast<uint4*>(tile + sw128_off(row, static_cast<uint32_t>(4 * half + j))) = o;
  }
}

// ------------------------------------------------------------ the GEMM kernel
enum : unsigned {
  kErrPfFull = 16u,      // MMA issuer gave up waiting for a stage
  kErrPfEmpty = 32u,     // a producer gave up waiting for a free stage
  kErrPfDone = 64u,      // the epilogue gave up waiting for the accumulator
  kErrPfW = 128u,        // a wait on the packed-weight buffers gave up
};

// Roles (11 warps): warp 0 copies X tiles (B), warp 1 issues the MMAs and
// owns the TMEM allocation, warp 2 copies packed weight rows (one 144-byte
// super-block per row per copy, two buffers), warps 3..10 decode (two
// threads per weight row: low-nibble and high-nibble halves) and then run
// the epilogue (warp w reads TMEM lanes 32 * (w % 4) .. + 31, columns of its
// half of the tile).
template <int kAcc>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_q4k_kernel(const __grid_constant__
                                                                    PrefillParams p) {
  constexpr int kPfStages = PfCfg<kAcc>::kStages;
  constexpr uint32_t kPfStage = PfCfg<kAcc>::kStage;
  extern __shared__ __align__(1024) uint8_t pf_smem_raw[];
  const uint32_t raw = smem_addr(pf_smem_raw);
  uint8_t* stages = pf_smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* wbuf = stages + kPfStages * kPfStage;                 // 2 x kPfWBuf
  uint64_t* full = reinterpret_cast<uint64_t*>(wbuf + 2 * kPfWBuf);
  uint64_t* empty = full + kPfStages;
  uint64_t* wfull = empty + kPfStages;
  uint64_t* wempty = wfull + 2;
  uint64_t* done = wempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int n_groups = p.n_tiles_n / kAcc;
  const int tm = static_cast<int>(blockIdx.x) / n_groups;
  const int tg = static_cast<int>(blockIdx.x) - tm * n_groups;   // token tiles kAcc*tg ..
  const int64_t m0 = static_cast<int64_t>(tm) * kPfM;
  const int KC = p.KC;
  const int KB = KC / 4;
  const int64_t rem = p.rows - m0;
  const int live_rows = static_cast<int>(rem < kPfM ? rem : kPfM);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&full[s], kPfDecoders + 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&wfull[b], 1);
      mbar_init(&wempty[b], kPfDecoders);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, PfCfg<kAcc>::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_launch_dependents();
  pdl_wait();   // X16 is written by the packing kernel just before

  bool ok = true;
  if (warp == 0) {
    // ---- B producer: one 32 KB bulk copy per stage
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const uint8_t* xb = p.X16 + static_cast<int64_t>(tg) * kAcc * KC * kPfBTile;
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kPfStages;
        const uint32_t ph = static_cast<uint32_t>(kc / kPfStages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u)) {
          atomicOr(&g_err_prefill, kErrPfEmpty);
          break;
        }
        mbar_arrive_expect_tx(&full[s], kAcc * kPfBTile);
#pragma unroll
        for (int a = 0; a < kAcc; ++a)
          bulk_copy_g2s(stages + s * kPfStage + kPfATile + a * kPfBTile,
                        xb + (static_cast<int64_t>(a) * KC + kc) * kPfBTile, kPfBTile, &full[s],
                        pol);
      }
    }
  } else if (warp == 2) {
    // ---- W producer: super-block kb of the tile's 128 rows, one 2-D tensor
    // copy (rows past the matrix end are zero-filled and still counted)
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int kb = 0; kb < KB; ++kb) {
        const int b = kb & 1;
        const uint32_t ph = static_cast<uint32_t>(kb >> 1) & 1u;
        if (!mbar_wait(&wempty[b], ph ^ 1u)) {
          atomicOr(&g_err_prefill, kErrPfW);
          break;
        }
        mbar_arrive_expect_tx(&wfull[b], kPfWBuf);
        tma_load_2d(wbuf + b * kPfWBuf, &p.wmap, kb * 144, static_cast<int>(m0), &wfull[b], pol);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kPfStages;
        const uint32_t ph = static_cast<uint32_t>(kc / kPfStages) & 1u;
        if (!mbar_wait(&full[s], ph)) {
          atomicOr(&g_err_prefill, kErrPfFull);
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_addr(stages + s * kPfStage);
#pragma unroll
        for (int k = 0; k < kPfK / 16; ++k) {
#pragma unroll
          for (int t = 0; t < kAcc; ++t)
            tc_mma_f16(tmem + static_cast<uint32_t>(t * kPfN), sw128_desc(a + 32u * k),
                       sw128_desc(a + kPfATile + t * kPfBTile + 32u * k), kPfIdesc,
                       (kc | k) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
      }
      // the accumulator is final once every MMA above has completed
      tc_commit(done);
    }
  } else {
    // ---- decoders: thread d -> weight row d / 2 of the tile, half d % 2
    const int d = static_cast<int>(threadIdx.x) - 96;
    const uint32_t row = static_cast<uint32_t>(d >> 1);
    const int half = d & 1;
    const bool live = static_cast<int>(row) < live_rows;
    for (int kc = 0; kc < KC; ++kc) {
      const int s = kc % kPfStages;
      const uint32_t ph = static_cast<uint32_t>(kc / kPfStages) & 1u;
      const int kb = kc >> 2, c = kc & 3, b = kb & 1;
      if (c == 0 && !mbar_wait(&wfull[b], static_cast<uint32_t>(kb >> 1) & 1u)) {
        atomicOr(&g_err_prefill, kErrPfW);
        ok = false;
        break;
      }
      if (!mbar_wait(&empty[s], ph ^ 1u)) {
        atomicOr(&g_err_prefill, kErrPfEmpty);
        ok = false;
        break;
      }
      uint8_t* tile = stages + s * kPfStage;
      if (live) {
        const uint8_t* bp = wbuf + b * kPfWBuf + row * 144u;
        const uint4 hd = *reinterpret_cast<const uint4*>(bp);
        const uint4 q0 = *reinterpret_cast<const uint4*>(bp + 16 + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4*>(bp + 32 + 32 * c);
        q4k_half_to_f16(hd, q0, q1, c, half, tile, row);
      } else {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(tile + sw128_off(row, static_cast<uint32_t>(4 * half + j))) =
              z;
      }
      fence_proxy_async_smem();   // generic-proxy stores -> visible to the MMA
      mbar_arrive(&full[s]);
      if (c == 3) mbar_arrive(&wempty[b]);   // this super-block's bytes are read
    }
    // ---- epilogue
    if (!mbar_wait(done, 0u)) {
      atomicOr(&g_err_prefill, kErrPfDone);
      ok = false;
    }
    tc_fence_after();
    if (ok) {
      const int q = warp & 3;
      // warps 3..6 take the first half of the kAcc * 256 columns, 7..10 the
      // rest; column c is token n0 + c (the accumulators are adjacent)
      constexpr int kCols = kAcc * kPfN / 2;
      const int colh = (warp - 3) >> 2;
      const int64_t rr = m0 + 32 * q + lane;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16);
      const int64_t n0 = static_cast<int64_t>(tg) * kAcc * kPfN;
      for (int cc = colh * kCols; cc < (colh + 1) * kCols; cc += 16) {
        uint32_t v[16];
        tc_ld16(tbase + static_cast<uint32_t>(cc), v);
        tc_wait_ld();
        if (rr < p.rows) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int64_t n = n0 + cc + j;
            if (n < p.N) p.Y[n * p.rows + rr] = __uint_as_float(v[j]);
          }
        }
      }
    }
  }
  // every MMA has completed before the accumulator is freed: wait (bounded)
  // for the final commit on all paths, including after a timeout
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0 && !mbar_wait(done, 0u)) atomicOr(&g_err_prefill, kErrPfDone);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, PfCfg<kAcc>::kTmemCols);
  }
}

// ------------------------------------------------------------ host side
// Token tiles of 256; the workspace always has room for an even count (the
// two-accumulator kernel reads tiles in pairs, the last one zero when odd).
static int64_t token_tiles(int64_t n_tokens) { return (n_tokens + kPfN - 1) / kPfN; }

size_t prefill_workspace_bytes(int64_t hidden, int64_t n_tokens) {
  const int64_t t = token_tiles(n_tokens);
  const int64_t padded = t >= 2 ? (t + 1) / 2 * 2 : t;
  return static_cast<size_t>(padded) * kPfN * static_cast<size_t>(hidden) * 2;
}

// One or two accumulators per CTA: two halve the weight decoding per token
// but give a CTA about 1.72x the work of a one-accumulator CTA (measured on
// GB300 at 10240 x 2560: two stages instead of three), so they pay when they
// save a wave: compare waves x relative CTA time.
static int prefill_acc(int64_t rows, int64_t n_tokens, int sms) {
  const int64_t mt = (rows + kPfM - 1) / kPfM, t1 = token_tiles(n_tokens);
  if (t1 < 2) return 1;
  const int64_t r1 = (mt * t1 + sms - 1) / sms;
  const int64_t r2 = (mt * ((t1 + 1) / 2) + sms - 1) / sms;
  return r2 * 172 < r1 * 100 ? 2 : 1;
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

template <int kAcc>
static cudaError_t launch_prefill_kernel(const PrefillParams& p, int grid, cudaStream_t st) {
  // set on every launch (cheap): no per-device cache shared between threads
  const cudaError_t e = cudaFuncSetAttribute(prefill_q4k_kernel<kAcc>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(PfCfg<kAcc>::kSmem));
  if (e != cudaSuccess) return e;
  return launch_pdl_pf(prefill_q4k_kernel<kAcc>, grid, kPfThreads, PfCfg<kAcc>::kSmem, st, p);
}

cudaError_t launch_prefill_q4k(const uint8_t* W, const float* X, float* Y, int64_t rows,
                               int64_t K, int64_t N, uint8_t* ws, cudaStream_t st) {
  const int acc = prefill_acc(rows, N, device_sms());
  const int64_t t1 = token_tiles(N);
  const int n_tiles_n = static_cast<int>(acc == 2 ? (t1 + 1) / 2 * 2 : t1);
  const int n_tiles_m = static_cast<int>((rows + kPfM - 1) / kPfM);
  const int64_t pack_total = static_cast<int64_t>(n_tiles_n) * kPfN * (K / 8);
  const int64_t pack_blocks = std::min<int64_t>((pack_total + 255) / 256, 8 * device_sms());
  cudaError_t e = launch_pdl_pf(prefill_pack_x_kernel, static_cast<int>(pack_blocks), 256, 0, st,
                                X, ws, N, K, n_tiles_n);
  if (e != cudaSuccess) return e;
  PrefillParams p;
  if (!encode_w_map(&p.wmap, W, rows, K)) return cudaErrorInvalidValue;
  p.W = W;
  p.X16 = ws;
  p.Y = Y;
  p.rows = rows;
  p.K = K;
  p.N = N;
  p.KC = static_cast<int>(K / kPfK);
  p.n_tiles_n = n_tiles_n;
  const int grid = n_tiles_m * (n_tiles_n / acc);
  return acc == 2 ? launch_prefill_kernel<2>(p, grid, st) : launch_prefill_kernel<1>(p, grid, st);
}

unsigned read_clear_prefill_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_prefill, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_prefill, &z, sizeof(z));
  return v;
}

}  // namespace qws
