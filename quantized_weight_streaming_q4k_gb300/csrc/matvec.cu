// matvec.cu -- standalone streaming kernels: quantized matvec (any format,
// optional column split), fused QKV (three stacked segments), gate/up with the
// GEGLU epilogue, the split-K reduction, rms_norm and residual_add.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "launch.h"

namespace qws {

__device__ unsigned g_err_matvec;

struct MatvecParams {
  Phase P;                 // phase of column slice 0
  const float* x;          // [B][x_stride]
  int64_t x_stride;
  const uint8_t* xq;       // Q8_0 activations [B][xq_stride bytes] (kDirect units)
  int64_t xq_stride;
  int cps;                 // CTAs per column slice
  int64_t w_slice_off;     // byte offset between column slices within a row
  int64_t x_slice_off;     // column offset between slices
  int64_t y_slice_off;     // float offset between slices' partial outputs
  uint32_t S, stage_bytes, red_floats, xs_floats;
};

struct OnePhase {
  Phase P;
  __device__ __forceinline__ int count() const { return 1; }
  __device__ __forceinline__ Phase get(int) const { return P; }
};

template <class Unit, class Epi>
__global__ void __launch_bounds__(kRoleThreads + kMaxConsumers)
    matvec_kernel(const __grid_constant__ MatvecParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_launch_dependents();
  const Ring R = make_ring(smem, p.S, p.stage_bytes, p.red_floats, p.xs_floats);
  const int C = static_cast<int>(blockDim.x) - kRoleThreads;
  // this CTA's column slice
  const int slice = static_cast<int>(blockIdx.x) / p.cps;
  Phase P = p.P;
  P.cta0 = slice * p.cps;
  P.ncta = p.cps;
  if (slice > 0) {
    P.seg[0].W += slice * p.w_slice_off;
    P.seg[0].y += slice * p.y_slice_off;
  }
  if (threadIdx.x == 0) ring_init(R, C / 32);
  __syncthreads();
  RingPos pos;
  if (threadIdx.x < kProducerThreads) {
    // weights are never written by another kernel: stream them right away
    if (threadIdx.x == 0) run_producer(OnePhase{P}, R, &g_err_matvec);
  } else if (threadIdx.x < kRoleThreads) {
    pdl_wait();   // y may still be read by the previous kernel
    reduce_phase(P, R, pos, Epi{}, &g_err_matvec);
  } else {
    pdl_wait();   // x may come from the previous kernel
    const int ctid = static_cast<int>(threadIdx.x) - kRoleThreads;
    if constexpr (Unit::kDirect)
      consume_phase<Unit>(P, R, pos, XOfQ8{p.xq, p.xq_stride}, ctid, C, &g_err_matvec);
    else
      consume_phase<Unit>(P, R, pos, XOfPlain{p.x + slice * p.x_slice_off, p.x_stride}, ctid, C,
                          &g_err_matvec);
  }
}

// quantize_q8: one warp per 32-value block.  amax by a warp max over the
// bit patterns of |x| (order-preserving for non-negative floats); every
// decision in f32 with explicitly rounded operations: d = amax / 127,
// id = 1 / d (0 when d = 0), q = round-half-away(x * id); d is stored as
// binary16 (round to nearest even).  x must be finite; xq must be 2-byte
// aligned (blocks are written as halfwords).
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float* __restrict__ x,
                                                            uint8_t* __restrict__ xq,
                                                            int64_t nblocks) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t wpb = blockDim.x >> 5;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * wpb;
  for (int64_t k = blockIdx.x * wpb + (threadIdx.x >> 5); k < nblocks; k += nw) {
    const float v = x[k * 32 + lane];
    const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v))));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    const int q = static_cast<int>(roundf(__fmul_rn(v, id)));
    // the block is 2-byte aligned: 17 halfwords, d then 16 code pairs
    const unsigned qb = static_cast<unsigned>(q) & 0xFFu;
    const unsigned next = __shfl_down_sync(0xFFFFFFFFu, qb, 1);
    unsigned short* blk = reinterpret_cast<unsigned short*>(xq + k * 34);
    if ((lane & 1) == 0) blk[1 + (lane >> 1)] = static_cast<unsigned short>(qb | (next << 8));
    if (lane == 0) blk[0] = __half_as_ushort(__float2half_rn(d));
  }
}

__global__ void splitk_reduce_kernel(const float* __restrict__ part, float* __restrict__ y,
                                     int64_t n, int splits) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float acc = part[i];
    for (int s = 1; s < splits; ++s) acc += part[s * n + i];
    y[i] = acc;
  }
}

// One CTA per vector; sum of squares in a fixed order (per-thread strided
// partials, then a fixed shuffle tree and a fixed pass over the warp sums).
__global__ void __launch_bounds__(1024) rms_norm_kernel(const float* __restrict__ x,
                                                        const float* __restrict__ w,
                                                        float* __restrict__ y, int64_t n,
                                                        float eps) {
  __shared__ float wsum[32];
  __shared__ float inv_s;
  pdl_launch_dependents();
  pdl_wait();
  const float* xb = x + blockIdx.x * n;
  float* yb = y + blockIdx.x * n;
  float ss = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(xb[i], xb[i], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += wsum[i];
    inv_s = 1.0f / sqrtf(t / static_cast<float>(n) + eps);
  }
  __syncthreads();
  const float inv = inv_s;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) yb[i] = xb[i] * inv * w[i];
}

// residual_norm: h <- h + y, then x = h / sqrt(mean(h^2) + eps) * w, one CTA
// per vector, same fixed-order reduction as rms_norm_kernel.
__global__ void __launch_bounds__(1024) residual_rms_norm_kernel(float* __restrict__ h,
                                                                 const float* __restrict__ y,
                                                                 const float* __restrict__ w,
                                                                 float* __restrict__ x, int64_t n,
                                                                 float eps) {
  __shared__ float wsum[32];
  __shared__ float inv_s;
  pdl_launch_dependents();
  pdl_wait();
  float* hb = h + blockIdx.x * n;
  const float* yb = y + blockIdx.x * n;
  float* xb = x + blockIdx.x * n;
  float ss = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const float r = hb[i] + yb[i];
    hb[i] = r;
    ss = fmaf(r, r, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += wsum[i];
    inv_s = 1.0f / sqrtf(t / static_cast<float>(n) + eps);
  }
  __syncthreads();
  const float inv = inv_s;
  // each thread reads back the h values it wrote itself
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) xb[i] = hb[i] * inv * w[i];
}

// rms_norm_q8 / residual_norm_q8: the norm of rms_norm_kernel (or of
// residual_rms_norm_kernel, with h <- h + y first) and, in the same launch,
// its output quantized to Q8_0 blocks exactly as quantize_q8_0_kernel does,
// one warp per block.  The normalized vector itself is not stored.
template <bool kResidual>
__global__ void __launch_bounds__(1024) norm_q8_kernel(float* __restrict__ h,
                                                       const float* __restrict__ y,
                                                       const float* __restrict__ w,
                                                       uint8_t* __restrict__ xq, int64_t n,
                                                       float eps) {
  __shared__ float wsum[32];
  __shared__ float inv_s;
  pdl_launch_dependents();
  pdl_wait();
  float* hb = h + blockIdx.x * n;
  const float* yb = kResidual ? y + blockIdx.x * n : nullptr;
  float ss = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    float r = hb[i];
    if constexpr (kResidual) {
      r = r + yb[i];
      hb[i] = r;
    }
    ss = fmaf(r, r, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();   // also makes the h written above visible to the block
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += wsum[i];
    inv_s = 1.0f / sqrtf(t / static_cast<float>(n) + eps);
  }
  __syncthreads();
  const float inv = inv_s;
  const int lane = threadIdx.x & 31;
  const int64_t nblk = n / 32;
  uint8_t* xqb = xq + blockIdx.x * (nblk * 34);
  for (int64_t k = threadIdx.x >> 5; k < nblk; k += blockDim.x >> 5) {
    const int64_t i = k * 32 + lane;
    const float v = hb[i] * inv * w[i];
    const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v))));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    const int q = static_cast<int>(roundf(__fmul_rn(v, id)));
    const unsigned qb = static_cast<unsigned>(q) & 0xFFu;
    const unsigned next = __shfl_down_sync(0xFFFFFFFFu, qb, 1);
    unsigned short* blk = reinterpret_cast<unsigned short*>(xqb + k * 34);
    if ((lane & 1) == 0) blk[1 + (lane >> 1)] = static_cast<unsigned short>(qb | (next << 8));
    if (lane == 0) blk[0] = __half_as_ushort(__float2half_rn(d));
  }
}

__global__ void residual_add_kernel(float* __restrict__ h, const float* __restrict__ y,
                                    int64_t n) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    h[i] += y[i];
}

// Self-test of the failure path: the engine's bounded mbarrier wait on a
// barrier that nothing ever arrives at (no copy is issued), with the given
// wait limit.  The wait gives up, records kErrFullWait and the kernel
// returns; nothing is in flight.
__global__ void selftest_mbar_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, limit)) atomicOr(&g_err_matvec, kErrFullWait);
  __syncthreads();
}

cudaError_t launch_selftest_mbar(long long limit, cudaStream_t st) {
  selftest_mbar_kernel<<<1, 32, 0, st>>>(limit);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host side
// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes (see pdl_wait / pdl_launch_dependents).
template <class... KArgs, class... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int threads, size_t smem,
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

int device_sms() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  sms = sms > 0 ? sms : 1;
  if (dev >= 0 && dev < 64) cache[dev] = sms;
  return sms;
}

// Per (device, kernel, threads, smem): the dynamic-smem opt-in is set once and
// the occupancy is queried once.
struct KernelCacheEntry {
  int dev;
  const void* fn;
  int threads;
  size_t smem;
  int bps;
};

static int cached_blocks_per_sm(const void* fn, int threads, size_t smem) {
  static std::mutex mu;
  static KernelCacheEntry entries[256];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (entries[i].dev == dev && entries[i].fn == fn && entries[i].threads == threads &&
        entries[i].smem == smem)
      return entries[i].bps;
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  int bps = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, fn, threads, smem) != cudaSuccess)
    bps = 0;
  if (bps < 1) bps = 1;
  if (n < 256) entries[n++] = KernelCacheEntry{dev, fn, threads, smem, bps};
  return bps;
}

template <class Unit, class Epi>
static int blocks_per_sm(int threads, size_t smem) {
  return cached_blocks_per_sm(reinterpret_cast<const void*>(matvec_kernel<Unit, Epi>), threads,
                              smem);
}

template <class Unit, class Epi>
static cudaError_t launch_one(const MatvecParams& p, int threads, size_t smem, int grid,
                              cudaStream_t st) {
  blocks_per_sm<Unit, Epi>(threads, smem);  // makes sure the smem opt-in is set
  return launch_pdl(matvec_kernel<Unit, Epi>, grid, threads, smem, st, p);
}

// Tile plan, ring depth and parameters of one streaming launch (without the
// activation pointers and the CTA split, which depend on the kernel).
static bool plan_matvec(int fmt, int epi, const Seg* segs, int nseg, const uint8_t* W2,
                        int64_t K, int B, int splits, bool staged, MatvecParams& p,
                        int& threads, size_t& smem, std::string* why) {
  const int sms = device_sms();
  const int64_t Ks = K / splits;
  int64_t rows_total = 0;
  for (int i = 0; i < nseg; ++i) rows_total += segs[i].rows;
  TilePlan tp;
  std::string reason;
  // the 8-bit path (units reading their own activations) keeps 46 KB tiles:
  // it streams at the HBM rate already, and 64 KB measured 58.7 against 56.6
  // us for the 262144 x 2560 lm_head
  const uint32_t target = staged ? kTileTarget : 46u * 1024u;
  if (!plan_tiles(fmt, epi, Ks, B, rows_total * splits, sms, target, tp, reason)) {
    if (why) *why = reason;
    return false;
  }
  p = MatvecParams{};
  Phase& P = p.P;
  P.fmt = fmt;
  P.epi = epi;
  P.nseg = nseg;
  P.n_tiles = 0;
  for (int i = 0; i < nseg; ++i) {
    P.seg[i] = segs[i];
    P.seg[i].tiles = static_cast<int>((segs[i].rows + tp.T - 1) / tp.T);
    P.n_tiles += P.seg[i].tiles;
  }
  P.W2 = W2;
  P.K = Ks;
  P.row_bytes = row_bytes_of(fmt, Ks);
  P.row_stride = row_bytes_of(fmt, K);
  P.B = B;
  P.U = tp.U;
  P.G = tp.G;
  P.T = tp.T;
  P.T2 = tp.T;
  P.n1 = 0x7FFFFFFF;   // one tile size
  p.w_slice_off = P.row_bytes;
  p.x_slice_off = Ks;
  p.y_slice_off = static_cast<int64_t>(B) * segs[0].rows;
  p.stage_bytes = round_up(tp.stage_need + 16, 128);
  p.red_floats = tp.red_floats;
  p.xs_floats = staged ? static_cast<uint32_t>(unit_weights(fmt) * red_stride(tp.U)) : 0u;
  // ring: as deep as the shared-memory budget allows (one CTA per SM), 2..16
  p.S = 16;
  while (p.S > 2 && ring_smem_bytes(p.S, p.stage_bytes, p.red_floats, p.xs_floats) > kSmemBudget)
    --p.S;
  smem = ring_smem_bytes(p.S, p.stage_bytes, p.red_floats, p.xs_floats);
  threads = kRoleThreads + tp.C;
  return true;
}

// CTAs per column slice: enough to cover the slice's tiles, and all slices
// together about fill the device (bps CTAs per SM).
static int split_grid(MatvecParams& p, int bps, int splits) {
  const int64_t slots = static_cast<int64_t>(bps) * device_sms();
  int64_t cps = std::max<int64_t>(1, slots / splits);
  cps = std::min<int64_t>(cps, p.P.n_tiles);
  p.cps = static_cast<int>(cps);
  p.P.cta0 = 0;
  p.P.ncta = p.cps;
  return static_cast<int>(cps * splits);
}

cudaError_t launch_matvec(int fmt, int epi, const Seg* segs, int nseg, const uint8_t* W2,
                          const float* x, int64_t K, int B, int splits, cudaStream_t st,
                          std::string* why) {
  MatvecParams p;
  int threads = 0;
  size_t smem = 0;
  if (!plan_matvec(fmt, epi, segs, nseg, W2, K, B, splits, true, p, threads, smem, why))
    return cudaErrorInvalidValue;
  p.x = x;
  p.x_stride = K;
  int bps = 1;
  switch (fmt * 4 + epi) {
    case 12 * 4 + EPI_STORE: bps = blocks_per_sm<UnitQ4K, EpiStore>(threads, smem); break;
    case 12 * 4 + EPI_GEGLU: bps = blocks_per_sm<UnitQ4K, EpiGeglu>(threads, smem); break;
    case 12 * 4 + EPI_SWIGLU: bps = blocks_per_sm<UnitQ4K, EpiSwiglu>(threads, smem); break;
    case 14 * 4 + EPI_STORE: bps = blocks_per_sm<UnitQ6K, EpiStore>(threads, smem); break;
    case 2 * 4 + EPI_STORE: bps = blocks_per_sm<UnitQ40, EpiStore>(threads, smem); break;
    default:
      if (why) *why = "unsupported format / epilogue";
      return cudaErrorInvalidValue;
  }
  const int grid = split_grid(p, bps, splits);
  switch (fmt * 4 + epi) {
    case 12 * 4 + EPI_STORE: return launch_one<UnitQ4K, EpiStore>(p, threads, smem, grid, st);
    case 12 * 4 + EPI_GEGLU: return launch_one<UnitQ4K, EpiGeglu>(p, threads, smem, grid, st);
    case 12 * 4 + EPI_SWIGLU: return launch_one<UnitQ4K, EpiSwiglu>(p, threads, smem, grid, st);
    case 14 * 4 + EPI_STORE: return launch_one<UnitQ6K, EpiStore>(p, threads, smem, grid, st);
    default: return launch_one<UnitQ40, EpiStore>(p, threads, smem, grid, st);
  }
}

cudaError_t launch_matvec_q8(int wfmt, const Seg* segs, int nseg, const uint8_t* xq, int64_t K,
                             int B, cudaStream_t st, std::string* why) {
  MatvecParams p;
  int threads = 0;
  size_t smem = 0;
  if (!plan_matvec(wfmt, EPI_STORE, segs, nseg, nullptr, K, B, 1, false, p, threads, smem, why))
    return cudaErrorInvalidValue;
  p.xq = xq;
  p.xq_stride = K / 32 * 34;
  if (wfmt == 2) {
    const int grid = split_grid(p, blocks_per_sm<UnitQ40xQ8, EpiStore>(threads, smem), 1);
    return launch_one<UnitQ40xQ8, EpiStore>(p, threads, smem, grid, st);
  }
  if (wfmt == 8) {
    const int grid = split_grid(p, blocks_per_sm<UnitQ80xQ8, EpiStore>(threads, smem), 1);
    return launch_one<UnitQ80xQ8, EpiStore>(p, threads, smem, grid, st);
  }
  if (why) *why = "weights must be Q4_0 or Q8_0";
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_q8_0(const float* x, uint8_t* xq, int64_t nblocks, cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((nblocks + 7) / 8, 8 * device_sms());
  return launch_pdl(quantize_q8_0_kernel, static_cast<int>(std::max<int64_t>(blocks, 1)),
                    threads, 0, st, x, xq, nblocks);
}

cudaError_t launch_splitk_reduce(const float* part, float* y, int64_t n, int splits,
                                 cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((n + threads - 1) / threads, 4 * device_sms());
  return launch_pdl(splitk_reduce_kernel, static_cast<int>(std::max<int64_t>(blocks, 1)), threads,
                    0, st, part, y, n, splits);
}

cudaError_t launch_rms_norm(const float* x, const float* w, float* y, int64_t n, float eps,
                            int batch, cudaStream_t st) {
  const int threads = n >= 1024 ? 1024 : static_cast<int>((n + 31) / 32 * 32);
  return launch_pdl(rms_norm_kernel, batch, threads, 0, st, x, w, y, n, eps);
}

cudaError_t launch_residual_rms_norm(float* h, const float* y, const float* w, float* x,
                                    int64_t n, float eps, int batch, cudaStream_t st) {
  const int threads = n >= 1024 ? 1024 : static_cast<int>((n + 31) / 32 * 32);
  return launch_pdl(residual_rms_norm_kernel, batch, threads, 0, st, h, y, w, x, n, eps);
}

cudaError_t launch_norm_q8(float* h, const float* y, const float* w, uint8_t* xq, int64_t n,
                           float eps, int batch, bool residual, cudaStream_t st) {
  const int threads = n >= 1024 ? 1024 : static_cast<int>((n + 31) / 32 * 32);
  return residual ? launch_pdl(norm_q8_kernel<true>, batch, threads, 0, st, h, y, w, xq, n, eps)
                  : launch_pdl(norm_q8_kernel<false>, batch, threads, 0, st, h, y, w, xq, n, eps);
}

cudaError_t launch_residual_add(float* h, const float* y, int64_t n, int batch,
                                cudaStream_t st) {
  const int64_t total = n * batch;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, 4 * device_sms());
  return launch_pdl(residual_add_kernel, static_cast<int>(std::max<int64_t>(blocks, 1)), threads,
                    0, st, h, y, total);
}

unsigned read_clear_matvec_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_matvec, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_matvec, &z, sizeof(z));
  return v;
}

}  // namespace qws
