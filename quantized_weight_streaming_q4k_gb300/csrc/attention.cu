// attention.cu -- decode-time attention over a KV cache (sequence length > 1):
// rope_at_pos, kv_append and kv_attention (infer-compute README §Shaders rows
// "RoPE" and "Attention": rope_at_pos, kv_append, kv_attention with GQA and
// softcap; infer-inference README §BLAS-Fused Attention: scores, scale and
// optional softcap, softmax, weighted sum of values).
//
// kv_attention is bound by reading the caches (2 * n_kv * n_ctx * head_dim
// floats), so it is split along the positions (flash-decoding style):
//   * kernel 1, grid (splits, n_kv): CTA (j, g) owns the blocks of P
//     positions b = j, j + splits, ... of kv head g (so the CTAs of a head
//     sweep its cache side by side) and every query head of g's group.  A
//     copy warp streams each block's k rows and v rows into a shared-memory
//     ring (1-D TMA bulk copies); warp w takes rows w, w + 8, ... of a
//     block; lane L holds
//     columns [L*hd/32, (L+1)*hd/32) of q, k, v and of the running output, so
//     a warp reads each k and v row as one coalesced run.  Per position: the
//     group's scores by warp-shuffle sums, optional softcap, then the online
//     softmax update (running max m, sum l, output acc).  The 16 warps are
//     merged in shared memory in a fixed order and the CTA writes its
//     (m, l, acc) partial to the workspace.
//   * kernel 2, one CTA per query head and 32 columns: merges the splits
//     (eight interleaved partial sums per column, added in a fixed order):
//     out = sum_j e^(m_j - M) acc_j / sum_j e^(m_j - M) l_j.
// Everything is in a fixed order, so results are identical run to run.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "launch.h"

namespace qws {

__device__ unsigned g_err_attention;

constexpr int kAttWarps = 16;                   // consumer warps
constexpr int kAttThreads = 32 + kAttWarps * 32;  // + one copy warp
constexpr int kAttStages = 3;
constexpr uint32_t kAttStageBytes = 64 * 1024;  // P k rows + P v rows, P = 8192 / head_dim

// ------------------------------------------------------------------ rope
// (x_i, x_{i+r/2}) rotated by theta_i = pos * base^(-2i/r), i < r/2, every head;
// the angle and its sine / cosine in f64 (computed once per launch on the
// host: FP64 arithmetic on this GPU is slow), the rotation in f64, rounded
// once.
constexpr int kMaxRotDim = 512;
struct RopeTable {
  double c[kMaxRotDim / 2], s[kMaxRotDim / 2];   // cos / sin of pos * base^(-2i / rot_dim)
};

static RopeTable rope_table(int rot_dim, int64_t pos, double base) {
  RopeTable tab;
  for (int i = 0; i < rot_dim / 2; ++i) {
    const double theta = static_cast<double>(pos) * std::pow(base, -2.0 * i / rot_dim);
    tab.c[i] = std::cos(theta);
    tab.s[i] = std::sin(theta);
  }
  return tab;
}

void rope_table_f32(int rot_dim, int64_t pos, double base, float* c, float* s) {
  const RopeTable tab = rope_table(rot_dim, pos, base);
  for (int i = 0; i < rot_dim / 2; ++i) {
    c[i] = static_cast<float>(tab.c[i]);
    s[i] = static_cast<float>(tab.s[i]);
  }
}

__global__ void rope_kernel(float* __restrict__ x, int n_heads, int head_dim, int rot_dim,
                            const __grid_constant__ RopeTable tab) {
  pdl_launch_dependents();
  pdl_wait();
  const int half = rot_dim / 2;
  const int64_t n = static_cast<int64_t>(n_heads) * half;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int h = static_cast<int>(t / half);
    const int i = static_cast<int>(t - static_cast<int64_t>(h) * half);
    const double s = tab.s[i], c = tab.c[i];
    float* xh = x + static_cast<int64_t>(h) * head_dim;
    const double a = xh[i], b = xh[i + half];
    xh[i] = static_cast<float>(a * c - b * s);
    xh[i + half] = static_cast<float>(a * s + b * c);
  }
}

// ------------------------------------------------------------------ kv_append
__global__ void kv_append_kernel(float* __restrict__ kc, float* __restrict__ vc,
                                 const float* __restrict__ k, const float* __restrict__ v,
                                 int n_kv, int head_dim, int64_t max_seq, int64_t pos) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t n = static_cast<int64_t>(n_kv) * head_dim;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t g = t / head_dim, i = t - g * head_dim;
    const int64_t dst = (g * max_seq + pos) * head_dim + i;
    kc[dst] = k[t];
    vc[dst] = v[t];
  }
}

// ------------------------------------------------------------------ kv_attention
struct AttParams {
  const float* q;      // [n_q][hd]
  const float* kc;     // [n_kv][max_seq][hd]
  const float* vc;
  float* part;         // [n_kv][splits][group][hd + 2]: acc..., m, l
  float* out;          // [n_q][hd]
  unsigned long long* out_words;   // or, when set: {value, stamp} words [n_q][hd]
  unsigned stamp;
  int n_q, n_kv, hd, group, splits;
  int64_t max_seq, n_ctx;
  float scale, softcap;
  // RoPE and append fused in (the decode step on the chain kernel), when qw
  // is set: q comes as {value, stamp} words, rotated at pos here; k and v of
  // position pos come as words too: the CTA whose split holds pos rotates k,
  // writes k and v into the caches (kc_w, vc_w) and uses them for that row
  // in place of the cache row its copy warp loaded.
  // The rotation here is in f32 (FP64 arithmetic on this GPU is slow
  // enough that the f64 rotation of rope_kernel tripled the split's time):
  // cosine and sine of the f64 angle rounded to f32, then a * c - b * s by
  // one product and one FMA, a few units of 2^-24 relative to |a| + |b|.
  const unsigned long long *qw, *kw, *vw;
  float *kc_w, *vc_w;
  int64_t pos;
  int rot_dim;
  float tc[kMaxRotDim / 2], ts[kMaxRotDim / 2];
};

// Element i of a head of words x rotated at pos (f32; see AttParams).
__device__ __forceinline__ float rope_word(const unsigned long long* x, int i, int rot_dim,
                                           const float* tc, const float* ts) {
  auto val = [](unsigned long long w) { return __uint_as_float(static_cast<unsigned>(w)); };
  if (i >= rot_dim) return val(x[i]);
  const int half = rot_dim / 2;
  const int j = i < half ? i : i - half;
  const float a = val(x[j]), b = val(x[j + half]);
  return i < half ? fmaf(a, tc[j], -(b * ts[j])) : fmaf(a, ts[j], b * tc[j]);
}

template <int kPL, int kG>   // columns per lane = hd / 32; query heads per kv head
__global__ void __launch_bounds__(kAttThreads, 1) kv_attention_split_kernel(
    const __grid_constant__ AttParams p) {
  __shared__ float sm_m[kAttWarps][kG], sm_l[kAttWarps][kG];
  // fused mode: the group's rotated q, and k (rotated) and v of position pos
  __shared__ float sq[kG][kPL * 32], skv[2][kPL * 32];
  __shared__ __align__(8) uint64_t full[kAttStages], empty[kAttStages];
  extern __shared__ __align__(128) uint8_t att_ring[];   // kAttStages x kAttStageBytes
  const int warp = static_cast<int>(threadIdx.x >> 5) - 1;   // -1: the copy warp
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x, g = blockIdx.y;
  constexpr int G = kG;
  constexpr int P = kAttStageBytes / (2 * kPL * 32 * 4);     // positions per stage
  // blocks of P positions are dealt to the splits in turn (block b to split
  // b % splits), so that the CTAs of one kv head sweep its cache together
  const int64_t n_blocks = (p.n_ctx + P - 1) / P;
  const int n_stages =
      j < n_blocks ? static_cast<int>((n_blocks - j + p.splits - 1) / p.splits) : 0;
  const size_t row = static_cast<size_t>(kPL) * 32 * 4;      // bytes of one k or v row
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAttWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  if (warp < 0) {
    // ---- copy warp: per stage, P consecutive k rows then P v rows (16 B aligned)
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int64_t head0 = static_cast<int64_t>(g) * p.max_seq * p.hd;
      const uint8_t* kg = reinterpret_cast<const uint8_t*>(p.kc + head0);
      const uint8_t* vg = reinterpret_cast<const uint8_t*>(p.vc + head0);
      for (int st = 0; st < n_stages; ++st) {
        const int s = st % kAttStages;
        const uint32_t ph = static_cast<uint32_t>(st / kAttStages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u)) {
          atomicOr(&g_err_attention, kErrEmptyWait);
          break;
        }
        const int64_t ta = (j + static_cast<int64_t>(st) * p.splits) * P;
        const uint32_t rows = static_cast<uint32_t>(min(static_cast<int64_t>(P), p.n_ctx - ta));
        const uint32_t bytes = rows * static_cast<uint32_t>(row);
        uint8_t* dst = att_ring + static_cast<size_t>(s) * kAttStageBytes;
        mbar_arrive_expect_tx(&full[s], 2u * bytes);
        bulk_copy_g2s(dst, kg + ta * row, bytes, &full[s], pol);
        bulk_copy_g2s(dst + P * row, vg + ta * row, bytes, &full[s], pol);
      }
      // do not leave with copies into shared memory in flight
      const int first = n_stages > kAttStages ? n_stages - kAttStages : 0;
      for (int st = first; st < n_stages; ++st)
        if (!mbar_wait(&full[st % kAttStages], static_cast<uint32_t>(st / kAttStages) & 1u))
          atomicOr(&g_err_attention, kErrDrain);
    }
    return;
  }
  const int c0 = lane * kPL;
  const bool fused = p.qw != nullptr;
  // fused mode: does this CTA's share of the blocks hold position pos?
  const bool has_pos = fused && (p.pos / P) % p.splits == j;
  if (fused) {
    // every element by one consumer thread, so the loads of all of them are
    // in flight together; then the warps read their columns from shared memory
    const int ct = static_cast<int>(threadIdx.x) - 32;
    for (int e = ct; e < kG * p.hd; e += kAttWarps * 32) {
      const int h = e / p.hd, i = e - h * p.hd;
      sq[h][i] = rope_word(p.qw + static_cast<int64_t>(g * G + h) * p.hd, i, p.rot_dim, p.tc,
                           p.ts);
    }
    if (has_pos) {
      const int64_t row = (static_cast<int64_t>(g) * p.max_seq + p.pos) * p.hd;
      for (int i = ct; i < p.hd; i += kAttWarps * 32) {
        const float kr =
            rope_word(p.kw + static_cast<int64_t>(g) * p.hd, i, p.rot_dim, p.tc, p.ts);
        const float vr =
            __uint_as_float(static_cast<unsigned>(p.vw[static_cast<int64_t>(g) * p.hd + i]));
        skv[0][i] = kr;
        skv[1][i] = vr;
        p.kc_w[row + i] = kr;
        p.vc_w[row + i] = vr;
      }
    }
    bar_sync(1, kAttWarps * 32);
  }
  float q[kG][kPL], acc[kG][kPL], m[kG], l[kG];
#pragma unroll
  for (int h = 0; h < kG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
    const int64_t hq = static_cast<int64_t>(g * G + h);
#pragma unroll
    for (int c = 0; c < kPL; ++c) {
      const float qv = fused ? sq[h][c0 + c] : p.q[hq * p.hd + c0 + c];
      q[h][c] = qv * p.scale;
      acc[h][c] = 0.f;
    }
  }
  for (int st = 0; st < n_stages; ++st) {
    const int s = st % kAttStages;
    const uint32_t ph = static_cast<uint32_t>(st / kAttStages) & 1u;
    if (!mbar_wait(&full[s], ph)) {
      atomicOr(&g_err_attention, kErrFullWait);
      break;
    }
    const int64_t ta = (j + static_cast<int64_t>(st) * p.splits) * P;
    const int rows = static_cast<int>(min(static_cast<int64_t>(P), p.n_ctx - ta));
    const float* kst =
        reinterpret_cast<const float*>(att_ring + static_cast<size_t>(s) * kAttStageBytes);
    const float* vst = kst + P * kPL * 32;
    for (int r = warp; r < rows; r += kAttWarps) {
      float kr[kPL], vr[kPL];
      if (has_pos && ta + r == p.pos) {
#pragma unroll
        for (int c = 0; c < kPL; ++c) {
          kr[c] = skv[0][c0 + c];
          vr[c] = skv[1][c0 + c];
        }
      } else {
#pragma unroll
      for (int c = 0; c < kPL; c += (kPL % 4 == 0 ? 4 : 1)) {
        if constexpr (kPL % 4 == 0) {
          const float4 a = *reinterpret_cast<const float4*>(kst + r * kPL * 32 + c0 + c);
          const float4 b = *reinterpret_cast<const float4*>(vst + r * kPL * 32 + c0 + c);
          kr[c] = a.x; kr[c + 1] = a.y; kr[c + 2] = a.z; kr[c + 3] = a.w;
          vr[c] = b.x; vr[c + 1] = b.y; vr[c + 2] = b.z; vr[c + 3] = b.w;
        } else {
          kr[c] = kst[r * kPL * 32 + c0 + c];
          vr[c] = vst[r * kPL * 32 + c0 + c];
        }
      }
      }
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        float sc = 0.f;
#pragma unroll
        for (int c = 0; c < kPL; ++c) sc = fmaf(q[h][c], kr[c], sc);
        sc = warp_sum(sc);
        if (p.softcap > 0.f) sc = p.softcap * tanhf(sc / p.softcap);
        const float mn = fmaxf(m[h], sc);
        const float alpha = expf(m[h] - mn);
        const float pr = expf(sc - mn);
        l[h] = fmaf(l[h], alpha, pr);
#pragma unroll
        for (int c = 0; c < kPL; ++c) acc[h][c] = fmaf(acc[h][c], alpha, pr * vr[c]);
        m[h] = mn;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // merge the warps in order 0..15; the ring is free once every consumer is
  // past its last stage (every copy it waited for has landed), so the
  // warps' outputs are parked there
  bar_sync(1, kAttWarps * 32);
  float* sm_acc = reinterpret_cast<float*>(att_ring);      // [kAttWarps][kG][hd]
#pragma unroll
  for (int h = 0; h < kG; ++h) {
    if (lane == 0) {
      sm_m[warp][h] = m[h];
      sm_l[warp][h] = l[h];
    }
#pragma unroll
    for (int c = 0; c < kPL; ++c) sm_acc[(warp * kG + h) * p.hd + c0 + c] = acc[h][c];
  }
  bar_sync(1, kAttWarps * 32);
  const int ct = static_cast<int>(threadIdx.x) - 32;
  for (int e = ct; e < G * p.hd; e += kAttWarps * 32) {
    const int h = e / p.hd, i = e - h * p.hd;
    float M = -INFINITY;
    for (int w = 0; w < kAttWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float a = 0.f, L = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kAttWarps; ++w) {
        const float f = expf(sm_m[w][h] - M);   // 0 for an empty warp
        a = fmaf(sm_acc[(w * kG + h) * p.hd + i], f, a);
        L = fmaf(sm_l[w][h], f, L);
      }
    }
    float* dst = p.part + ((static_cast<int64_t>(g) * p.splits + j) * G + h) * (p.hd + 2);
    dst[i] = a;
    if (i == 0) {
      dst[p.hd] = M;
      dst[p.hd + 1] = L;
    }
  }
}

// Partials of at most kMaxSplits splits (kv_attention_splits never exceeds
// the grid of 152 CTAs).  Grid (n_q, ceil(hd / 32)), 256 threads: CTA
// (hq, y) merges columns 32 y .. 32 y + 31 of query head hq; thread (s, c)
// adds the splits j = s, s + 8, ... of column c (their loads all in flight
// at once), then the eight sums are added in order s = 0..7.
//   out = sum_j e^(m_j - M) acc_j / sum_j e^(m_j - M) l_j,  M = max_j m_j.
constexpr int kMaxSplits = 256;
constexpr int kMergeLanes = 8;   // split lanes per column

__global__ void __launch_bounds__(256)
    kv_attention_merge_kernel(const __grid_constant__ AttParams p) {
  __shared__ float sm[kMaxSplits], sl[kMaxSplits], sf[kMaxSplits];
  __shared__ float red[kMergeLanes][32];
  __shared__ float sL;
  pdl_launch_dependents();
  pdl_wait();
  const int hq = blockIdx.x;                 // query head
  const int g = hq / p.group, h = hq - g * p.group;
  const int64_t stride = static_cast<int64_t>(p.group) * (p.hd + 2);
  const float* base = p.part + (static_cast<int64_t>(g) * p.splits * p.group + h) * (p.hd + 2);
  for (int j = threadIdx.x; j < p.splits; j += blockDim.x) {
    sm[j] = base[j * stride + p.hd];
    sl[j] = base[j * stride + p.hd + 1];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int j = 0; j < p.splits; ++j) M = fmaxf(M, sm[j]);
    float L = 0.f;
    for (int j = 0; j < p.splits; ++j) {
      const float f = sm[j] != -INFINITY ? expf(sm[j] - M) : 0.f;   // 0: an empty split
      sf[j] = f;
      L = fmaf(sl[j], f, L);
    }
    sL = L;
  }
  __syncthreads();
  const int c = threadIdx.x & 31, sidx = threadIdx.x >> 5;
  const int i = blockIdx.y * 32 + c;
  float a = 0.f;
  if (i < p.hd) {
    int j = sidx;
    for (; j + 3 * kMergeLanes < p.splits; j += 4 * kMergeLanes) {
      const float a0 = base[j * stride + i];
      const float a1 = base[(j + kMergeLanes) * stride + i];
      const float a2 = base[(j + 2 * kMergeLanes) * stride + i];
      const float a3 = base[(j + 3 * kMergeLanes) * stride + i];
      a = fmaf(a0, sf[j], a);
      a = fmaf(a1, sf[j + kMergeLanes], a);
      a = fmaf(a2, sf[j + 2 * kMergeLanes], a);
      a = fmaf(a3, sf[j + 3 * kMergeLanes], a);
    }
    for (; j < p.splits; j += kMergeLanes) a = fmaf(base[j * stride + i], sf[j], a);
  }
  red[sidx][c] = a;
  __syncthreads();
  if (sidx == 0 && i < p.hd) {
    float t = 0.f;
    for (int s2 = 0; s2 < kMergeLanes; ++s2) t += red[s2][c];
    const float r = t / sL;
    if (p.out_words)
      p.out_words[static_cast<int64_t>(hq) * p.hd + i] =
          static_cast<unsigned long long>(__float_as_uint(r)) |
          (static_cast<unsigned long long>(p.stamp) << 32);
    else
      p.out[static_cast<int64_t>(hq) * p.hd + i] = r;
  }
}

// ------------------------------------------------------------------ host side
// One CTA per SM of a 152-SM GB300 in total (n_kv rows of splits), at least
// 32 positions (one ring stage) per split.  Decode over a KV cache at 1025
// positions (same box): 1577.5 us per token with at least 64 positions per
// split, 1557.2 with 32, 1562.6 with 16; long caches fill the grid anyway.
int kv_attention_splits(int n_kv, int64_t n_ctx) {
  const int64_t by_len = (n_ctx + 31) / 32;
  const int64_t by_grid = std::max(1, (152 + n_kv - 1) / n_kv);
  return static_cast<int>(std::max<int64_t>(1, std::min(by_len, by_grid)));
}

size_t kv_attention_workspace_bytes(int n_q, int n_kv, int head_dim, int64_t n_ctx) {
  if (n_kv <= 0 || n_q % n_kv) return 0;
  const int splits = kv_attention_splits(n_kv, n_ctx);
  return static_cast<size_t>(n_kv) * splits * (n_q / n_kv) * (head_dim + 2) * sizeof(float);
}

template <class... KArgs, class... Args>
static cudaError_t launch_pdl_att(void (*kernel)(KArgs...), dim3 grid, int threads, size_t smem,
                                  cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
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

cudaError_t launch_rope(float* x, int n_heads, int head_dim, int rot_dim, int64_t pos,
                        double base, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(n_heads) * (rot_dim / 2);
  const int blocks =
      static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 1024)));
  if (rot_dim > kMaxRotDim) return cudaErrorInvalidValue;
  return launch_pdl_att(rope_kernel, dim3(blocks), 256, 0, st, x, n_heads, head_dim, rot_dim,
                        rope_table(rot_dim, pos, base));
}

cudaError_t launch_kv_append(float* kc, float* vc, const float* k, const float* v, int n_kv,
                             int head_dim, int64_t max_seq, int64_t pos, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(n_kv) * head_dim;
  const int blocks =
      static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 1024)));
  return launch_pdl_att(kv_append_kernel, dim3(blocks), 256, 0, st, kc, vc, k, v, n_kv, head_dim,
                        max_seq, pos);
}

template <int kPL, int kG>
static cudaError_t launch_split(const AttParams& p, dim3 grid, cudaStream_t st) {
  // set on every launch (cheap): no per-device cache shared between threads
  const size_t smem = static_cast<size_t>(kAttStages) * kAttStageBytes;
  const cudaError_t e = cudaFuncSetAttribute(kv_attention_split_kernel<kPL, kG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl_att(kv_attention_split_kernel<kPL, kG>, grid, kAttThreads, smem, st, p);
}

cudaError_t launch_kv_attention(const float* q, const float* kc, const float* vc, float* out,
                                int n_q, int n_kv, int head_dim, int64_t max_seq, int64_t n_ctx,
                                float scale, float softcap, float* ws, cudaStream_t st,
                                unsigned long long* out_words, unsigned stamp,
                                const KvFuse* fuse) {
  AttParams p;
  p.qw = p.kw = p.vw = nullptr;
  p.kc_w = p.vc_w = nullptr;
  p.pos = 0;
  p.rot_dim = 0;
  if (fuse) {
    if (fuse->rot_dim > kMaxRotDim) return cudaErrorInvalidValue;
    p.qw = fuse->q;
    p.kw = fuse->k;
    p.vw = fuse->v;
    p.kc_w = fuse->kc;
    p.vc_w = fuse->vc;
    p.pos = fuse->pos;
    p.rot_dim = fuse->rot_dim;
    const RopeTable tab = rope_table(fuse->rot_dim, fuse->pos, fuse->base);
    for (int i = 0; i < fuse->rot_dim / 2; ++i) {
      p.tc[i] = static_cast<float>(tab.c[i]);
      p.ts[i] = static_cast<float>(tab.s[i]);
    }
  }
  p.q = q;
  p.kc = kc;
  p.vc = vc;
  p.part = ws;
  p.out = out;
  p.out_words = out_words;
  p.stamp = stamp;
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.hd = head_dim;
  p.group = n_q / n_kv;
  p.splits = kv_attention_splits(n_kv, n_ctx);
  p.max_seq = max_seq;
  p.n_ctx = n_ctx;
  p.scale = scale;
  p.softcap = softcap;
  const dim3 grid(p.splits, n_kv);
  cudaError_t e;
  switch ((head_dim / 32) * 8 + p.group) {
#define QWS_ATT_CASE(PL, G) \
  case PL * 8 + G: e = launch_split<PL, G>(p, grid, st); break;
    QWS_ATT_CASE(1, 1) QWS_ATT_CASE(1, 2) QWS_ATT_CASE(1, 3) QWS_ATT_CASE(1, 4)
    QWS_ATT_CASE(2, 1) QWS_ATT_CASE(2, 2) QWS_ATT_CASE(2, 3) QWS_ATT_CASE(2, 4)
    QWS_ATT_CASE(4, 1) QWS_ATT_CASE(4, 2) QWS_ATT_CASE(4, 3) QWS_ATT_CASE(4, 4)
    QWS_ATT_CASE(8, 1) QWS_ATT_CASE(8, 2) QWS_ATT_CASE(8, 3) QWS_ATT_CASE(8, 4)
#undef QWS_ATT_CASE
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_pdl_att(kv_attention_merge_kernel, dim3(n_q, (head_dim + 31) / 32), 256, 0, st,
                        p);
}

unsigned read_clear_attention_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_attention, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_attention, &z, sizeof(z));
  return v;
}

}  // namespace qws
