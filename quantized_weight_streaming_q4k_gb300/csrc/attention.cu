// attention.cu -- decode-time attention over a KV cache (sequence length > 1):
// rope_at_pos, kv_append and kv_attention (infer-compute README §Shaders rows
// "RoPE" and "Attention": rope_at_pos, kv_append, kv_attention with GQA and
// softcap; infer-inference README §BLAS-Fused Attention: scores, scale and
// optional softcap, softmax, weighted sum of values).
//
// kv_attention is bound by reading the caches (2 * n_kv * n_ctx * head_dim
// floats), so it is split along the positions (flash-decoding style):
//   * kernel 1, grid (splits, n_kv): CTA (j, g) owns positions
//     [j * chunk, (j + 1) * chunk) of kv head g and every query head of g's
//     group.  Warp w takes positions j*chunk + w, + 8, ...; lane L holds
//     columns [L*hd/32, (L+1)*hd/32) of q, k, v and of the running output, so
//     a warp reads each k and v row as one coalesced run.  Per position: the
//     group's scores by warp-shuffle sums, optional softcap, then the online
//     softmax update (running max m, sum l, output acc).  The 8 warps are
//     merged in shared memory in a fixed order and the CTA writes its
//     (m, l, acc) partial to the workspace.
//   * kernel 2, one CTA per query head: merges the splits in order:
//     out = sum_j e^(m_j - M) acc_j / sum_j e^(m_j - M) l_j.
// Everything is in a fixed order, so results are identical run to run.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "launch.h"

namespace qws {

constexpr int kAttWarps = 8;
constexpr int kAttMaxGroup = 4;     // query heads per kv head
constexpr int kAttMaxPerLane = 8;   // head_dim / 32

// ------------------------------------------------------------------ rope
// (x_i, x_{i+r/2}) rotated by theta_i = pos * base^(-2i/r), i < r/2, every head;
// the angle and its sine / cosine in f64, the rotation in f64, rounded once.
__global__ void rope_kernel(float* __restrict__ x, int n_heads, int head_dim, int rot_dim,
                            int64_t pos, double base) {
  pdl_launch_dependents();
  pdl_wait();
  const int half = rot_dim / 2;
  const int64_t n = static_cast<int64_t>(n_heads) * half;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int h = static_cast<int>(t / half);
    const int i = static_cast<int>(t - static_cast<int64_t>(h) * half);
    const double theta =
        static_cast<double>(pos) * pow(base, -2.0 * static_cast<double>(i) / rot_dim);
    double s, c;
    sincos(theta, &s, &c);
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
  int n_q, n_kv, hd, group, splits;
  int64_t max_seq, n_ctx, chunk;
  float scale, softcap;
};

// kPL consecutive floats of a k row and of a v row (16-byte loads when kPL
// is a multiple of 4; the rows start on 16-byte boundaries then)
template <int kPL>
__device__ __forceinline__ void load_row(const float* k, const float* v, float (&kr)[kPL],
                                         float (&vr)[kPL]) {
  if constexpr (kPL % 4 == 0) {
#pragma unroll
    for (int c = 0; c < kPL; c += 4) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(k + c));
      const float4 b = __ldg(reinterpret_cast<const float4*>(v + c));
      kr[c] = a.x; kr[c + 1] = a.y; kr[c + 2] = a.z; kr[c + 3] = a.w;
      vr[c] = b.x; vr[c + 1] = b.y; vr[c + 2] = b.z; vr[c + 3] = b.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < kPL; ++c) {
      kr[c] = __ldg(k + c);
      vr[c] = __ldg(v + c);
    }
  }
}

template <int kPL>   // columns per lane = hd / 32
__global__ void __launch_bounds__(kAttWarps * 32) kv_attention_split_kernel(
    const __grid_constant__ AttParams p) {
  __shared__ float sm_m[kAttWarps][kAttMaxGroup], sm_l[kAttWarps][kAttMaxGroup];
  __shared__ float sm_acc[kAttWarps][kAttMaxGroup][kAttMaxPerLane * 32];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x, g = blockIdx.y;
  const int G = p.group;
  const int64_t t0 = static_cast<int64_t>(j) * p.chunk;
  const int64_t t1 = min(t0 + p.chunk, p.n_ctx);
  const float* kg = p.kc + static_cast<int64_t>(g) * p.max_seq * p.hd;
  const float* vg = p.vc + static_cast<int64_t>(g) * p.max_seq * p.hd;
  const int c0 = lane * kPL;

  float q[kAttMaxGroup][kPL], acc[kAttMaxGroup][kPL], m[kAttMaxGroup], l[kAttMaxGroup];
#pragma unroll
  for (int h = 0; h < kAttMaxGroup; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int c = 0; c < kPL; ++c) {
      q[h][c] = h < G ? p.q[static_cast<int64_t>(g * G + h) * p.hd + c0 + c] * p.scale : 0.f;
      acc[h][c] = 0.f;
    }
  }
  // the next position's k and v rows are loaded while this one is used
  float kn[kPL], vn[kPL];
  int64_t t = t0 + warp;
  if (t < t1) load_row<kPL>(kg + t * p.hd + c0, vg + t * p.hd + c0, kn, vn);
  for (; t < t1; t += kAttWarps) {
    float kr[kPL], vr[kPL];
#pragma unroll
    for (int c = 0; c < kPL; ++c) {
      kr[c] = kn[c];
      vr[c] = vn[c];
    }
    if (t + kAttWarps < t1)
      load_row<kPL>(kg + (t + kAttWarps) * p.hd + c0, vg + (t + kAttWarps) * p.hd + c0, kn, vn);
#pragma unroll
    for (int h = 0; h < kAttMaxGroup; ++h) {
      if (h >= G) break;
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < kPL; ++c) s = fmaf(q[h][c], kr[c], s);
      s = warp_sum(s);
      if (p.softcap > 0.f) s = p.softcap * tanhf(s / p.softcap);
      const float mn = fmaxf(m[h], s);
      const float alpha = expf(m[h] - mn);   // 0 on the first position (m = -inf)
      const float pr = expf(s - mn);
      l[h] = fmaf(l[h], alpha, pr);
#pragma unroll
      for (int c = 0; c < kPL; ++c) acc[h][c] = fmaf(acc[h][c], alpha, pr * vr[c]);
      m[h] = mn;
    }
  }
  // merge the warps in order 0..7
#pragma unroll
  for (int h = 0; h < kAttMaxGroup; ++h) {
    if (h >= G) break;
    if (lane == 0) {
      sm_m[warp][h] = m[h];
      sm_l[warp][h] = l[h];
    }
#pragma unroll
    for (int c = 0; c < kPL; ++c) sm_acc[warp][h][c0 + c] = acc[h][c];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * p.hd; e += blockDim.x) {
    const int h = e / p.hd, i = e - h * p.hd;
    float M = -INFINITY;
    for (int w = 0; w < kAttWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float a = 0.f, L = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kAttWarps; ++w) {
        const float f = expf(sm_m[w][h] - M);   // 0 for an empty warp
        a = fmaf(sm_acc[w][h][i], f, a);
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

__global__ void kv_attention_merge_kernel(const __grid_constant__ AttParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int hq = blockIdx.x;                 // query head
  const int g = hq / p.group, h = hq - g * p.group;
  const int64_t stride = static_cast<int64_t>(p.group) * (p.hd + 2);
  const float* base = p.part + (static_cast<int64_t>(g) * p.splits * p.group + h) * (p.hd + 2);
  float M = -INFINITY;
  for (int j = 0; j < p.splits; ++j) M = fmaxf(M, base[j * stride + p.hd]);
  float L = 0.f;
  for (int j = 0; j < p.splits; ++j) {
    const float mj = base[j * stride + p.hd];
    if (mj != -INFINITY) L = fmaf(base[j * stride + p.hd + 1], expf(mj - M), L);
  }
  for (int i = threadIdx.x; i < p.hd; i += blockDim.x) {
    float a = 0.f;
    for (int j = 0; j < p.splits; ++j) {
      const float mj = base[j * stride + p.hd];
      if (mj != -INFINITY) a = fmaf(base[j * stride + i], expf(mj - M), a);
    }
    p.out[static_cast<int64_t>(hq) * p.hd + i] = a / L;
  }
}

// ------------------------------------------------------------------ host side
int kv_attention_splits(int n_kv, int64_t n_ctx) {
  const int64_t by_len = (n_ctx + 127) / 128;
  const int64_t by_grid = std::max(1, 512 / n_kv);
  return static_cast<int>(std::max<int64_t>(1, std::min(by_len, by_grid)));
}

size_t kv_attention_workspace_bytes(int n_q, int n_kv, int head_dim, int64_t n_ctx) {
  if (n_kv <= 0 || n_q % n_kv) return 0;
  const int splits = kv_attention_splits(n_kv, n_ctx);
  return static_cast<size_t>(n_kv) * splits * (n_q / n_kv) * (head_dim + 2) * sizeof(float);
}

template <class... KArgs, class... Args>
static cudaError_t launch_pdl_att(void (*kernel)(KArgs...), dim3 grid, int threads,
                                  cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
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
  const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 1024)));
  return launch_pdl_att(rope_kernel, dim3(blocks), 256, st, x, n_heads, head_dim, rot_dim, pos,
                        base);
}

cudaError_t launch_kv_append(float* kc, float* vc, const float* k, const float* v, int n_kv,
                             int head_dim, int64_t max_seq, int64_t pos, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(n_kv) * head_dim;
  const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 1024)));
  return launch_pdl_att(kv_append_kernel, dim3(blocks), 256, st, kc, vc, k, v, n_kv, head_dim,
                        max_seq, pos);
}

cudaError_t launch_kv_attention(const float* q, const float* kc, const float* vc, float* out,
                                int n_q, int n_kv, int head_dim, int64_t max_seq, int64_t n_ctx,
                                float scale, float softcap, float* ws, cudaStream_t st) {
  AttParams p;
  p.q = q;
  p.kc = kc;
  p.vc = vc;
  p.part = ws;
  p.out = out;
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.hd = head_dim;
  p.group = n_q / n_kv;
  p.splits = kv_attention_splits(n_kv, n_ctx);
  p.max_seq = max_seq;
  p.n_ctx = n_ctx;
  p.chunk = (n_ctx + p.splits - 1) / p.splits;
  p.scale = scale;
  p.softcap = softcap;
  const dim3 grid(p.splits, n_kv);
  cudaError_t e;
  switch (head_dim / 32) {
    case 1: e = launch_pdl_att(kv_attention_split_kernel<1>, grid, kAttWarps * 32, st, p); break;
    case 2: e = launch_pdl_att(kv_attention_split_kernel<2>, grid, kAttWarps * 32, st, p); break;
    case 4: e = launch_pdl_att(kv_attention_split_kernel<4>, grid, kAttWarps * 32, st, p); break;
    case 8: e = launch_pdl_att(kv_attention_split_kernel<8>, grid, kAttWarps * 32, st, p); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_pdl_att(kv_attention_merge_kernel, dim3(n_q), 256, st, p);
}

}  // namespace qws
