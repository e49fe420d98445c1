// chain.cu -- the single-token decoder chain in one persistent cooperative
// launch (infer-compute README §Architecture: one command buffer for all
// layers; §Quick Start decode_token; infer-inference PERFORMANCE.md
// §Post-Norm Architecture for the Gemma-3 sandwich norms).
//
// Per layer four streaming phases run on the engine of engine.cuh:
//   QKV   : [q|k|v] = W_{q,k,v} n1,     n1 = rms_norm(h, w_in)
//   O     : o = W_o a,                  a  = v broadcast to the query heads
//   GU    : m = gelu(W_g n2) * (W_u n2), n2 = rms_norm(h1, w_pre_ffn),
//                                       h1 = h + rms_norm(o, w_post_attn)  (or h + o)
//   DOWN  : f = W_d m
// and the next layer's input is h = h1 + rms_norm(f, w_post_ffn) (or h1 + f).
// A phase's input vector depends on every output of the previous phase, so
// the grid meets at a barrier between phases; the producer warp does not:
// weights never depend on activations, so it keeps streaming the next phase's
// tiles into the ring while the grid waits.
//
// Per CTA, the consumers rebuild the phase's input vector themselves from the
// (L2-resident) previous outputs -- each needs only a few KB -- with sums of
// squares reduced in a fixed order, so every CTA computes bit-identical
// vectors; CTA 0 also stores h and h1 for the residual adds.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/qws.h"
#include "launch.h"

namespace qws {

__device__ unsigned g_err_chain;

constexpr int kMaxLayers = 64;
constexpr uint32_t kChainTileTarget = 23 * 1024;  // deeper ring, finer balance across CTAs
constexpr int kChainBar = 2;  // named barrier: reducer + consumers at phase starts

enum : int { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_DOWN = 3 };

struct ChainLayer {
  const uint8_t *Wq, *Wk, *Wv, *Wo, *Wg, *Wu, *Wd;
  const float *w_in, *w_pa, *w_pf, *w_pff;
};

struct KindPlan {
  int fmt, U, G, T;
  int64_t K, row_bytes;
};

struct ChainParams {
  ChainLayer L[kMaxLayers];
  int n_layers;
  int64_t H, I, QD, KD;      // hidden, inter, q_dim, kv_dim
  int n_q_heads, n_kv_heads, head_dim;
  float eps;
  int post_norms;
  KindPlan kp[4];
  // workspace vectors (device)
  float *q, *k, *v, *o, *m, *f, *hin, *h1;
  unsigned* counter;          // grid barrier arrivals (zeroed before launch)
  float* h;                   // user's h (in: layer 0 input, out: chain output)
  uint32_t S, stage_bytes, red_floats, xs_floats;
};

// Phase p = 4 * layer + kind.
struct ChainPhases {
  const ChainParams* p;
  __device__ __forceinline__ int count() const { return 4 * p->n_layers; }
  __device__ __forceinline__ Phase get(int ph) const {
    const int l = ph >> 2, kind = ph & 3;
    const ChainLayer& L = p->L[l];
    const KindPlan& kp = p->kp[kind];
    Phase P;
    P.fmt = kp.fmt;
    P.epi = kind == PH_GU ? EPI_GEGLU : EPI_STORE;
    P.W2 = nullptr;
    P.K = kp.K;
    P.row_bytes = kp.row_bytes;
    P.row_stride = kp.row_bytes;
    P.B = 1;
    P.U = kp.U;
    P.G = kp.G;
    P.T = kp.T;
    P.cta0 = 0;
    P.ncta = static_cast<int>(gridDim.x);
    P.nseg = 1;
    for (int i = 0; i < kMaxSeg; ++i) P.seg[i] = Seg{nullptr, nullptr, 0, 0};
    if (kind == PH_QKV) {
      P.nseg = 3;
      P.seg[0] = Seg{L.Wq, p->q, p->QD, static_cast<int>((p->QD + kp.T - 1) / kp.T)};
      P.seg[1] = Seg{L.Wk, p->k, p->KD, static_cast<int>((p->KD + kp.T - 1) / kp.T)};
      P.seg[2] = Seg{L.Wv, p->v, p->KD, static_cast<int>((p->KD + kp.T - 1) / kp.T)};
    } else if (kind == PH_O) {
      P.seg[0] = Seg{L.Wo, p->o, p->H, static_cast<int>((p->H + kp.T - 1) / kp.T)};
    } else if (kind == PH_GU) {
      P.seg[0] = Seg{L.Wg, p->m, p->I, static_cast<int>((p->I + kp.T - 1) / kp.T)};
      P.W2 = L.Wu;
    } else {
      P.seg[0] = Seg{L.Wd, p->f, p->H, static_cast<int>((p->H + kp.T - 1) / kp.T)};
    }
    P.n_tiles = P.seg[0].tiles + P.seg[1].tiles + P.seg[2].tiles;
    return P;
  }
};

// ----------------------------------------------------------------- helpers
// Sum over the C consumer threads in a fixed order: shuffle tree inside each
// warp, then every thread adds the warp sums 0..nw-1 in order.
__device__ __forceinline__ float block_sum(float v, float* wsum, int ctid, int C) {
  v = warp_sum(v);
  if ((ctid & 31) == 0) wsum[ctid >> 5] = v;
  bar_sync(kConsumerBar, C);
  float t = 0.f;
  for (int i = 0; i < (C >> 5); ++i) t += wsum[i];
  bar_sync(kConsumerBar, C);   // wsum may be reused right after
  return t;
}

// 1 / sqrt(mean(v^2) + eps) over n values read through ld_cg (other CTAs'
// outputs), identical in every CTA.  Loads go out 8 at a time.
__device__ __forceinline__ float inv_rms_global(const float* v, int64_t n, float eps,
                                                float* wsum, int ctid, int C) {
  constexpr int kChunk = 8;
  float ss = 0.f;
  for (int64_t base = ctid; base < n; base += static_cast<int64_t>(kChunk) * C) {
    float t[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int64_t i = base + static_cast<int64_t>(j) * C;
      t[j] = i < n ? ld_cg(v + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j) ss = fmaf(t[j], t[j], ss);
  }
  ss = block_sum(ss, wsum, ctid, C);
  return 1.0f / sqrtf(ss / static_cast<float>(n) + eps);
}

struct VecSrc {  // shared-memory vector
  const float* p;
  __device__ __forceinline__ float operator()(int64_t i) const { return p[i]; }
};

struct NormSrc {  // vec[i] * inv * w[i]
  const float* vec;
  const float* w;
  float inv;
  __device__ __forceinline__ float operator()(int64_t i) const {
    return __fmul_rn(__fmul_rn(vec[i], inv), w[i]);
  }
};

struct GatherSrc {  // attention at seq 1: query head i / hd reads kv head (i / hd) / group
  const float* v;
  int hd, group;
  __device__ __forceinline__ float operator()(int64_t i) const {
    const int head = static_cast<int>(i / hd);
    return ld_cg(v + static_cast<int64_t>(head / group) * hd + (i - static_cast<int64_t>(head) * hd));
  }
};

// vec[i] = base[i] + (post ? add[i] * inv * w[i] : add[i]); CTA 0 also stores
// it to global `store` (if non-null).  base and add may be written by other
// CTAs (read with ld_cg).  Loads go out 8 elements at a time.
__device__ __forceinline__ void residual_into(float* vec, const float* base, const float* add,
                                              const float* w, float inv, bool post,
                                              float* store, int64_t n, int ctid, int C) {
  constexpr int kChunk = 8;
  for (int64_t b0 = ctid; b0 < n; b0 += static_cast<int64_t>(kChunk) * C) {
    float a[kChunk], h[kChunk], ww[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int64_t i = b0 + static_cast<int64_t>(j) * C;
      const bool in = i < n;
      a[j] = in ? ld_cg(add + i) : 0.f;
      h[j] = in ? ld_cg(base + i) : 0.f;
      ww[j] = (in && post) ? w[i] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int64_t i = b0 + static_cast<int64_t>(j) * C;
      if (i < n) {
        // explicit roundings: the same value must come out of every call site
        const float r = __fadd_rn(h[j], post ? __fmul_rn(__fmul_rn(a[j], inv), ww[j]) : a[j]);
        vec[i] = r;
        if (store) store[i] = r;
      }
    }
  }
}

// vec[i] = src[i] (and store[i] = src[i] if store), loads 8 at a time.
__device__ __forceinline__ void copy_into(float* vec, const float* src, float* store, int64_t n,
                                          int ctid, int C) {
  constexpr int kChunk = 8;
  for (int64_t b0 = ctid; b0 < n; b0 += static_cast<int64_t>(kChunk) * C) {
    float t[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int64_t i = b0 + static_cast<int64_t>(j) * C;
      t[j] = i < n ? ld_cg(src + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int64_t i = b0 + static_cast<int64_t>(j) * C;
      if (i < n) {
        vec[i] = t[j];
        if (store) store[i] = t[j];
      }
    }
  }
}

// The per-format decode loops and the two reducer epilogues as separate
// functions: each gets the whole register budget instead of sharing one
// allocation with every other role and phase of the kernel.
__device__ __noinline__ bool chain_consume_q4k(const Phase& P, const Ring& R, RingPos& pos,
                                               int ctid, int C) {
  return consume_phase<UnitQ4K, false, false>(P, R, pos, XOfPlain{nullptr, 0}, ctid, C, &g_err_chain);
}
__device__ __noinline__ bool chain_consume_q6k(const Phase& P, const Ring& R, RingPos& pos,
                                               int ctid, int C) {
  return consume_phase<UnitQ6K, false, false>(P, R, pos, XOfPlain{nullptr, 0}, ctid, C, &g_err_chain);
}
__device__ __forceinline__ bool chain_reduce(const Phase& P, const Ring& R, RingPos& pos) {
  return P.epi == EPI_GEGLU ? reduce_phase(P, R, pos, EpiGeglu{}, &g_err_chain)
                            : reduce_phase(P, R, pos, EpiStore{}, &g_err_chain);
}

// Builds the input vector of phase ph into the staging buffer R.xs (all
// consumer threads; ends with a consumer barrier).  Kept out of line: it runs
// once per phase and must not inflate the decode loop's registers.
__device__ __noinline__ void chain_prologue(const ChainParams& p, int ph, const Ring& R,
                                            float* vec, float* wsum, bool q6, int ctid, int C);

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kRoleThreads + kMaxConsumers, 1)
    chain_kernel(const __grid_constant__ ChainParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R = make_ring(smem, p.S, p.stage_bytes, p.red_floats, p.xs_floats);
  // after the ring: [vec: H floats][wsum: 32 floats][abort flag]
  float* vec = reinterpret_cast<float*>(smem + ring_smem_bytes(p.S, p.stage_bytes, p.red_floats,
                                                                p.xs_floats));
  float* wsum = vec + p.H;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(wsum + 32);
  const int C = static_cast<int>(blockDim.x) - kRoleThreads;
  if (threadIdx.x == 0) {
    ring_init(R, C / 32);
    *abort_flag = 0;
  }
  __syncthreads();
  const ChainPhases phases{&p};
  const int nph = phases.count();

  if (threadIdx.x < kProducerThreads) {
    if (threadIdx.x == 0) run_producer(phases, R, &g_err_chain);
    return;
  }

  RingPos pos;
  if (threadIdx.x < kRoleThreads) {
    // ---------------- reducer: epilogues, then the grid barrier per phase
    const int lane = threadIdx.x & 31;
    for (int ph = 0; ph < nph; ++ph) {
      const Phase P = phases.get(ph);
      bool ok = chain_reduce(P, R, pos);
      __syncwarp();
      if (lane == 0) {
        if (ok) {
          // __syncwarp above orders the warp's epilogue stores before this
          // lane's release; the release-add publishes them at gpu scope
          red_release_gpu_add(p.counter, 1u);
          const unsigned target = static_cast<unsigned>(ph + 1) * gridDim.x;
          const long long t0 = clock64();
          while (ld_acquire_gpu(p.counter) < target) {
            if (clock64() - t0 > kWaitCycles) {
              atomicOr(&g_err_chain, kErrGridBarrier);
              ok = false;
              break;
            }
          }
        }
        if (!ok) *abort_flag = 1;
      }
      __syncwarp();
      bar_sync(kChainBar, C + 32);   // releases the consumers into the next phase
      if (*abort_flag) return;
    }
    return;
  }

  // ---------------- consumers
  const int ctid = static_cast<int>(threadIdx.x) - kRoleThreads;
  const bool down_q6k = p.kp[PH_DOWN].fmt == 14;
  for (int ph = 0; ph < nph; ++ph) {
    if (ph > 0) {
      bar_sync(kChainBar, C + 32);   // previous phase complete on every CTA
      if (*abort_flag) return;
    }
    const Phase P = phases.get(ph);
    // the phase's input vector, staged in R.xs (transposed per lane unit)
    const bool q6 = (ph & 3) == PH_DOWN && down_q6k;
    chain_prologue(p, ph, R, vec, wsum, q6, ctid, C);
    const bool ok = q6 ? chain_consume_q6k(P, R, pos, ctid, C)
                       : chain_consume_q4k(P, R, pos, ctid, C);
    if (!ok) *abort_flag = 1;   // the reducer will time out too and abort at the next barrier
  }
  // final residual: h = h1 + rms_norm(f, w_post_ffn) (or h1 + f)
  bar_sync(kChainBar, C + 32);
  if (*abort_flag) return;
  if (blockIdx.x == 0) {
    const bool post = p.post_norms != 0;
    const ChainLayer& Lp = p.L[p.n_layers - 1];
    const float inv_f = post ? inv_rms_global(p.f, p.H, p.eps, wsum, ctid, C) : 1.f;
    residual_into(vec, p.h1, p.f, Lp.w_pff, inv_f, post, p.h, p.H, ctid, C);
  }
}

// r = base + (post ? add * rms_inv(add) * wa : add)      (or r = base if !add)
// x = r * rms_inv(r) * wn                                 -> staged for Q4_K units
// store[i] = r[i] when store != nullptr.  All global loads of a thread are
// issued at once (one memory latency), provided H <= 8 * C.
__device__ __forceinline__ void resnorm_stage(const ChainParams& p, const Ring& R, float* wsum,
                                              const float* base, const float* add,
                                              const float* wa, const float* wn, float* store,
                                              int US, int ctid, int C) {
  constexpr int kJ = 8;
  const int64_t H = p.H;
  const bool post = p.post_norms != 0;
  float bs[kJ], ad[kJ], wwa[kJ], wwn[kJ];
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int64_t i = ctid + static_cast<int64_t>(j) * C;
    const bool in = i < H;
    bs[j] = in ? ld_cg(base + i) : 0.f;
    ad[j] = (in && add) ? ld_cg(add + i) : 0.f;
    wwa[j] = (in && add && post) ? wa[i] : 0.f;
    wwn[j] = in ? wn[i] : 0.f;
  }
  float inv1 = 1.f;
  if (add && post) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kJ; ++j) ss = fmaf(ad[j], ad[j], ss);
    inv1 = 1.0f / sqrtf(block_sum(ss, wsum, ctid, C) / static_cast<float>(H) + p.eps);
  }
  float ss2 = 0.f;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    // explicit roundings: every CTA and call site computes the same r
    float r = bs[j];
    if (add) r = __fadd_rn(bs[j], post ? __fmul_rn(__fmul_rn(ad[j], inv1), wwa[j]) : ad[j]);
    bs[j] = r;
    ss2 = fmaf(r, r, ss2);
  }
  if (store) {
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int64_t i = ctid + static_cast<int64_t>(j) * C;
      if (i < H) store[i] = bs[j];
    }
    __threadfence();   // published to other CTAs through the phase barrier
  }
  const float inv2 = 1.0f / sqrtf(block_sum(ss2, wsum, ctid, C) / static_cast<float>(H) + p.eps);
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int64_t i = ctid + static_cast<int64_t>(j) * C;
    if (i < H) {
      int u, l;
      UnitQ4K::unit_of(i, u, l);
      R.xs[l * US + u] = __fmul_rn(__fmul_rn(bs[j], inv2), wwn[j]);
    }
  }
}

__device__ __noinline__ void chain_prologue(const ChainParams& p, int ph, const Ring& R,
                                            float* vec, float* wsum, bool q6, int ctid, int C) {
  const int l = ph >> 2, kind = ph & 3;
  const ChainLayer& L = p.L[l];
  const int64_t H = p.H;
  const bool post = p.post_norms != 0;
  const KindPlan& kp = p.kp[kind];
  const int US = red_stride(kp.U);
  const bool fast = H <= 8 * static_cast<int64_t>(C);
  if ((kind == PH_QKV || kind == PH_GU) && fast) {
    if (kind == PH_QKV) {
      if (l == 0)
        resnorm_stage(p, R, wsum, p.h, nullptr, nullptr, L.w_in,
                      blockIdx.x == 0 ? p.hin : nullptr, US, ctid, C);
      else
        resnorm_stage(p, R, wsum, p.h1, p.f, p.L[l - 1].w_pff, L.w_in,
                      blockIdx.x == 0 ? p.hin : nullptr, US, ctid, C);
    } else {
      resnorm_stage(p, R, wsum, p.hin, p.o, L.w_pa, L.w_pf, blockIdx.x == 0 ? p.h1 : nullptr, US,
                    ctid, C);
    }
  } else if (kind == PH_QKV || kind == PH_GU) {
    // general sizes: several passes through shared memory
    if (kind == PH_QKV) {
      if (l == 0) {
        copy_into(vec, p.h, blockIdx.x == 0 ? p.hin : nullptr, H, ctid, C);
      } else {
        const ChainLayer& Lp = p.L[l - 1];
        const float inv_f = post ? inv_rms_global(p.f, H, p.eps, wsum, ctid, C) : 1.f;
        residual_into(vec, p.h1, p.f, Lp.w_pff, inv_f, post, blockIdx.x == 0 ? p.hin : nullptr,
                      H, ctid, C);
      }
    } else {
      const float inv_o = post ? inv_rms_global(p.o, H, p.eps, wsum, ctid, C) : 1.f;
      residual_into(vec, p.hin, p.o, L.w_pa, inv_o, post, blockIdx.x == 0 ? p.h1 : nullptr, H,
                    ctid, C);
    }
    bar_sync(kConsumerBar, C);
    float ss = 0.f;
    for (int64_t i = ctid; i < H; i += C) ss = fmaf(vec[i], vec[i], ss);
    const float inv =
        1.0f / sqrtf(block_sum(ss, wsum, ctid, C) / static_cast<float>(H) + p.eps);
    stage_x<UnitQ4K>(R.xs, US, NormSrc{vec, kind == PH_QKV ? L.w_in : L.w_pf, inv}, kp.K, ctid,
                     C);
  } else if (kind == PH_O) {
    stage_x<UnitQ4K>(R.xs, US, GatherSrc{p.v, p.head_dim, p.n_q_heads / p.n_kv_heads}, kp.K, ctid,
                     C);
  } else if (q6) {
    stage_x<UnitQ6K, XCoherent, 32>(R.xs, US, XCoherent{p.m}, kp.K, ctid, C);
  } else {
    stage_x<UnitQ4K, XCoherent, 32>(R.xs, US, XCoherent{p.m}, kp.K, ctid, C);
  }
  // stores of h / h1 by CTA 0 are published by the reducer's release at the
  // end of this phase (they precede it in CTA order through the barriers)
  bar_sync(kConsumerBar, C);
}

// ------------------------------------------------------------------ host side
static int64_t align_floats(int64_t n) { return (n + 63) / 64 * 64; }

size_t chain_workspace_bytes(int64_t hidden, int64_t inter) {
  // q, k, v sized for the largest heads layout the dims allow are passed at
  // call time; here: q <= hidden*... keep generous fixed layout:
  // q [hidden*4], k [hidden*4], v [hidden*4], o, f, hin, h1 [hidden], m [inter]
  if (hidden <= 0 || inter <= 0) return 0;
  const int64_t fl = 3 * align_floats(4 * hidden) + 4 * align_floats(hidden) + align_floats(inter);
  return static_cast<size_t>(fl) * sizeof(float) + 256;
}

unsigned read_clear_chain_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_chain, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_chain, &z, sizeof(z));
  return v;
}

}  // namespace qws

using namespace qws;

// Argument checks and launch (called by qws_decode_chain in abi.cu); kept in
// this translation unit with the workspace layout it depends on.
qws_status qws::decode_chain(const qws_layer* layers, int n_layers, float* h,
                                 const qws_dims* d, void* ws, size_t ws_bytes, cudaStream_t st,
                                 std::string& err) {
  auto bad = [&](qws_status s, const char* m) {
    err = m;
    return s;
  };
  if (!layers || !h || !d || !ws) return bad(QWS_ERR_NULL, "qws_decode_chain: NULL argument");
  if (n_layers < 1 || n_layers > kMaxLayers)
    return bad(QWS_ERR_SHAPE, "qws_decode_chain: n_layers must be in [1, 64]");
  const int64_t H = d->hidden, I = d->inter;
  if (d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 ||
      d->n_q_heads % d->n_kv_heads)
    return bad(QWS_ERR_SHAPE, "qws_decode_chain: bad head counts");
  const int64_t QD = static_cast<int64_t>(d->n_q_heads) * d->head_dim;
  const int64_t KD = static_cast<int64_t>(d->n_kv_heads) * d->head_dim;
  auto ok_dim = [](int64_t v) { return v > 0 && v % 256 == 0 && v <= 20480; };
  if (!ok_dim(H) || !ok_dim(I) || !ok_dim(QD) || KD % 64 || KD <= 0 || QD > 4 * H || KD > 4 * H)
    return bad(QWS_ERR_SHAPE,
               "qws_decode_chain: hidden, inter, q_dim must be multiples of 256 in (0, 20480], "
               "q_dim and kv_dim <= 4 * hidden");
  if (!(d->eps >= 0.f)) return bad(QWS_ERR_SHAPE, "qws_decode_chain: eps must be >= 0");
  if (reinterpret_cast<uintptr_t>(h) % 4 || reinterpret_cast<uintptr_t>(ws) % 16)
    return bad(QWS_ERR_ALIGN, "qws_decode_chain: h must be 4-byte and ws 16-byte aligned");
  if (ws_bytes < chain_workspace_bytes(H, I))
    return bad(QWS_ERR_WORKSPACE, "qws_decode_chain: workspace too small");
  ChainParams p;
  std::memset(&p, 0, sizeof(p));
  for (int l = 0; l < n_layers; ++l) {
    const qws_layer& L = layers[l];
    const void* ws8[7] = {L.Wq, L.Wk, L.Wv, L.Wo, L.Wg, L.Wu, L.Wd};
    for (const void* w : ws8) {
      if (!w) return bad(QWS_ERR_NULL, "qws_decode_chain: a weight pointer is NULL");
      if (reinterpret_cast<uintptr_t>(w) % 16)
        return bad(QWS_ERR_ALIGN, "qws_decode_chain: weights must be 16-byte aligned");
    }
    const float* nw[4] = {L.w_in, L.w_post_attn, L.w_pre_ffn, L.w_post_ffn};
    for (int i = 0; i < 4; ++i) {
      if (!nw[i] && (i == 0 || i == 2 || d->post_norms))
        return bad(QWS_ERR_NULL, "qws_decode_chain: a norm weight pointer is NULL");
      if (reinterpret_cast<uintptr_t>(nw[i]) % 4)
        return bad(QWS_ERR_ALIGN, "qws_decode_chain: norm weights must be 4-byte aligned");
    }
    if (L.fmt_qkv != QWS_Q4_K || L.fmt_o != QWS_Q4_K || L.fmt_gu != QWS_Q4_K ||
        (L.fmt_down != QWS_Q4_K && L.fmt_down != QWS_Q6_K) || L.fmt_down != layers[0].fmt_down)
      return bad(QWS_ERR_FORMAT,
                 "qws_decode_chain: q/k/v/o/gate/up must be Q4_K; down Q4_K or Q6_K (same in "
                 "every layer)");
    p.L[l] = ChainLayer{static_cast<const uint8_t*>(L.Wq), static_cast<const uint8_t*>(L.Wk),
                        static_cast<const uint8_t*>(L.Wv), static_cast<const uint8_t*>(L.Wo),
                        static_cast<const uint8_t*>(L.Wg), static_cast<const uint8_t*>(L.Wu),
                        static_cast<const uint8_t*>(L.Wd), L.w_in, L.w_post_attn, L.w_pre_ffn,
                        L.w_post_ffn};
  }
  p.n_layers = n_layers;
  p.H = H;
  p.I = I;
  p.QD = QD;
  p.KD = KD;
  p.n_q_heads = d->n_q_heads;
  p.n_kv_heads = d->n_kv_heads;
  p.head_dim = d->head_dim;
  p.eps = d->eps;
  p.post_norms = d->post_norms ? 1 : 0;
  p.h = h;

  // workspace carve-up (floats)
  float* w = static_cast<float*>(ws);
  p.q = w;
  w += align_floats(4 * H);
  p.k = w;
  w += align_floats(4 * H);
  p.v = w;
  w += align_floats(4 * H);
  p.o = w;
  w += align_floats(H);
  p.f = w;
  w += align_floats(H);
  p.hin = w;
  w += align_floats(H);
  p.h1 = w;
  w += align_floats(H);
  p.m = w;
  w += align_floats(I);
  p.counter = reinterpret_cast<unsigned*>(w);

  const int sms = device_sms();
  // tile plans per phase kind (same consumer count for all)
  const int fmt_down = layers[0].fmt_down;
  struct K {
    int fmt, epi;
    int64_t K, rows;
  } kinds[4] = {{QWS_Q4_K, EPI_STORE, H, QD + 2 * KD},
                {QWS_Q4_K, EPI_STORE, QD, H},
                {QWS_Q4_K, EPI_GEGLU, H, I},
                {fmt_down, EPI_STORE, I, H}};
  uint32_t stage_need = 0, red = 0, xs = 0;
  for (int i = 0; i < 4; ++i) {
    TilePlan tp;
    std::string why;
    if (!plan_tiles(kinds[i].fmt, kinds[i].epi, kinds[i].K, 1, kinds[i].rows, sms,
                    kChainTileTarget, tp, why)) {
      err = "qws_decode_chain: " + why;
      return QWS_ERR_SHAPE;
    }
    // all kinds run with the same thread count: C = kMaxConsumers
    p.kp[i] = KindPlan{kinds[i].fmt, tp.U, tp.G, tp.T, kinds[i].K,
                       row_bytes_of(kinds[i].fmt, kinds[i].K)};
    stage_need = std::max(stage_need, tp.stage_need);
    red = std::max(red, tp.red_floats);
    xs = std::max<uint32_t>(xs, unit_weights(kinds[i].fmt) * red_stride(tp.U));
  }
  p.stage_bytes = round_up(stage_need + 16, 128);
  p.red_floats = red;
  p.xs_floats = xs;
  const size_t tail = (static_cast<size_t>(H) + 32 + 4) * sizeof(float);
  p.S = 16;
  while (p.S > 2 && ring_smem_bytes(p.S, p.stage_bytes, p.red_floats, p.xs_floats) + tail >
                        kSmemBudget)
    --p.S;
  const size_t smem = ring_smem_bytes(p.S, p.stage_bytes, p.red_floats, p.xs_floats) + tail;
  const int threads = kRoleThreads + kMaxConsumers;

  static std::mutex mu;
  static int attr_dev[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr_dev[dev]) {
      int optin = 0;
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
      attr_dev[dev] = 1;
    }
  }
  int bps = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, chain_kernel, threads, smem);
  if (bps < 1) {
    err = "qws_decode_chain: kernel does not fit on an SM";
    return QWS_ERR_CUDA;
  }
  const int grid = sms;  // one CTA per SM: all co-resident (cooperative launch)
  cudaError_t e = cudaMemsetAsync(p.counter, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) {
    err = std::string("qws_decode_chain: ") + cudaGetErrorString(e);
    return QWS_ERR_CUDA;
  }
  void* args[] = {&p};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(chain_kernel), dim3(grid),
                                  dim3(threads), args, smem, st);
  if (e != cudaSuccess) {
    err = std::string("qws_decode_chain: ") + cudaGetErrorName(e) + " " + cudaGetErrorString(e);
    return QWS_ERR_CUDA;
  }
  return QWS_OK;
}
