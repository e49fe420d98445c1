// decode_kv.cu -- one decode step over a KV cache: every decoder layer at
// sequence position pos (infer-compute README §Architecture, the decode path
// norm -> QKV -> attend -> O -> FFN; §Shaders rows "RoPE" rope_at_pos and
// "Attention" kv_append / kv_attention; infer-inference PERFORMANCE.md
// §Post-Norm Architecture for the Gemma-3 sandwich norms).
//
// Shapes that fit the decode chain (hidden <= 5120, q_dim and kv_dim <= 4 *
// hidden) run on the chain kernel: one chain launch per layer for the
// projections, norms and residuals, with the rope / append and attention
// launches between them (decode_kv_chain, chain.cu).  Other shapes take the
// launch sequence below.
//
// Per layer, on one stream, each launch with programmatic stream
// serialisation (the next launch's weight stream starts while the previous
// one drains):
//   QKV      [q|k|v] = W_{q,k,v} n                  streaming matvec, 3 segments
//   RoPE     q, k rotated at pos                     one launch over n_q + n_kv heads
//   append   k, v written at position pos of the layer's caches
//   attend   a = attention of q over positions 0..pos (split + merge)
//   O        o = W_o a                               streaming matvec
//   resnorm  h <- h + rms_norm(o) w_pa ; n <- rms_norm(h) w_pf   (one CTA)
//   GU       m = gelu(W_g n) * (W_u n)               streaming matvec, GEGLU epilogue
//   down     f = W_d m                               streaming matvec
//   resnorm  h <- h + rms_norm(f) w_pff ; n <- rms_norm(h) w_in of the next layer
// The first layer's input norm is one rms_norm launch.  Without post norms
// the residuals add o and f as they are.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>

#include "../../include/qws.h"
#include "launch.h"

namespace qws {

// h <- h + (post ? rms_norm(y) * wa : y);  x <- rms_norm(h) * wn  (when wn).
// One CTA; sums of squares reduced in a fixed order (per-thread strided
// partials, a fixed shuffle tree, then the warp sums in order).
__global__ void __launch_bounds__(1024) post_norm_residual_kernel(
    float* __restrict__ h, const float* __restrict__ y, const float* __restrict__ wa,
    const float* __restrict__ wn, float* __restrict__ x, int64_t n, float eps, int post) {
  __shared__ float wsum[32];
  __shared__ float inv_s;
  pdl_launch_dependents();
  pdl_wait();
  const int nw = static_cast<int>(blockDim.x >> 5);
  auto block_inv = [&](float ss) {
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int i = 0; i < nw; ++i) t += wsum[i];
      inv_s = 1.0f / sqrtf(t / static_cast<float>(n) + eps);
    }
    __syncthreads();
    const float inv = inv_s;
    __syncthreads();   // wsum / inv_s may be reused
    return inv;
  };
  float inv1 = 1.f;
  if (post) {
    float ss = 0.f;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(y[i], y[i], ss);
    inv1 = block_inv(ss);
  }
  float ss2 = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const float r = post ? h[i] + y[i] * inv1 * wa[i] : h[i] + y[i];
    h[i] = r;   // each thread reads back only what it wrote itself
    ss2 = fmaf(r, r, ss2);
  }
  if (!wn) return;
  const float inv2 = block_inv(ss2);
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) x[i] = h[i] * inv2 * wn[i];
}

namespace {

int64_t align64(int64_t v) { return (v + 63) / 64 * 64; }

struct KvLayout {
  int64_t q, k, v, a, o, n, m, f, att;   // float offsets into the workspace
  size_t bytes;
};

KvLayout kv_layout(int64_t H, int64_t I, int64_t QD, int64_t KD, int n_q, int n_kv, int hd,
                   int64_t max_seq) {
  KvLayout L;
  int64_t at = 0;
  L.q = at;                 // q, k, v contiguous: RoPE covers q and k in one launch
  L.k = L.q + QD;
  L.v = L.k + KD;
  at = align64(L.v + KD);
  L.a = at;
  at = align64(at + QD);
  L.o = at;
  at = align64(at + H);
  L.n = at;
  at = align64(at + H);
  L.m = at;
  at = align64(at + I);
  L.f = at;
  at = align64(at + H);
  L.att = at;
  at += static_cast<int64_t>(kv_attention_workspace_bytes(n_q, n_kv, hd, max_seq) / sizeof(float));
  L.bytes = static_cast<size_t>(align64(at)) * sizeof(float);
  return L;
}

}  // namespace

size_t decode_kv_workspace_bytes(const qws_dims* d, int64_t max_seq) {
  if (!d || d->hidden <= 0 || d->inter <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 ||
      d->head_dim <= 0 || max_seq < 1 || d->n_q_heads % d->n_kv_heads)
    return 0;
  const int64_t QD = static_cast<int64_t>(d->n_q_heads) * d->head_dim;
  const int64_t KD = static_cast<int64_t>(d->n_kv_heads) * d->head_dim;
  const size_t seq = kv_layout(d->hidden, d->inter, QD, KD, d->n_q_heads, d->n_kv_heads,
                               d->head_dim, max_seq)
                         .bytes;
  return decode_kv_chain_fits(d) ? std::max(seq, decode_kv_chain_workspace_bytes(d, max_seq))
                                 : seq;
}

static cudaError_t launch_post_norm_residual(float* h, const float* y, const float* wa,
                                             const float* wn, float* x, int64_t n, float eps,
                                             bool post, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, post_norm_residual_kernel, h, y, wa, wn, x, n, eps,
                            post ? 1 : 0);
}

qws_status decode_kv(const qws_layer* layers, int n_layers, float* h, const qws_dims* d,
                     const qws_kv* kv, void* ws, size_t ws_bytes, cudaStream_t st,
                     std::string& err) {
  auto bad = [&](qws_status s, const std::string& m) {
    err = "qws_decode_kv: " + m;
    return s;
  };
  if (!layers || !h || !d || !kv || !ws) return bad(QWS_ERR_NULL, "NULL argument");
  if (n_layers < 1) return bad(QWS_ERR_SHAPE, "n_layers must be >= 1");
  const int64_t H = d->hidden, I = d->inter;
  const int nq = d->n_q_heads, nkv = d->n_kv_heads, hd = d->head_dim;
  if (nkv < 1 || nq < nkv || nq % nkv || nq / nkv > 4)
    return bad(QWS_ERR_SHAPE, "n_q_heads / n_kv_heads must be an integer in 1..4");
  if (hd != 32 && hd != 64 && hd != 128 && hd != 256)
    return bad(QWS_ERR_SHAPE, "head_dim must be 32, 64, 128 or 256");
  const int64_t QD = static_cast<int64_t>(nq) * hd, KD = static_cast<int64_t>(nkv) * hd;
  auto ok_dim = [](int64_t v) { return v > 0 && v % 256 == 0 && v <= 20480; };
  if (!ok_dim(H) || !ok_dim(I) || !ok_dim(QD) || KD % 64)
    return bad(QWS_ERR_SHAPE,
               "hidden, inter and q_dim must be multiples of 256 in (0, 20480], kv_dim of 64");
  if (!(d->eps >= 0.f)) return bad(QWS_ERR_SHAPE, "eps must be >= 0");
  if (!kv->k_caches || !kv->v_caches) return bad(QWS_ERR_NULL, "cache pointer arrays are NULL");
  if (kv->max_seq < 1 || kv->pos < 0 || kv->pos >= kv->max_seq)
    return bad(QWS_ERR_SHAPE, "need 0 <= pos < max_seq");
  if (kv->rot_dim < 2 || kv->rot_dim % 2 || kv->rot_dim > hd || !(kv->rope_base > 0.0))
    return bad(QWS_ERR_SHAPE, "need an even 0 < rot_dim <= head_dim and rope_base > 0");
  if (!std::isfinite(kv->attn_scale) || !(kv->softcap >= 0.f) || !std::isfinite(kv->softcap))
    return bad(QWS_ERR_SHAPE, "attn_scale must be finite and softcap >= 0");
  if (reinterpret_cast<uintptr_t>(h) % 16 || reinterpret_cast<uintptr_t>(ws) % 16)
    return bad(QWS_ERR_ALIGN, "h and ws must be 16-byte aligned");
  const KvLayout Lw = kv_layout(H, I, QD, KD, nq, nkv, hd, kv->max_seq);
  if (ws_bytes < decode_kv_workspace_bytes(d, kv->max_seq))
    return bad(QWS_ERR_WORKSPACE, "workspace too small");
  for (int l = 0; l < n_layers; ++l) {
    const qws_layer& L = layers[l];
    const void* wts[7] = {L.Wq, L.Wk, L.Wv, L.Wo, L.Wg, L.Wu, L.Wd};
    for (const void* w : wts) {
      if (!w) return bad(QWS_ERR_NULL, "a weight pointer is NULL");
      if (reinterpret_cast<uintptr_t>(w) % 16)
        return bad(QWS_ERR_ALIGN, "weights must be 16-byte aligned");
    }
    const float* nw[4] = {L.w_in, L.w_post_attn, L.w_pre_ffn, L.w_post_ffn};
    for (int i = 0; i < 4; ++i)
      if (!nw[i] && (i == 0 || i == 2 || d->post_norms))
        return bad(QWS_ERR_NULL, "a norm weight pointer is NULL");
    if (L.fmt_qkv != QWS_Q4_K || L.fmt_o != QWS_Q4_K || L.fmt_gu != QWS_Q4_K ||
        (L.fmt_down != QWS_Q4_K && L.fmt_down != QWS_Q6_K))
      return bad(QWS_ERR_FORMAT, "q/k/v/o/gate/up must be Q4_K; down Q4_K or Q6_K");
    const float* kc = kv->k_caches[l];
    const float* vc = kv->v_caches[l];
    if (!kc || !vc) return bad(QWS_ERR_NULL, "a cache pointer is NULL");
    if (reinterpret_cast<uintptr_t>(kc) % 16 || reinterpret_cast<uintptr_t>(vc) % 16)
      return bad(QWS_ERR_ALIGN, "caches must be 16-byte aligned");
  }
  bool same_down = true;   // the chain takes one down-projection format
  for (int l = 1; l < n_layers; ++l)
    same_down = same_down && layers[l].fmt_down == layers[0].fmt_down;
  if (same_down && decode_kv_chain_fits(d))
    return decode_kv_chain(layers, n_layers, h, d, kv, ws, ws_bytes, st, err);

  float* w = static_cast<float*>(ws);
  float *q = w + Lw.q, *k = w + Lw.k, *v = w + Lw.v, *a = w + Lw.a, *o = w + Lw.o;
  float *n = w + Lw.n, *m = w + Lw.m, *f = w + Lw.f, *att = w + Lw.att;
  const bool post = d->post_norms != 0;
  std::string why;
  auto cuda = [&](cudaError_t e, const char* what) {
    err = std::string("qws_decode_kv: ") + what + ": " +
          (why.empty() ? cudaGetErrorString(e) : why);
    return QWS_ERR_CUDA;
  };
  cudaError_t e = launch_rms_norm(h, layers[0].w_in, n, H, d->eps, 1, st);
  if (e != cudaSuccess) return cuda(e, "input norm");
  for (int l = 0; l < n_layers; ++l) {
    const qws_layer& L = layers[l];
    const uint8_t* Wq = static_cast<const uint8_t*>(L.Wq);
    const Seg qkv[3] = {Seg{Wq, q, QD, 0}, Seg{static_cast<const uint8_t*>(L.Wk), k, KD, 0},
                        Seg{static_cast<const uint8_t*>(L.Wv), v, KD, 0}};
    e = launch_matvec(QWS_Q4_K, EPI_STORE, qkv, 3, nullptr, n, H, 1, 1, st, &why);
    if (e != cudaSuccess) return cuda(e, "QKV");
    e = launch_rope(q, nq + nkv, hd, kv->rot_dim, kv->pos, kv->rope_base, st);
    if (e != cudaSuccess) return cuda(e, "RoPE");
    e = launch_kv_append(kv->k_caches[l], kv->v_caches[l], k, v, nkv, hd, kv->max_seq, kv->pos,
                         st);
    if (e != cudaSuccess) return cuda(e, "kv_append");
    e = launch_kv_attention(q, kv->k_caches[l], kv->v_caches[l], a, nq, nkv, hd, kv->max_seq,
                            kv->pos + 1, kv->attn_scale, kv->softcap, att, st);
    if (e != cudaSuccess) return cuda(e, "kv_attention");
    const Seg so{static_cast<const uint8_t*>(L.Wo), o, H, 0};
    e = launch_matvec(QWS_Q4_K, EPI_STORE, &so, 1, nullptr, a, QD, 1, 1, st, &why);
    if (e != cudaSuccess) return cuda(e, "O projection");
    e = launch_post_norm_residual(h, o, L.w_post_attn, L.w_pre_ffn, n, H, d->eps, post, st);
    if (e != cudaSuccess) return cuda(e, "attention residual");
    const Seg sg{static_cast<const uint8_t*>(L.Wg), m, I, 0};
    e = launch_matvec(QWS_Q4_K, EPI_GEGLU, &sg, 1, static_cast<const uint8_t*>(L.Wu), n, H, 1,
                      1, st, &why);
    if (e != cudaSuccess) return cuda(e, "gate/up");
    const Seg sd{static_cast<const uint8_t*>(L.Wd), f, H, 0};
    e = launch_matvec(L.fmt_down, EPI_STORE, &sd, 1, nullptr, m, I, 1, 1, st, &why);
    if (e != cudaSuccess) return cuda(e, "down");
    const float* wn_next = l + 1 < n_layers ? layers[l + 1].w_in : nullptr;
    e = launch_post_norm_residual(h, f, L.w_post_ffn, wn_next, n, H, d->eps, post, st);
    if (e != cudaSuccess) return cuda(e, "FFN residual");
  }
  return QWS_OK;
}

}  // namespace qws
