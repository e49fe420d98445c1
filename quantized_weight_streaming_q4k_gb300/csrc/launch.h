// launch.h -- host-side planning and launchers shared by the C-ABI layer.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <string>

#include "../../include/qws.h"
#include "engine.cuh"

namespace qws {

inline int64_t block_weights(int fmt) { return fmt == 2 || fmt == 8 ? 32 : 256; }
inline int64_t block_bytes(int fmt) {
  return fmt == 2 ? 18 : fmt == 8 ? 34 : fmt == 12 ? 144 : fmt == 14 ? 210 : 0;
}
inline int64_t row_bytes_of(int fmt, int64_t K) { return K / block_weights(fmt) * block_bytes(fmt); }

inline int64_t gcd64(int64_t a, int64_t b) {
  while (b) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Tile / ring geometry of one phase.
struct TilePlan {
  int U, G, T, C;
  uint32_t stage_need;   // bytes of the largest tile (both matrices when paired)
  uint32_t red_floats;
};

// Chooses row slots G and rows per tile T for a phase with K columns and B
// activation vectors.  T is a multiple of G (every slot gets the same number
// of rows) and of the rows that make T * row_bytes a multiple of 16 (aligned
// bulk copies).  rows_hint sizes tiles so that small matrices still spread
// over the grid.  Returns false (with a reason) if the shape does not fit.
inline bool plan_tiles(int fmt, int epi, int64_t K, int B, int64_t rows_hint, int sms,
                       uint32_t tile_target, TilePlan& tp, std::string& why) {
  const int64_t RB = row_bytes_of(fmt, K);
  const int uw = unit_weights(fmt);
  if (K % uw) {
    why = "hidden is not a multiple of the lane unit";
    return false;
  }
  const int64_t U = K / uw;
  if (U > kMaxConsumers) {
    why = "more than 320 lane units per row (hidden too large for one pass)";
    return false;
  }
  const int64_t gmax = kMaxConsumers / (U * B);
  if (gmax < 1) {
    why = "batch * hidden / 64 exceeds 320 lanes";
    return false;
  }
  const int pairm = epi != EPI_STORE ? 2 : 1;
  const int64_t align = 16 / gcd64(RB, 16);
  int64_t G = gmax, T0 = 0;
  for (; G >= 1; --G) {
    T0 = G / gcd64(G, align) * align;
    if (T0 * RB * pairm <= 64 * 1024) break;
  }
  if (G < 1) {
    G = 1;
    T0 = align;
  }
  int64_t m = static_cast<int64_t>(tile_target) / (T0 * RB * pairm);
  if (m < 1) m = 1;
  // small matrices: aim for about one tile per CTA slot of the grid
  const int64_t per = (rows_hint + 2 * sms - 1) / (2 * static_cast<int64_t>(sms));
  const int64_t m_small = (per + T0 - 1) / T0;
  const int64_t m_max = m;
  if (m_small >= 1 && m_small < m) m = m_small;
  // but at least two rows per row slot: the decode loop interleaves two rows'
  // independent chains, and a slot given one row runs it alone
  const int64_t m_ilp = (2 * G + pairm * T0 - 1) / (pairm * T0);
  if (m < m_ilp) m = std::min(m_ilp, m_max);
  tp.U = static_cast<int>(U);
  tp.G = static_cast<int>(G);
  tp.T = static_cast<int>(T0 * m);
  tp.C = static_cast<int>((B * G * U + 31) / 32 * 32);
  tp.stage_need = static_cast<uint32_t>(tp.T * RB * pairm);
  tp.red_floats = static_cast<uint32_t>(B * tp.T * pairm * red_pitch(static_cast<int>(U)));
  return true;
}

inline uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// dynamic shared memory a streaming CTA uses (one CTA per SM), and the
// target bytes of one tile (per stage).  Measured for the 262144 x 2560
// matvecs (same box, two passes; Q4_K / Q6_K / Q4_0 in us): 46 KB 83.7 /
// 132.6 / 77.3, 56 KB 83.6 / 120.6 / 77.2, 64 KB 81.1 / 120.6 / 74.3,
// 72 KB 91.2 / 130.8 / 86.7, 80 KB 87.8 / 130.8 / 82.8, 92 KB 84.7 / 133.8 /
// 80.5: the rows per lane slot of a tile against the ring's depth.
constexpr size_t kSmemBudget = 216 * 1024;
constexpr uint32_t kTileTarget = 64 * 1024;

// ---------------------------------------------------------------- launchers
// All return cudaSuccess or the CUDA error; *why gets a message on failure.
int device_sms();

// y (or split partials) for segments of one format; epi = EPI_STORE/EPI_GEGLU.
cudaError_t launch_matvec(int fmt, int epi, const Seg* segs, int nseg, const uint8_t* W2,
                          const float* x, int64_t K, int B, int splits, cudaStream_t st,
                          std::string* why);
// Q4_0 (wfmt 2) or Q8_0 (wfmt 8) weights times Q8_0 activations xq
// ([B][K / 32 * 34] bytes), no column split.
cudaError_t launch_matvec_q8(int wfmt, const Seg* segs, int nseg, const uint8_t* xq, int64_t K,
                             int B, cudaStream_t st, std::string* why);
// rms_norm (after h += y when residual) quantized to Q8_0 in one launch;
// h is read only (const-cast) when !residual
cudaError_t launch_norm_q8(float* h, const float* y, const float* w, uint8_t* xq, int64_t n,
                           float eps, int batch, bool residual, cudaStream_t st);
// x (nblocks * 32 floats) -> nblocks Q8_0 blocks
cudaError_t launch_quantize_q8_0(const float* x, uint8_t* xq, int64_t nblocks, cudaStream_t st);
// attention over a KV cache (attention.cu)
size_t kv_attention_workspace_bytes(int n_q, int n_kv, int head_dim, int64_t n_ctx);
unsigned read_clear_attention_errors();
cudaError_t launch_rope(float* x, int n_heads, int head_dim, int rot_dim, int64_t pos,
                        double base, cudaStream_t st);
cudaError_t launch_kv_append(float* kc, float* vc, const float* k, const float* v, int n_kv,
                             int head_dim, int64_t max_seq, int64_t pos, cudaStream_t st);
// RoPE and append fused into kv_attention: q, k, v as {value, stamp} words,
// q and k rotated at pos (rot_dim, base), k and v written at pos of kc / vc
// (the same caches the attention reads; q is then unused)
// cos / sin of pos * base^(-2i / rot_dim), i < rot_dim / 2 (rot_dim <= 512),
// from the f64 angle, rounded to f32
void rope_table_f32(int rot_dim, int64_t pos, double base, float* c, float* s);
int kv_attention_splits(int n_kv, int64_t n_ctx);

struct KvFuse {
  const unsigned long long *q, *k, *v;
  float *kc, *vc;
  int64_t pos;
  int rot_dim;
  double base;
};
// out_words set: the result goes there as {value, stamp} words instead of out
cudaError_t launch_kv_attention(const float* q, const float* kc, const float* vc, float* out,
                                int n_q, int n_kv, int head_dim, int64_t max_seq, int64_t n_ctx,
                                float scale, float softcap, float* ws, cudaStream_t st,
                                unsigned long long* out_words = nullptr, unsigned stamp = 0,
                                const KvFuse* fuse = nullptr);
// 2..8 vectors, each weight decoded once (batchmv.cu): fmt 2 Q4_0 / 12 Q4_K
// with f32 x; 102 Q4_0 / 108 Q8_0 with Q8_0 activations xq (x unused)
bool batch_q4_eligible(int fmt, int64_t K, int B);
cudaError_t launch_batch_q4_matvec(int fmt, const uint8_t* W, const float* x, float* y,
                                   int64_t rows, int64_t K, int B, cudaStream_t st,
                                   const uint8_t* xq = nullptr);
unsigned read_clear_batchmv_errors();
// prefill (prefill.cu): X packed to f16 tiles in ws, then the tcgen05 GEMM
size_t prefill_workspace_bytes(int64_t hidden, int64_t n_tokens);
cudaError_t launch_prefill_q4k(const uint8_t* W, const float* X, float* Y, int64_t rows,
                               int64_t K, int64_t N, uint8_t* ws, cudaStream_t st);
unsigned read_clear_prefill_errors();
// y[b][r] = sum_s part[s][b][r]
cudaError_t launch_splitk_reduce(const float* part, float* y, int64_t n, int splits,
                                 cudaStream_t st);
cudaError_t launch_rms_norm(const float* x, const float* w, float* y, int64_t n, float eps,
                            int batch, cudaStream_t st);
cudaError_t launch_residual_add(float* h, const float* y, int64_t n, int batch, cudaStream_t st);
cudaError_t launch_residual_rms_norm(float* h, const float* y, const float* w, float* x,
                                    int64_t n, float eps, int batch, cudaStream_t st);
unsigned read_clear_matvec_errors();
cudaError_t launch_selftest_mbar(long long limit, cudaStream_t st);
cudaError_t launch_selftest_poll(void* word8, long long limit, cudaStream_t st);

// message returned by qws_last_error() on the calling thread (abi.cu)
void set_last_error(const char* msg);

// one decode step over a KV cache (decode_kv.cu)
size_t decode_kv_workspace_bytes(const qws_dims* d, int64_t max_seq);
qws_status decode_kv(const qws_layer* layers, int n_layers, float* h, const qws_dims* d,
                     const qws_kv* kv, void* ws, size_t ws_bytes, cudaStream_t st,
                     std::string& err);

// decode chain (chain.cu)
size_t chain_workspace_bytes(int64_t hidden, int64_t inter);
unsigned read_clear_chain_errors();
// w_final / hn (both or neither): also hn = rms_norm(h_out, w_final) in the
// same launch (qws_decode_chain_final_norm).
qws_status decode_chain(const qws_layer* layers, int n_layers, float* h, const qws_dims* d,
                        void* ws, size_t ws_bytes, cudaStream_t st, std::string& err,
                        const float* w_final = nullptr, float* hn = nullptr,
                        const char* fn = "qws_decode_chain");
// The decode step over a KV cache on the chain kernel: true when the shapes
// fit the chain (hidden <= 5120, q_dim and kv_dim <= 4 * hidden); the
// workspace the step needs then (chain words, attention output words and
// the attention partials).
bool decode_kv_chain_fits(const qws_dims* d);
size_t decode_kv_chain_workspace_bytes(const qws_dims* d, int64_t max_seq);
// Arguments checked by the caller (decode_kv); layers in groups of <= 64.
qws_status decode_kv_chain(const qws_layer* layers, int n_layers, float* h, const qws_dims* d,
                           const qws_kv* kv, void* ws, size_t ws_bytes, cudaStream_t st,
                           std::string& err);

}  // namespace qws
