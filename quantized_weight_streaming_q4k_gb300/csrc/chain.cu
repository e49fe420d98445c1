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
//
// Synchronisation without grid barriers.  A phase's input depends on every
// output of the previous phase.  Every output element is stored as one 64-bit
// word {value, stamp}, stamp = 1 + the index of the phase that wrote it, and a
// CTA starting phase p loads the words it needs until their stamps say they
// come from phase p-1 (bounded polling): the data and the "it is ready" signal
// arrive in the same round trip.  The producer warp never waits for
// activations: weights do not depend on them, so it keeps streaming the next
// phases' tiles into the ring.
//
// Write-after-read: before overwriting a buffer, a writer checks (one load,
// normally already satisfied) that every CTA has finished the phase prologue
// that last read the old contents; each CTA bumps a counter after each
// prologue.  The vectors h and h1 that the keeper CTA stores alternate
// between two buffers by layer parity, so that check does not wait in
// practice.
//
// Every CTA rebuilds a phase's input vector itself from the (L2-resident)
// previous outputs; sums of squares are reduced in a fixed order, so every CTA
// computes bit-identical vectors.  The keeper is the grid's last CTA: tiles
// are dealt from CTA 0 up, so it never owns more tiles than any other CTA, and
// its extra work (storing h, h1 and the final h) stays off the critical path.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "../../include/qws.h"
#include "launch.h"

namespace qws {

__device__ unsigned g_err_chain;

constexpr int kMaxLayers = 64;
// measured optimum at 4 stages (inlined prologue / decode)
constexpr uint32_t kChainTileTarget = 46 * 1024;
constexpr uint32_t kChainStages = 4;
// Tiles of a phase the producer may copy before this CTA has built the
// phase's input vector; the later ones wait for it, so that their bytes do
// not share the SM's path from L2 with the prologue's polls.  With a 3-stage
// ring this holds back the one tile that would otherwise land during the
// boundary.  Measured on the 34-layer Gemma-3-4B chain (same box, two
// passes): 1015 -> 983 us per token with 2, 1010 with 1; gating only the
// gate/up phases 990, only the down phases 1011.  Over a KV cache: gated when
// the attention runs inside (one launch per token: 1404.9 -> 1394.2 us), but
// not when the chain runs as one launch per layer between the attention
// launches (each launch starts with an empty ring: 1573 ungated, 1613 gated).
constexpr int kGateTiles = 2;
constexpr int64_t kMaxChainHidden = 16 * kMaxConsumers;  // residual vectors: 16 per thread

enum : int { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_DOWN = 3 };

struct ChainLayer {
  const uint8_t *Wq, *Wk, *Wv, *Wo, *Wg, *Wu, *Wd;
  const float *w_in, *w_pa, *w_pf, *w_pff;
};

struct KindPlan {
  int fmt, U, G, T;
  int T2, n1;        // balanced last round: tiles from n1 on hold T2 rows
  int64_t K, row_bytes;
};

using Word = unsigned long long;  // {value bits, stamp << 32}

struct ChainParams {
  ChainLayer L[kMaxLayers];
  int n_layers;
  int64_t H, I, QD, KD;      // hidden, inter, q_dim, kv_dim
  int n_q_heads, n_kv_heads, head_dim;
  float eps;
  int post_norms;
  KindPlan kp[4];
  // stamped workspace vectors (device); hin and h1 hold two buffers of H each
  Word *q, *k, *v, *o, *m, *f, *hin, *h1;
  // [4 * n_layers]: CTAs done with each phase's prologue (zeroed per token)
  unsigned* prologues;
  float* h;                   // the caller's h (in: layer 0 input, out: chain output)
  // optional final norm of the last layer's output (keeper CTA): hn = rms_norm(h, w_final)
  const float* w_final;
  float* hn;
  uint32_t S, stage_bytes, red_floats, xs_floats;
  // This launch runs phases [ph_begin, ph_end) of the token; several launches
  // with the same parameters and workspace (cleared once per token) run a
  // token in pieces.  With att set (decode over a KV cache), the O phase of
  // layer l reads the attention output there (q_dim stamped words, stamp
  // 4 l + 1, written between launches) instead of gathering v.
  int ph_begin, ph_end;
  Word* att;
  // Attention inside the O prologue (fused_att = 1; decode over a KV cache,
  // every layer in one launch).  Step 1: work item (kv head g, chunk j) --
  // positions [j * chunk_len, (j + 1) * chunk_len) of n_ctx = pos + 1 -- is
  // taken by CTA (g * chunks + j) mod grid and leaves its partial (acc[hd],
  // m, l per query head of the group) as stamped words in part; the item
  // holding pos rotates k and writes k and v into the caches.  Step 2: CTA
  // b merges attention outputs [b * per, (b + 1) * per) into att.  Stamps:
  // 4 l + 1 (part and att of layer l; both buffers are cleared per token).
  int fused_att;
  float *kc[kMaxLayers], *vc[kMaxLayers];
  int64_t max_seq, pos;
  int chunks, chunk_len, rot_dim;
  float att_scale, softcap;
  Word* part;
  float rtc[256], rts[256];   // cos / sin of pos * base^(-2i / rot_dim), f32
};

__device__ __forceinline__ Word ld_word(const Word* p) {
  Word w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
__device__ __forceinline__ void st_word(Word* p, float v, unsigned stamp) {
  const Word w = static_cast<Word>(__float_as_uint(v)) | (static_cast<Word>(stamp) << 32);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned stamp_of(Word w) { return static_cast<unsigned>(w >> 32); }
__device__ __forceinline__ float value_of(Word w) {
  return __uint_as_float(static_cast<unsigned>(w & 0xFFFFFFFFu));
}

// Waits (bounded) until every CTA has finished the prologue of phase ph.
// Release / acquire: a CTA counts its prologue with a release add after a
// barrier that follows every load of that prologue, and a writer reads the
// full count with an acquire load before it stores, so by the memory model
// the prologue's loads cannot observe the later stores (a reader that ever
// met a newer stamp would time out, not read a wrong value, in any case).
__device__ __forceinline__ bool wait_prologues(const ChainParams& p, int ph) {
  if (ph < 0) return true;
  const unsigned* c = p.prologues + ph;
  if (ld_acquire_gpu(c) >= gridDim.x) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(c) < gridDim.x) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(&g_err_chain, kErrGridBarrier);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Phase p = 4 * layer + kind; its outputs carry stamp p + 1.  get(p) takes
// the absolute phase index; Range views this launch's phases from 0.
// kQFirst: the QKV phase's segments in the order q, k, v (the decode over a
// KV cache) instead of v, k, q (the chain at sequence length 1).
template <bool kQFirst>
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
    P.T2 = kp.T2;
    P.n1 = kp.n1;
    P.cta0 = 0;
    P.ncta = static_cast<int>(gridDim.x);
    P.nseg = 1;
    // a segment's y names its stamped destination (Word*), which only the
    // chain's epilogue uses
    auto dst = [](Word* w) { return reinterpret_cast<float*>(w); };
    for (int i = 0; i < kMaxSeg; ++i) P.seg[i] = Seg{nullptr, nullptr, 0, 0};
    // tiles of a one-segment phase: n1 tiles of T rows, the rest of T2 rows
    auto tiles = [&](int64_t rows) {
      const int64_t big = static_cast<int64_t>(kp.n1) * kp.T;
      if (rows <= big) return static_cast<int>((rows + kp.T - 1) / kp.T);
      return kp.n1 + static_cast<int>((rows - big + kp.T2 - 1) / kp.T2);
    };
    if (kind == PH_QKV) {
      // v first: at sequence length 1 the O phase needs only v, and v's tiles
      // are then dealt in the first round, finished before the CTAs' last
      // tiles (q and k feed nothing downstream).  Over a KV cache q goes
      // first instead: every attention item needs the group's q, only the
      // items holding pos need k and v, and they take that row last.
      P.nseg = 3;
      const int tkv = static_cast<int>((p->KD + kp.T - 1) / kp.T);
      const int tq = static_cast<int>((p->QD + kp.T - 1) / kp.T);
      if constexpr (kQFirst) {
        P.seg[0] = Seg{L.Wq, dst(p->q), p->QD, tq};
        P.seg[1] = Seg{L.Wk, dst(p->k), p->KD, tkv};
        P.seg[2] = Seg{L.Wv, dst(p->v), p->KD, tkv};
      } else {
        P.seg[0] = Seg{L.Wv, dst(p->v), p->KD, tkv};
        P.seg[1] = Seg{L.Wk, dst(p->k), p->KD, tkv};
        P.seg[2] = Seg{L.Wq, dst(p->q), p->QD, tq};
      }
    } else if (kind == PH_O) {
      P.seg[0] = Seg{L.Wo, dst(p->o), p->H, tiles(p->H)};
    } else if (kind == PH_GU) {
      P.seg[0] = Seg{L.Wg, dst(p->m), p->I, tiles(p->I)};
      P.W2 = L.Wu;
    } else {
      P.seg[0] = Seg{L.Wd, dst(p->f), p->H, tiles(p->H)};
    }
    P.n_tiles = P.seg[0].tiles + P.seg[1].tiles + P.seg[2].tiles;
    return P;
  }
  struct Range {
    const ChainPhases* all;
    int begin, end;
    __device__ __forceinline__ int count() const { return end - begin; }
    __device__ __forceinline__ Phase get(int i) const { return all->get(begin + i); }
  };
};

// Reducer epilogue: stores each reduced row (GEGLU for the gate/up pair) as a
// stamped word in the segment's destination (q / k / v, o, m or f).  The
// reducer checks before the phase that every CTA has finished the prologue
// that last read the buffer's old contents: phase ph - 3 (v by O, o by GU, m
// by DOWN, f by the next QKV -- each three phases later than its writer).
struct EpiStamped {
  int ph;
  __device__ __forceinline__ void operator()(const Phase& P, const TileRef& tr, int, int o, float v,
                                             float v2) const {
    Word* dst = reinterpret_cast<Word*>(tr.y);
    const float val = (ph & 3) == PH_GU ? gelu_tanh(v) * v2 : v;
    st_word(dst + tr.r0 + o, val, static_cast<unsigned>(ph + 1));
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
// The same sum without the closing barrier: the caller does not write `buf`
// again before a later barrier of all C threads (the prologue's two norms
// take the two halves of the warp-sum area).
__device__ __forceinline__ float block_sum_once(float v, float* buf, int ctid, int C) {
  v = warp_sum(v);
  if ((ctid & 31) == 0) buf[ctid >> 5] = v;
  bar_sync(kConsumerBar, C);
  float t = 0.f;
  for (int i = 0; i < (C >> 5); ++i) t += buf[i];
  return t;
}

constexpr int kC = kMaxConsumers;   // the chain always runs this many consumer threads

// Polls the words b[j * kC] (j < kJ, b + j * kC < end) until each carries stamp
// `want` and hands each value to put(j, value) as it arrives.  The first round
// issues every load at once, so a vector costs one L2 round trip when it is
// ready.  Bounded: returns false (error bit set) on timeout.
template <int kJ, class Put>
__device__ __forceinline__ bool poll_stamped(const Word* b, const Word* end, unsigned want,
                                             Put&& put, long long limit = kWaitCycles) {
  unsigned pending = 0;
#pragma unroll
  for (int j = 0; j < kJ; ++j)
    if (b + j * kC < end) pending |= 1u << j;
  long long t0 = 0;
  bool first = true;
  while (pending) {
    Word w[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) w[j] = (pending >> j & 1u) ? ld_word(b + j * kC) : 0ull;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      if ((pending >> j & 1u) && stamp_of(w[j]) == want) {
        put(j, value_of(w[j]));
        pending &= ~(1u << j);
      }
    }
    if (!pending) break;
    if (first) {
      t0 = clock64();
      first = false;
    } else if (clock64() - t0 > limit) {
      atomicOr(&g_err_chain, kErrFullWait);
      return false;
    }
  }
  return true;
}

// r = base + (post ? add * rms_inv(add) * wa : add)      (r = base when add == null)
// x = r * rms_inv(r) * wn  -> staged for Q4_K lane units (transposed)
// Element ctid + j * kC of each vector lives in thread ctid's registers
// (H <= kJ * kC).  When store != null (keeper CTA) r is also stored as stamped
// words, after the write-after-read check against phase store_war.  `base` is
// the caller's plain h when base_plain != null (layer 0), else a stamped
// vector.  kEarlyW: load the norm weights together with the vectors (one round
// trip; more registers).
template <int kJ, bool kEarlyW>
__device__ __forceinline__ bool resnorm_stage(const ChainParams& p, const Ring& R, float* wsum,
                                              const Word* base, unsigned base_stamp,
                                              const float* base_plain, const Word* add,
                                              unsigned add_stamp, const float* wa,
                                              const float* wn, Word* store, unsigned store_stamp,
                                              int store_war, unsigned war_seen, int US,
                                              int ctid) {
  const int64_t H = p.H;
  const bool post = p.post_norms != 0;
  float bs[kJ], ad[kJ], wwa[kJ], wwn[kJ];
  if constexpr (kEarlyW) {
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int64_t i = ctid + static_cast<int64_t>(j) * kC;
      wwa[j] = (i < H && add && post) ? wa[i] : 0.f;
      wwn[j] = i < H ? wn[i] : 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int64_t i = ctid + static_cast<int64_t>(j) * kC;
    bs[j] = (i < H && base_plain) ? base_plain[i] : 0.f;
    ad[j] = 0.f;
  }
  bool ok = true;
  if (!base_plain)
    ok = poll_stamped<kJ>(base + ctid, base + H, base_stamp, [&](int j, float v) { bs[j] = v; });
  if (add)
    ok = poll_stamped<kJ>(add + ctid, add + H, add_stamp, [&](int j, float v) { ad[j] = v; }) && ok;
  if constexpr (!kEarlyW) {
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int64_t i = ctid + static_cast<int64_t>(j) * kC;
      wwa[j] = (i < H && add && post) ? wa[i] : 0.f;
      wwn[j] = i < H ? wn[i] : 0.f;
    }
  }
  float inv1 = 1.f;
  if (add && post) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kJ; ++j) ss = fmaf(ad[j], ad[j], ss);
    inv1 = 1.0f / sqrtf(block_sum_once(ss, wsum, ctid, kC) / static_cast<float>(H) + p.eps);
  }
  float ss2 = 0.f;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    // explicit roundings: every CTA computes the same r
    float r = bs[j];
    if (add) r = __fadd_rn(bs[j], post ? __fmul_rn(__fmul_rn(ad[j], inv1), wwa[j]) : ad[j]);
    bs[j] = r;
    ss2 = fmaf(r, r, ss2);
  }
  if (store) {
    // war_seen: the count loaded at the prologue's start (usually full already)
    if (war_seen < gridDim.x && !wait_prologues(p, store_war)) ok = false;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int64_t i = ctid + static_cast<int64_t>(j) * kC;
      if (i < H) st_word(store + i, bs[j], store_stamp);
    }
  }
  const float inv2 =
      1.0f / sqrtf(block_sum_once(ss2, wsum + 32, ctid, kC) / static_cast<float>(H) + p.eps);
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int64_t i = ctid + static_cast<int64_t>(j) * kC;
    if (i < H) {
      int u, l;
      UnitQ4K::unit_of(i, u, l);
      R.xs[l * US + u] = __fmul_rn(__fmul_rn(bs[j], inv2), wwn[j]);
    }
  }
  return ok;
}

// Stages a stamped vector of n values for the lane units of Unit, kJ values per
// thread per round trip.
template <class Unit, int kJ>
__device__ __forceinline__ bool stage_stamped(const Ring& R, int US, const Word* src,
                                              unsigned want, int64_t n, int ctid) {
  bool ok = true;
  for (int64_t b0 = ctid; b0 < n; b0 += static_cast<int64_t>(kJ) * kC) {
    ok = poll_stamped<kJ>(src + b0, src + n, want,
                          [&](int j, float v) {
                            int u, l;
                            Unit::unit_of(b0 + static_cast<int64_t>(j) * kC, u, l);
                            R.xs[l * US + u] = v;
                          }) &&
         ok;
  }
  return ok;
}

// ------------------------------------------------------------ fused attention
// Polls up to kN stamped words at addresses a[0..n) until each carries stamp
// `want`; their values go to v[].  All pending loads go out together.
template <int kN>
__device__ __forceinline__ bool poll_words(const Word* const (&a)[kN], int n, unsigned want,
                                           float (&v)[kN]) {
  unsigned pending = 0;
#pragma unroll
  for (int k = 0; k < kN; ++k)
    if (k < n) pending |= 1u << k;
  long long t0 = 0;
  bool first = true;
  while (pending) {
    Word w[kN];
#pragma unroll
    for (int k = 0; k < kN; ++k) w[k] = (pending >> k & 1u) ? ld_word(a[k]) : 0ull;
#pragma unroll
    for (int k = 0; k < kN; ++k)
      if ((pending >> k & 1u) && stamp_of(w[k]) == want) {
        v[k] = value_of(w[k]);
        pending &= ~(1u << k);
      }
    if (!pending) break;
    if (first) {
      t0 = clock64();
      first = false;
    } else if (clock64() - t0 > kWaitCycles) {
      atomicOr(&g_err_chain, kErrFullWait);
      return false;
    }
  }
  return true;
}

// Shared-memory floats the fused attention steps use (inside the staging
// buffer, before the O projection's vector is staged there).
constexpr int kAttWarpsC = kMaxConsumers / 32;   // 10 consumer warps
constexpr int kAttGH = 512;                       // group heads x head_dim staged
constexpr int kAttMergeBatch = 48;                // outputs merged per round (at most)
// staging-buffer floats of the split step: rotated q, k / v of pos, raw q,
// the warps' partial outputs, m and l (the merge step's need, three floats
// per merged output and chunk, is added by the host)
__host__ __device__ constexpr int att_split_floats() {
  return 4 * kAttGH + kAttWarpsC * kAttGH + 2 * kAttWarpsC * 4;
}

// Element i of a head (raw values at x) rotated at pos (f32 cos / sin).
__device__ __forceinline__ float rope_at(const float* x, int i, int rot_dim, const float* tc,
                                         const float* ts) {
  if (i >= rot_dim) return x[i];
  const int half = rot_dim / 2;
  const int j = i < half ? i : i - half;
  const float a = x[j], b = x[j + half];
  return i < half ? fmaf(a, tc[j], -(b * ts[j])) : fmaf(a, ts[j], b * tc[j]);
}

// Step 1 of the fused attention for layer l: this CTA's work items.
// Per item the group's q (and, for the item holding pos, k and v) come from
// the QKV phase's stamped words (stamp 4 l + 1); warp w takes positions
// p0 + w, p0 + w + 10, ...; lane L holds columns [L kPL, (L + 1) kPL) of q,
// k, v and the running output; the warps are merged in order 0..9 and the
// item's partial is stored as stamped words.
template <int kPL, int kG>
__device__ __forceinline__ bool att_split(const ChainParams& p, int l, float* sm, int ctid) {
  constexpr int hd = kPL * 32;
  const unsigned want = static_cast<unsigned>(4 * l + 1);
  const int warp = ctid >> 5, lane = ctid & 31, c0 = lane * kPL;
  const int64_t n_ctx = p.pos + 1;
  const int items = p.n_kv_heads * p.chunks;
  float* sq = sm;                          // [kG][hd] rotated q
  float* skv = sm + kAttGH;                // [2][hd] k (rotated), v of pos
  float* sraw = sm + 2 * kAttGH;           // [kG][hd] raw q, then [2][hd] raw k, v
  float* sacc = sm + 4 * kAttGH;           // [10][kG][hd]
  float* smm = sacc + kAttWarpsC * kAttGH;  // [10][4]
  float* sml = smm + kAttWarpsC * 4;
  const float* kcl = p.kc[l];
  const float* vcl = p.vc[l];
  bool ok = true;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int g = item / p.chunks, j = item - g * p.chunks;
    const int64_t p0 = static_cast<int64_t>(j) * p.chunk_len;
    const int64_t p1 = min(p0 + p.chunk_len, n_ctx);
    const bool has_pos = p.pos >= p0 && p.pos < p1;
    // raw q of the group's heads (contiguous)
    ok = poll_stamped<2>(p.q + static_cast<int64_t>(g) * kG * hd + ctid,
                         p.q + static_cast<int64_t>(g + 1) * kG * hd, want,
                         [&](int jj, float v) { sraw[ctid + jj * kC] = v; }) &&
         ok;
    bar_sync(kConsumerBar, kC);
    for (int e = ctid; e < kG * hd; e += kC) {
      const int h = e / hd, i = e - h * hd;
      sq[e] = rope_at(sraw + h * hd, i, p.rot_dim, p.rtc, p.rts);
    }
    bar_sync(kConsumerBar, kC);
    float q[kG][kPL], acc[kG][kPL], m[kG], lsum[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      m[h] = -INFINITY;
      lsum[h] = 0.f;
#pragma unroll
      for (int c = 0; c < kPL; ++c) {
        q[h][c] = sq[h * hd + c0 + c] * p.att_scale;
        acc[h][c] = 0.f;
      }
    }
    const float* kh = kcl + static_cast<int64_t>(g) * p.max_seq * hd + c0;
    const float* vh = vcl + static_cast<int64_t>(g) * p.max_seq * hd + c0;
    // one position's update of the running (m, l, acc) of every head
    auto update = [&](const float (&kr)[kPL], const float (&vr)[kPL]) {
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
        lsum[h] = fmaf(lsum[h], alpha, pr);
#pragma unroll
        for (int c = 0; c < kPL; ++c) acc[h][c] = fmaf(acc[h][c], alpha, pr * vr[c]);
        m[h] = mn;
      }
    };
    // the cached positions (pos, when it is in this item, comes last)
    const int64_t pe = has_pos ? p.pos : p1;
    for (int64_t r0 = p0 + warp; r0 < pe; r0 += 2 * kAttWarpsC) {
      // two positions per round: both rows' loads in flight together
      float kr[2][kPL], vr[2][kPL];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int64_t r = min(r0 + u * kAttWarpsC, pe - 1);
#pragma unroll
        for (int c = 0; c < kPL; c += 4) {
          const float4 a = *reinterpret_cast<const float4*>(kh + r * hd + c);
          const float4 b = *reinterpret_cast<const float4*>(vh + r * hd + c);
          kr[u][c] = a.x; kr[u][c + 1] = a.y; kr[u][c + 2] = a.z; kr[u][c + 3] = a.w;
          vr[u][c] = b.x; vr[u][c + 1] = b.y; vr[u][c + 2] = b.z; vr[u][c + 3] = b.w;
        }
      }
      update(kr[0], vr[0]);
      if (r0 + kAttWarpsC < pe) update(kr[1], vr[1]);
    }
    if (has_pos) {
      // k (rotated) and v of pos from the QKV phase; into the caches; then
      // warp 0 takes the row
      ok = poll_stamped<1>(p.k + static_cast<int64_t>(g) * hd + ctid,
                           p.k + static_cast<int64_t>(g + 1) * hd, want,
                           [&](int, float v) { sraw[ctid] = v; }) &&
           ok;
      ok = poll_stamped<1>(p.v + static_cast<int64_t>(g) * hd + ctid,
                           p.v + static_cast<int64_t>(g + 1) * hd, want,
                           [&](int, float v) { sraw[hd + ctid] = v; }) &&
           ok;
      bar_sync(kConsumerBar, kC);
      const int64_t row = (static_cast<int64_t>(g) * p.max_seq + p.pos) * hd;
      for (int i = ctid; i < hd; i += kC) {
        const float kr = rope_at(sraw, i, p.rot_dim, p.rtc, p.rts);
        const float vr = sraw[hd + i];
        skv[i] = kr;
        skv[hd + i] = vr;
        p.kc[l][row + i] = kr;
        p.vc[l][row + i] = vr;
      }
      bar_sync(kConsumerBar, kC);
      if (warp == 0) {
        float kr[kPL], vr[kPL];
#pragma unroll
        for (int c = 0; c < kPL; ++c) {
          kr[c] = skv[c0 + c];
          vr[c] = skv[hd + c0 + c];
        }
        update(kr, vr);
      }
    }
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      if (lane == 0) {
        smm[warp * 4 + h] = m[h];
        sml[warp * 4 + h] = lsum[h];
      }
#pragma unroll
      for (int c = 0; c < kPL; ++c) sacc[(warp * kG + h) * hd + c0 + c] = acc[h][c];
    }
    bar_sync(kConsumerBar, kC);
    for (int e = ctid; e < kG * hd; e += kC) {
      const int h = e / hd, i = e - h * hd;
      float M = -INFINITY;
      for (int w = 0; w < kAttWarpsC; ++w) M = fmaxf(M, smm[w * 4 + h]);
      float a = 0.f, L = 0.f;
      if (M != -INFINITY) {
        for (int w = 0; w < kAttWarpsC; ++w) {
          const float f = expf(smm[w * 4 + h] - M);   // 0 for a warp with no position
          a = fmaf(sacc[(w * kG + h) * hd + i], f, a);
          L = fmaf(sml[w * 4 + h], f, L);
        }
      }
      Word* dst = p.part + ((static_cast<int64_t>(g) * p.chunks + j) * kG + h) * (hd + 2);
      st_word(dst + i, a, want);
      if (i == 0) {
        st_word(dst + hd, M, want);
        st_word(dst + hd + 1, L, want);
      }
    }
    bar_sync(kConsumerBar, kC);   // shared memory is reused by the next item
  }
  return ok;
}

// Step 2: attention outputs [o0, o1) of layer l from the items' partials,
// min(kAttMergeBatch, per) outputs per round (the staging-buffer floats the
// host reserves: three per output of a round and chunk); out = sum_j
// e^(m_j - M) acc_j / sum_j e^(m_j - M) l_j (M = max_j m_j).
__device__ __forceinline__ bool att_merge(const ChainParams& p, int l, float* sm, int ctid) {
  const unsigned want = static_cast<unsigned>(4 * l + 1);
  const int hd = p.head_dim, G = p.n_q_heads / p.n_kv_heads, C = p.chunks;
  const int64_t n_out = static_cast<int64_t>(p.n_q_heads) * hd;
  const int64_t per = (n_out + gridDim.x - 1) / gridDim.x;
  const int64_t o0 = blockIdx.x * per, o1 = min(o0 + per, n_out);
  const int bmax = static_cast<int>(min(static_cast<int64_t>(kAttMergeBatch), per));
  float* sa = sm;                                   // [bmax][C] acc
  float* smv = sa + bmax * C;                       // [bmax][C] m
  float* slv = smv + bmax * C;                      // [bmax][C] l
  bool ok = true;
  for (int64_t b0 = o0; b0 < o1; b0 += bmax) {
    const int nb = static_cast<int>(min(static_cast<int64_t>(bmax), o1 - b0));
    for (int t0 = 0; t0 < nb * C; t0 += kC) {
      const int t = t0 + ctid;
      if (t < nb * C) {
        const int k = t / C, j = t - k * C;
        const int64_t o = b0 + k;
        const int hq = static_cast<int>(o / hd), i = static_cast<int>(o - static_cast<int64_t>(hq) * hd);
        const int g = hq / G, h = hq - g * G;
        const Word* src = p.part + ((static_cast<int64_t>(g) * C + j) * G + h) * (hd + 2);
        const Word* a[3] = {src + i, src + hd, src + hd + 1};
        float v[3];
        ok = poll_words<3>(a, 3, want, v) && ok;
        sa[t] = v[0];
        smv[t] = v[1];
        slv[t] = v[2];
      }
    }
    bar_sync(kConsumerBar, kC);
    // warp w combines outputs w, w + 10, ...; lane c takes chunks c, c + 32, ...
    // (lane sums in order, then the warp's shuffle tree: a fixed order)
    const int warp = ctid >> 5, lane = ctid & 31;
    for (int k = warp; k < nb; k += kAttWarpsC) {
      const float* ma = smv + k * C;
      float M = -INFINITY;
      for (int j = lane; j < C; j += 32) M = fmaxf(M, ma[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
      float a = 0.f, L = 0.f;
      for (int j = lane; j < C; j += 32) {
        const float f = ma[j] != -INFINITY ? expf(ma[j] - M) : 0.f;   // 0: an empty chunk
        a = fmaf(sa[k * C + j], f, a);
        L = fmaf(slv[k * C + j], f, L);
      }
      a = warp_sum(a);
      L = warp_sum(L);
      if (lane == 0) st_word(p.att + b0 + k, a / L, want);
    }
    bar_sync(kConsumerBar, kC);
  }
  return ok;
}

// Both steps with the shapes the fused path takes (head_dim / group).
__device__ __forceinline__ bool att_fused(const ChainParams& p, int l, float* sm, int ctid) {
  const int G = p.n_q_heads / p.n_kv_heads;
  bool ok;
  switch (p.head_dim * 8 + G) {
    case 256 * 8 + 1: ok = att_split<8, 1>(p, l, sm, ctid); break;
    case 256 * 8 + 2: ok = att_split<8, 2>(p, l, sm, ctid); break;
    case 128 * 8 + 1: ok = att_split<4, 1>(p, l, sm, ctid); break;
    case 128 * 8 + 2: ok = att_split<4, 2>(p, l, sm, ctid); break;
    default: ok = att_split<4, 4>(p, l, sm, ctid); break;   // 128 * 8 + 4
  }
  return att_merge(p, l, sm, ctid) && ok;
}

// Stages the seq-1 attention output for the O projection: query head i / hd
// takes kv head (i / hd) / group, i.e. column i reads v[(head / group) * hd + i % hd].
template <int kJ>
__device__ __forceinline__ bool stage_gather(const Ring& R, int US, const Word* v, unsigned want,
                                             int64_t n, int hd, int group, int ctid) {
  bool ok = true;
  // 32-bit index arithmetic (n <= 4 * 20480): the 64-bit division it replaces
  // is a long software sequence on the boundary's critical path
  const unsigned uhd = static_cast<unsigned>(hd), ugroup = static_cast<unsigned>(group);
  for (int64_t b0 = ctid; b0 < n; b0 += static_cast<int64_t>(kJ) * kC) {
    unsigned pending = 0;
    const Word* at[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int64_t i = b0 + static_cast<int64_t>(j) * kC;
      at[j] = v;
      if (i < n) {
        const unsigned ui = static_cast<unsigned>(i);
        const unsigned head = ui / uhd;
        at[j] = v + (head / ugroup) * uhd + (ui - head * uhd);
        pending |= 1u << j;
      }
    }
    long long t0 = 0;
    bool first = true;
    while (pending) {
      Word w[kJ];
#pragma unroll
      for (int j = 0; j < kJ; ++j) w[j] = (pending >> j & 1u) ? ld_word(at[j]) : 0ull;
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        if ((pending >> j & 1u) && stamp_of(w[j]) == want) {
          int u, l;
          UnitQ4K::unit_of(b0 + static_cast<int64_t>(j) * kC, u, l);
          R.xs[l * US + u] = value_of(w[j]);
          pending &= ~(1u << j);
        }
      }
      if (!pending) break;
      if (first) {
        t0 = clock64();
        first = false;
      } else if (clock64() - t0 > kWaitCycles) {
        atomicOr(&g_err_chain, kErrFullWait);
        ok = false;
        break;
      }
    }
  }
  return ok;
}

// Builds the input vector of phase ph into R.xs, then counts this CTA's
// prologue as finished.  Inlined, like the decode loop below: a call would
// save and restore the caller's live registers through local memory at every
// phase boundary, on the critical path (measured: 1316 -> 1172 us per
// 34-layer token once both are inlined).  kWide: hidden > 8 * 320 (16 values
// per thread in the residual / norm step); a separate instantiation, so the
// common case carries none of its registers.
template <bool kWide, bool kKV>
__device__ __forceinline__ bool chain_prologue(const ChainParams& p, int ph, const Ring& R,
                                            float* wsum, volatile int* gate, bool q6, int ctid,
                                            int C) {
  const int l = ph >> 2, kind = ph & 3;
  const ChainLayer& L = p.L[l];
  const KindPlan& kp = p.kp[kind];
  const int US = red_stride(kp.U);
  const unsigned prev = static_cast<unsigned>(ph);   // stamp of the previous phase's outputs
  bool ok = true;
  // the keeper overwrites hin[l & 1] (QKV; last read by GU(l - 2)) or h1[l & 1]
  // (GU; last read by QKV(l - 1)): load that count now, check it before the
  // stores, so its latency hides behind the loads of the vectors
  unsigned war_seen = gridDim.x;
  if (blockIdx.x == gridDim.x - 1 && (kind == PH_QKV || kind == PH_GU)) {
    const int w = kind == PH_QKV ? 4 * l - 6 : 4 * l - 4;
    if (w >= 0) war_seen = ld_acquire_gpu(p.prologues + w);
  }
  // every consumer thread of this CTA is done with R.xs of the previous phase
  bar_sync(kConsumerBar, C);
  if (kind == PH_QKV || kind == PH_GU) {
    const Word* base;
    const float* base_plain = nullptr;
    const Word* add = nullptr;
    const float *wa = nullptr, *wn;
    unsigned base_stamp = 0, add_stamp = prev;
    Word* store;
    int war;
    if (kind == PH_QKV) {
      // h = layer input: the caller's h, or h1 + norm(f) of the previous layer;
      // the keeper CTA keeps it in hin[l & 1] for the GU residual
      base = l ? p.h1 + ((l - 1) & 1) * p.H : nullptr;
      base_stamp = static_cast<unsigned>(4 * l - 1);
      base_plain = l ? nullptr : p.h;
      add = l ? p.f : nullptr;
      wa = l ? p.L[l - 1].w_pff : nullptr;
      wn = L.w_in;
      store = blockIdx.x == gridDim.x - 1 ? p.hin + (l & 1) * p.H : nullptr;
      war = 4 * l - 6;   // GU(l - 2) read hin[l & 1] last
    } else {
      // h1 = h + rms_norm(o, w_post_attn) (or h + o); the keeper keeps it in h1[l & 1]
      base = p.hin + (l & 1) * p.H;
      base_stamp = static_cast<unsigned>(4 * l + 1);
      add = p.o;
      wa = L.w_pa;
      wn = L.w_pf;
      store = blockIdx.x == gridDim.x - 1 ? p.h1 + (l & 1) * p.H : nullptr;
      war = 4 * l - 4;   // QKV(l - 1) read h1[l & 1] last
    }
    if constexpr (kWide)
      ok = resnorm_stage<16, false>(p, R, wsum, base, base_stamp, base_plain, add, add_stamp, wa,
                                    wn, store, static_cast<unsigned>(ph + 1), war, war_seen, US,
                                    ctid);
    else
      ok = resnorm_stage<8, true>(p, R, wsum, base, base_stamp, base_plain, add, add_stamp, wa,
                                  wn, store, static_cast<unsigned>(ph + 1), war, war_seen, US,
                                  ctid);
  } else if (kind == PH_O) {
    if constexpr (kKV) {
      // attention of layer l inside this launch (the staging buffer is free
      // until the O vector is staged below)
      if (p.fused_att) ok = att_fused(p, l, R.xs, ctid);
      ok = stage_stamped<UnitQ4K, 16>(R, US, p.att, prev, kp.K, ctid) && ok;
    }
    else
      ok = stage_gather<8>(R, US, p.v, prev, kp.K, p.head_dim, p.n_q_heads / p.n_kv_heads, ctid);
  } else if (q6) {
    ok = stage_stamped<UnitQ6K, 16>(R, US, p.m, prev, kp.K, ctid);
  } else {
    ok = stage_stamped<UnitQ4K, 16>(R, US, p.m, prev, kp.K, ctid);
  }
  bar_sync(kConsumerBar, C);
  // this CTA has read everything its prologue needed
  if (ctid == 0) {
    red_release_gpu_add(p.prologues + ph, 1u);
    *gate = ph + 1;   // the producer may copy the rest of phase ph's tiles
  }
  return ok;
}

// Final residual on the keeper CTA: h = h1 + rms_norm(f, w_post_ffn) (or h1 + f),
// then, when hn is set, hn = rms_norm(h, w_final) (the model's final norm, so
// that the next kernel reads its input straight from this launch).
template <int kJ>
__device__ __noinline__ bool chain_final(const ChainParams& p, float* wsum, int ctid, int C) {
  const int Ll = p.n_layers - 1;
  const bool post = p.post_norms != 0;
  float hv[kJ], fv[kJ], wp[kJ], wf[kJ];
  const Word* h1 = p.h1 + (Ll & 1) * p.H;
  // the norm weights first: their loads overlap the polls below
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int64_t i = ctid + static_cast<int64_t>(j) * kC;
    wp[j] = (i < p.H && post) ? p.L[Ll].w_pff[i] : 0.f;
    wf[j] = (i < p.H && p.hn) ? p.w_final[i] : 0.f;
  }
  // every CTA is past its last prologue, so none still reads the caller's h
  bool ok = wait_prologues(p, 4 * p.n_layers - 1);
#pragma unroll
  for (int j = 0; j < kJ; ++j) hv[j] = fv[j] = 0.f;
  ok = poll_stamped<kJ>(h1 + ctid, h1 + p.H, static_cast<unsigned>(4 * Ll + 3),
                        [&](int j, float v) { hv[j] = v; }) &&
       ok;
  ok = poll_stamped<kJ>(p.f + ctid, p.f + p.H, static_cast<unsigned>(4 * Ll + 4),
                        [&](int j, float v) { fv[j] = v; }) &&
       ok;
  float inv = 1.f;
  if (post) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kJ; ++j) ss = fmaf(fv[j], fv[j], ss);
    inv = 1.0f / sqrtf(block_sum(ss, wsum, ctid, C) / static_cast<float>(p.H) + p.eps);
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    const int64_t i = ctid + static_cast<int64_t>(j) * kC;
    if (i < p.H) {
      hv[j] = __fadd_rn(hv[j], post ? __fmul_rn(__fmul_rn(fv[j], inv), wp[j]) : fv[j]);
      p.h[i] = hv[j];
      ss = fmaf(hv[j], hv[j], ss);
    }
  }
  if (p.hn) {
    const float inv_f =
        1.0f / sqrtf(block_sum(ss, wsum, ctid, C) / static_cast<float>(p.H) + p.eps);
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int64_t i = ctid + static_cast<int64_t>(j) * kC;
      if (i < p.H) p.hn[i] = __fmul_rn(__fmul_rn(hv[j], inv_f), wf[j]);
    }
  }
  return ok;
}

// The decode loop of every phase, fed with scalars only: it rebuilds the ring
// from the dynamic shared-memory base, so no structure goes through local
// memory (UnitChain serves both formats).  Returns the new ring position
// (s, ph, n) packed with an ok bit.
__device__ __forceinline__ unsigned long long chain_consume(
    int fmt, int epi, int nseg, int rows0, int rows1, int rows2, int tiles0, int tiles1,
    int tiles2, int T, int T2, int n1, int U, int G, int row_bytes, int n_tiles, unsigned S,
    unsigned stage_bytes,
    unsigned red_floats, unsigned xs_floats, unsigned pos_s, unsigned pos_ph, unsigned pos_n,
    int ctid, int C) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R = make_ring(smem, S, stage_bytes, red_floats, xs_floats);
  Phase P;
  P.fmt = fmt;
  P.epi = epi;
  P.nseg = nseg;
  P.seg[0] = Seg{nullptr, nullptr, rows0, tiles0};
  P.seg[1] = Seg{nullptr, nullptr, rows1, tiles1};
  P.seg[2] = Seg{nullptr, nullptr, rows2, tiles2};
  P.W2 = nullptr;
  P.K = 0;
  P.row_bytes = row_bytes;
  P.row_stride = row_bytes;
  P.B = 1;
  P.U = U;
  P.G = G;
  P.T = T;
  P.T2 = T2;
  P.n1 = n1;
  P.n_tiles = n_tiles;
  P.cta0 = 0;
  P.ncta = static_cast<int>(gridDim.x);
  RingPos pos;
  pos.s = pos_s;
  pos.ph = pos_ph;
  pos.n = pos_n;
  const bool ok = consume_phase<UnitChain, false, false>(P, R, pos, XOfPlain{nullptr, 0}, ctid, C,
                                                         &g_err_chain);
  return static_cast<unsigned long long>(pos.s) | (static_cast<unsigned long long>(pos.ph) << 8) |
         (static_cast<unsigned long long>(pos.n) << 16) | (ok ? (1ull << 63) : 0ull);
}

// Asks L2 to fetch n bytes at w (skipped unless 16-byte aligned and sized).
__device__ __forceinline__ void prefetch_l2(const float* w, int64_t n) {
  if (w && (reinterpret_cast<uintptr_t>(w) & 15) == 0 && n % 16 == 0)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(w),
                 "r"(static_cast<unsigned>(n))
                 : "memory");
}

// Holds the copy of tile j >= kGateTiles of launch phase i (> 0) until this
// CTA's consumers have finished that phase's prologue.  Bounded.
struct ChainGate {
  volatile int* done;   // last finished prologue: absolute phase + 1
  int begin;            // absolute index of launch phase 0
  __device__ __forceinline__ bool operator()(int i, int j) const {
    const int want = begin + i + 1;
    if (i == 0 || j < kGateTiles || *done >= want) return true;
    const long long t0 = clock64();
    while (*done < want) {
      if (clock64() - t0 > kWaitCycles) return false;
      __nanosleep(32);
    }
    return true;
  }
};

// ------------------------------------------------------------------ kernel
template <bool kWide, bool kKV>
__global__ void __launch_bounds__(kRoleThreads + kMaxConsumers, 1)
    chain_kernel(const __grid_constant__ ChainParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  // A kernel launched after this one with a programmatic dependency may be
  // scheduled from now on: it waits for this grid's completion before it
  // touches data of this launch, and its blocks only find room on SMs whose
  // chain CTA has exited, so e.g. the next matvec's weight copies overlap
  // the final residual of the keeper CTA instead of following it.
  pdl_launch_dependents();
  const Ring R = make_ring(smem, p.S, p.stage_bytes, p.red_floats, p.xs_floats);
  float* wsum = reinterpret_cast<float*>(smem + ring_smem_bytes(p.S, p.stage_bytes, p.red_floats,
                                                                 p.xs_floats));
  // the last prologue this CTA finished (phase + 1), read by the producer
  volatile int* gate = reinterpret_cast<volatile int*>(wsum + 64);
  const int C = static_cast<int>(blockDim.x) - kRoleThreads;
  if (threadIdx.x == 0) {
    ring_init(R, C / 32);
    *gate = 0;
  }
  __syncthreads();
  const ChainPhases<kKV> phases{&p};

  if (threadIdx.x < kProducerThreads) {
    if (threadIdx.x == 0) {
      // warm L2 with this CTA's share of the (small, static) norm weights
      for (int l = blockIdx.x; l < p.n_layers; l += gridDim.x) {
        prefetch_l2(p.L[l].w_in, p.H * 4);
        prefetch_l2(p.L[l].w_pa, p.H * 4);
        prefetch_l2(p.L[l].w_pf, p.H * 4);
        prefetch_l2(p.L[l].w_pff, p.H * 4);
      }
      if (blockIdx.x == gridDim.x - 1) prefetch_l2(p.w_final, p.H * 4);
      if (kKV && !p.fused_att)   // launches per layer: ungated (see kGateTiles)
        run_producer(typename ChainPhases<kKV>::Range{&phases, p.ph_begin, p.ph_end}, R,
                     &g_err_chain);
      else
        run_producer(typename ChainPhases<kKV>::Range{&phases, p.ph_begin, p.ph_end}, R,
                     &g_err_chain,
                     ChainGate{gate, p.ph_begin});
    }
    return;
  }

  RingPos pos;
  if (threadIdx.x < kRoleThreads) {
    // ---------------- reducer: sums and stamped stores, phase after phase
    for (int ph = p.ph_begin; ph < p.ph_end; ++ph) {
      const Phase P = phases.get(ph);
      // (one load, normally already satisfied; it overlaps the consumers'
      // work on the phase's first tile).  A phase before this launch's first
      // ran in an earlier launch, which has finished.
      if (ph - 3 >= p.ph_begin && !wait_prologues(p, ph - 3)) return;
      if (!reduce_phase(P, R, pos, EpiStamped{ph}, &g_err_chain)) return;
    }
    return;
  }

  // ---------------- consumers
  const int ctid = static_cast<int>(threadIdx.x) - kRoleThreads;
  const bool down_q6k = p.kp[PH_DOWN].fmt == 14;
  for (int ph = p.ph_begin; ph < p.ph_end; ++ph) {
    const Phase P = phases.get(ph);
    const bool q6 = (ph & 3) == PH_DOWN && down_q6k;
    if (!chain_prologue<kWide, kKV>(p, ph, R, wsum, gate, q6, ctid, C)) return;
    const unsigned long long r = chain_consume(
        P.fmt, P.epi, P.nseg, static_cast<int>(P.seg[0].rows), static_cast<int>(P.seg[1].rows),
        static_cast<int>(P.seg[2].rows), P.seg[0].tiles, P.seg[1].tiles, P.seg[2].tiles, P.T,
        P.T2, P.n1, P.U, P.G, static_cast<int>(P.row_bytes), P.n_tiles, p.S, p.stage_bytes,
        p.red_floats,
        p.xs_floats, pos.s, pos.ph, pos.n, ctid, C);
    pos.s = static_cast<uint32_t>(r & 0xFFu);
    pos.ph = static_cast<uint32_t>((r >> 8) & 1u);
    pos.n = static_cast<uint32_t>((r >> 16) & 0xFFFFFFFFu);
    if ((r >> 63) == 0) return;
  }
  if (p.ph_end == 4 * p.n_layers && blockIdx.x == gridDim.x - 1) {
    if constexpr (kWide)
      chain_final<16>(p, wsum, ctid, C);
    else
      chain_final<8>(p, wsum, ctid, C);
  }
}

// Self-test of the failure path: the chain's stamped-word poll on a word
// whose stamp nothing ever writes (the word is cleared by the host first), with
// the given wait limit.  The poll gives up, records kErrFullWait and the
// kernel returns; nothing else is in flight.
__global__ void selftest_poll_kernel(const Word* word, long long limit) {
  if (threadIdx.x != 0) return;
  float sink = 0.f;
  poll_stamped<1>(word, word + 1, 1u, [&](int, float v) { sink = v; }, limit);
  if (sink != 0.f) atomicOr(&g_err_chain, 0u);   // keeps the poll's result live
}

cudaError_t launch_selftest_poll(void* word8, long long limit, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(word8, 0, sizeof(Word), st);
  if (e != cudaSuccess) return e;
  selftest_poll_kernel<<<1, 32, 0, st>>>(static_cast<const Word*>(word8), limit);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host side
static int64_t align64(int64_t n) { return (n + 63) / 64 * 64; }

// Workspace (8-byte words): q, k, v [4 * hidden each, enough for q_dim and
// kv_dim <= 4 * hidden], o [hidden], f [hidden], m [inter], hin [2 * hidden],
// h1 [2 * hidden], then one prologue counter per phase (4 * kMaxLayers).
size_t chain_workspace_bytes(int64_t hidden, int64_t inter) {
  if (hidden <= 0 || inter <= 0) return 0;
  const int64_t words = 3 * align64(4 * hidden) + 2 * align64(hidden) + align64(inter) +
                        2 * align64(2 * hidden);
  return static_cast<size_t>(words) * sizeof(Word) + 4 * kMaxLayers * sizeof(unsigned) + 256;
}

unsigned read_clear_chain_errors() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_chain, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_err_chain, &z, sizeof(z));
  return v;
}

}  // namespace qws

using namespace qws;

namespace {

// One prepared chain: parameters, kernel and launch shape.  Launches of
// phase ranges of one token share it (and the workspace, cleared once).
struct ChainLaunch {
  ChainParams p;
  const void* kfn = nullptr;
  int grid = 0, threads = 0;
  size_t smem = 0, clear_bytes = 0;
};

// Argument checks, parameters and launch shape; ws holds the chain's words.
// kv: the O phase reads an attention output (ChainParams::att) instead of
// gathering v (the decode step over a KV cache).
qws_status chain_prepare(const char* fn, const qws_layer* layers, int n_layers, float* h,
                         const qws_dims* d, void* ws, size_t ws_bytes, bool kv, ChainLaunch& cl,
                         std::string& err, uint32_t min_xs = 0) {
  auto bad = [&](qws_status s, const char* m) {
    err = std::string(fn) + ": " + m;
    return s;
  };
  if (!layers || !h || !d || !ws) return bad(QWS_ERR_NULL, "NULL argument");
  if (n_layers < 1 || n_layers > kMaxLayers)
    return bad(QWS_ERR_SHAPE, "n_layers must be in [1, 64]");
  const int64_t H = d->hidden, I = d->inter;
  if (d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 ||
      d->n_q_heads % d->n_kv_heads)
    return bad(QWS_ERR_SHAPE, "bad head counts");
  const int64_t QD = static_cast<int64_t>(d->n_q_heads) * d->head_dim;
  const int64_t KD = static_cast<int64_t>(d->n_kv_heads) * d->head_dim;
  auto ok_dim = [](int64_t v) { return v > 0 && v % 256 == 0 && v <= 20480; };
  if (!ok_dim(H) || !ok_dim(I) || !ok_dim(QD) || KD % 64 || KD <= 0 || QD > 4 * H || KD > 4 * H)
    return bad(QWS_ERR_SHAPE,
               "hidden, inter, q_dim must be multiples of 256 in (0, 20480], "
               "q_dim and kv_dim <= 4 * hidden");
  if (H > kMaxChainHidden) return bad(QWS_ERR_SHAPE, "hidden must be <= 5120");
  if (!(d->eps >= 0.f)) return bad(QWS_ERR_SHAPE, "eps must be >= 0");
  if (reinterpret_cast<uintptr_t>(h) % 4 || reinterpret_cast<uintptr_t>(ws) % 16)
    return bad(QWS_ERR_ALIGN, "h must be 4-byte and ws 16-byte aligned");
  if (ws_bytes < chain_workspace_bytes(H, I)) return bad(QWS_ERR_WORKSPACE, "workspace too small");
  ChainParams& p = cl.p;
  std::memset(&p, 0, sizeof(p));
  for (int l = 0; l < n_layers; ++l) {
    const qws_layer& L = layers[l];
    const void* ws8[7] = {L.Wq, L.Wk, L.Wv, L.Wo, L.Wg, L.Wu, L.Wd};
    for (const void* w : ws8) {
      if (!w) return bad(QWS_ERR_NULL, "a weight pointer is NULL");
      if (reinterpret_cast<uintptr_t>(w) % 16)
        return bad(QWS_ERR_ALIGN, "weights must be 16-byte aligned");
    }
    const float* nw[4] = {L.w_in, L.w_post_attn, L.w_pre_ffn, L.w_post_ffn};
    for (int i = 0; i < 4; ++i) {
      if (!nw[i] && (i == 0 || i == 2 || d->post_norms))
        return bad(QWS_ERR_NULL, "a norm weight pointer is NULL");
      if (reinterpret_cast<uintptr_t>(nw[i]) % 4)
        return bad(QWS_ERR_ALIGN, "norm weights must be 4-byte aligned");
    }
    if (L.fmt_qkv != QWS_Q4_K || L.fmt_o != QWS_Q4_K || L.fmt_gu != QWS_Q4_K ||
        (L.fmt_down != QWS_Q4_K && L.fmt_down != QWS_Q6_K) || L.fmt_down != layers[0].fmt_down)
      return bad(QWS_ERR_FORMAT,
                 "q/k/v/o/gate/up must be Q4_K; down Q4_K or Q6_K (same in "
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
  p.ph_begin = 0;
  p.ph_end = 4 * n_layers;

  // workspace carve-up (8-byte {value, stamp} words), then the counter
  Word* w = static_cast<Word*>(ws);
  p.q = w;
  w += align64(4 * H);
  p.k = w;
  w += align64(4 * H);
  p.v = w;
  w += align64(4 * H);
  p.o = w;
  w += align64(H);
  p.f = w;
  w += align64(H);
  p.m = w;
  w += align64(I);
  p.hin = w;
  w += align64(2 * H);
  p.h1 = w;
  w += align64(2 * H);
  p.prologues = reinterpret_cast<unsigned*>(w);
  const size_t clear_bytes =
      static_cast<size_t>(reinterpret_cast<uint8_t*>(w) - static_cast<uint8_t*>(ws)) +
      4 * kMaxLayers * sizeof(unsigned);

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
      err = "" + why;
      return QWS_ERR_SHAPE;
    }
    // all kinds run with the same thread count: C = kMaxConsumers
    // One-segment phases end in a balanced round: whole rounds of T-row
    // tiles (one per CTA), then the remaining rows in tiles of T2 <= T rows,
    // at most one per CTA.  With T-row tiles alone a phase of R rows takes
    // ceil(R / (T * sms)) tile times on the CTAs that hold an extra tile.
    // T2 is a multiple of the rows that keep every tile's first byte 16-byte
    // aligned (the bulk copies need it; T is one already).
    int T2 = tp.T, n1 = 0x7FFFFFFF;
    if (i != PH_QKV) {
      const int64_t R = kinds[i].rows;
      const int64_t RB = row_bytes_of(kinds[i].fmt, kinds[i].K);
      const int64_t align = 16 / gcd64(RB, 16);
      const int64_t full = R / (static_cast<int64_t>(tp.T) * sms);
      const int64_t rem = R - full * tp.T * sms;
      n1 = static_cast<int>(full * sms);
      const int64_t t2 = ((rem + sms - 1) / sms + align - 1) / align * align;
      T2 = rem > 0 ? static_cast<int>(std::min<int64_t>(tp.T, t2)) : tp.T;
    }
    p.kp[i] = KindPlan{kinds[i].fmt, tp.U,  tp.G, tp.T, T2, n1, kinds[i].K,
                       row_bytes_of(kinds[i].fmt, kinds[i].K)};
    stage_need = std::max(stage_need, tp.stage_need);
    red = std::max(red, tp.red_floats);
    xs = std::max<uint32_t>(xs, unit_weights(kinds[i].fmt) * red_stride(tp.U));
  }
  p.stage_bytes = round_up(stage_need + 16, 128);
  p.red_floats = red;
  p.xs_floats = std::max(xs, min_xs);   // the fused attention's scratch, when larger
  const size_t tail = 64 * sizeof(float) + 16;   // warp sums, producer gate
  // Ring depth: at most kChainStages.  A deeper ring prefetches more of the
  // next phase, and that DRAM traffic slows the L2 loads on every CTA's
  // critical path at each phase boundary (measured on GB300: 7 stages 1416,
  // 6: 1336, 4: 1291, 3: 1315, 2: 1503 us per 34-layer token).
  p.S = kChainStages;
  while (p.S > 2 && ring_smem_bytes(p.S, p.stage_bytes, p.red_floats, p.xs_floats) + tail >
                        kSmemBudget)
    --p.S;
  cl.smem = ring_smem_bytes(p.S, p.stage_bytes, p.red_floats, p.xs_floats) + tail;
  cl.threads = kRoleThreads + kMaxConsumers;
  cl.clear_bytes = clear_bytes;

  // hidden > 8 * 320 takes the wide prologue instantiation
  const bool wide = p.H > 8 * static_cast<int64_t>(kMaxConsumers);
  cl.kfn = wide ? (kv ? reinterpret_cast<const void*>(chain_kernel<true, true>)
                      : reinterpret_cast<const void*>(chain_kernel<true, false>))
                : (kv ? reinterpret_cast<const void*>(chain_kernel<false, true>)
                      : reinterpret_cast<const void*>(chain_kernel<false, false>));
  // set on every launch (cheap next to the chain): nothing cached per device
  int dev = 0;
  cudaGetDevice(&dev);
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncSetAttribute(cl.kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  int bps = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, cl.kfn, cl.threads, cl.smem);
  if (bps < 1) {
    err = std::string(fn) + ": kernel does not fit on an SM";
    return QWS_ERR_CUDA;
  }
  cl.grid = sms;  // one CTA per SM: all co-resident (cooperative launch)
  return QWS_OK;
}

// Stamps left by an earlier token must not look current: clear every word
// (once per token, before its first launch).
cudaError_t chain_clear(const ChainLaunch& cl, void* ws, cudaStream_t st) {
  return cudaMemsetAsync(ws, 0, cl.clear_bytes, st);
}

// Runs phases [ph_begin, ph_end) of the token.
cudaError_t chain_run(ChainLaunch& cl, int ph_begin, int ph_end, cudaStream_t st) {
  cl.p.ph_begin = ph_begin;
  cl.p.ph_end = ph_end;
  void* args[] = {&cl.p};
  return cudaLaunchCooperativeKernel(cl.kfn, dim3(cl.grid), dim3(cl.threads), args, cl.smem, st);
}

}  // namespace

// Argument checks and launch (called by qws_decode_chain in abi.cu); kept in
// this translation unit with the workspace layout it depends on.
qws_status qws::decode_chain(const qws_layer* layers, int n_layers, float* h,
                                 const qws_dims* d, void* ws, size_t ws_bytes, cudaStream_t st,
                                 std::string& err, const float* w_final, float* hn,
                                 const char* fn) {
  if (hn || w_final) {
    if (!hn || !w_final) {
      err = std::string(fn) + ": w_final and hn must both be given";
      return QWS_ERR_NULL;
    }
    if (reinterpret_cast<uintptr_t>(hn) % 4 || reinterpret_cast<uintptr_t>(w_final) % 4) {
      err = std::string(fn) + ": w_final and hn must be 4-byte aligned";
      return QWS_ERR_ALIGN;
    }
    // the keeper writes h[i] and hn[i] from the same thread, h first
    const uintptr_t a = reinterpret_cast<uintptr_t>(h), b = reinterpret_cast<uintptr_t>(hn);
    const uintptr_t n = d ? static_cast<uintptr_t>(std::max<int64_t>(d->hidden, 0)) * 4 : 0;
    if (h && a < b + n && b < a + n) {
      err = std::string(fn) + ": hn must not overlap h";
      return QWS_ERR_SHAPE;
    }
  }
  ChainLaunch cl;
  const qws_status rc = chain_prepare(fn, layers, n_layers, h, d, ws, ws_bytes, false, cl, err);
  if (rc != QWS_OK) return rc;
  cl.p.w_final = w_final;
  cl.p.hn = hn;
  cudaError_t e = chain_clear(cl, ws, st);
  if (e == cudaSuccess) e = chain_run(cl, 0, 4 * n_layers, st);
  if (e != cudaSuccess) {
    err = std::string(fn) + ": " + cudaGetErrorName(e) + " " + cudaGetErrorString(e);
    return QWS_ERR_CUDA;
  }
  return QWS_OK;
}

// ------------------------------------------------------------ KV-cache decode
// One decode step over a KV cache on the chain kernel (infer-compute README
// §Architecture, the decode path norm -> QKV -> attend -> O -> FFN).  Per
// token, in groups of at most 64 layers (the chain's parameter block), the
// chain runs in pieces between the attention steps:
//   chain   phase QKV of the group's first layer
//   per layer l of the group:
//     attention       split + merge over positions 0..pos, from the chain's
//                     stamped q, k, v words: the split rotates q and k at pos
//                     and the CTA whose positions hold pos writes k and v
//                     into the caches; the merge writes the output as
//                     stamped words (stamp 4 l + 1)
//     chain           phases O(l), gate/up(l), down(l) and QKV(l + 1) (the
//                     group's last piece ends with the final residual)
// The chain's residuals, norms and stamps carry over between its launches
// (the workspace is cleared once per group); every launch is stream-ordered
// after the attention output it reads.
namespace {

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct KvChainLayout {
  size_t chain, att, part, bytes;   // byte offsets, total
};

KvChainLayout kv_chain_layout(const qws_dims* d, int64_t max_seq) {
  KvChainLayout L{};
  const int64_t QD = static_cast<int64_t>(d->n_q_heads) * d->head_dim;
  L.chain = 0;
  L.att = align256(chain_workspace_bytes(d->hidden, d->inter));
  L.part = L.att + align256(static_cast<size_t>(QD) * sizeof(Word));
  // the standalone kernels' float partials, or the fused steps' stamped ones
  L.bytes = L.part + align256(2 * kv_attention_workspace_bytes(d->n_q_heads, d->n_kv_heads,
                                                               d->head_dim, max_seq));
  return L;
}

}  // namespace

bool qws::decode_kv_chain_fits(const qws_dims* d) {
  if (!d || d->hidden <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0)
    return false;
  const int64_t H = d->hidden;
  const int64_t QD = static_cast<int64_t>(d->n_q_heads) * d->head_dim;
  const int64_t KD = static_cast<int64_t>(d->n_kv_heads) * d->head_dim;
  return H <= kMaxChainHidden && QD <= 4 * H && KD <= 4 * H;
}

size_t qws::decode_kv_chain_workspace_bytes(const qws_dims* d, int64_t max_seq) {
  return kv_chain_layout(d, max_seq).bytes;
}

qws_status qws::decode_kv_chain(const qws_layer* layers, int n_layers, float* h,
                                const qws_dims* d, const qws_kv* kv, void* ws, size_t ws_bytes,
                                cudaStream_t st, std::string& err) {
  const KvChainLayout Lw = kv_chain_layout(d, kv->max_seq);
  if (ws_bytes < Lw.bytes) {
    err = "qws_decode_kv: workspace too small";
    return QWS_ERR_WORKSPACE;
  }
  uint8_t* base = static_cast<uint8_t*>(ws);
  Word* att = reinterpret_cast<Word*>(base + Lw.att);
  float* part = reinterpret_cast<float*>(base + Lw.part);
  const int nq = d->n_q_heads, nkv = d->n_kv_heads, hd = d->head_dim;
  auto cuda = [&](cudaError_t e, const char* what) {
    err = std::string("qws_decode_kv: ") + what + ": " + cudaGetErrorName(e) + " " +
          cudaGetErrorString(e);
    return QWS_ERR_CUDA;
  };
  // attention inside the chain's O prologue: one launch per group of layers
  const int G = nq / nkv;
  const bool fused = (hd == 256 && G <= 2) || (hd == 128 && (G == 1 || G == 2 || G == 4));
  const int64_t n_ctx = kv->pos + 1;
  const int chunks = kv_attention_splits(nkv, n_ctx);
  const int64_t n_out = static_cast<int64_t>(nq) * hd;
  const int per = static_cast<int>((n_out + device_sms() - 1) / device_sms());
  const uint32_t att_floats = static_cast<uint32_t>(
      std::max(att_split_floats(), 3 * std::min(kAttMergeBatch, per) * chunks));
  for (int g0 = 0; g0 < n_layers; g0 += kMaxLayers) {
    const int n = std::min(kMaxLayers, n_layers - g0);
    ChainLaunch cl;
    const qws_status rc = chain_prepare("qws_decode_kv", layers + g0, n, h, d, ws, Lw.att, true,
                                        cl, err, fused ? att_floats : 0u);
    if (rc != QWS_OK) return rc;
    cl.p.att = att;
    if (fused) {
      ChainParams& p = cl.p;
      p.fused_att = 1;
      for (int l = 0; l < n; ++l) {
        p.kc[l] = kv->k_caches[g0 + l];
        p.vc[l] = kv->v_caches[g0 + l];
      }
      p.max_seq = kv->max_seq;
      p.pos = kv->pos;
      p.chunks = chunks;
      p.chunk_len = static_cast<int>((n_ctx + chunks - 1) / chunks);
      p.rot_dim = kv->rot_dim;
      p.att_scale = kv->attn_scale;
      p.softcap = kv->softcap;
      p.part = reinterpret_cast<Word*>(part);
      rope_table_f32(kv->rot_dim, kv->pos, kv->rope_base, p.rtc, p.rts);
      // every stamped word of the group, the attention's included
      cudaError_t e = cudaMemsetAsync(ws, 0, Lw.bytes, st);
      if (e != cudaSuccess) return cuda(e, "clear");
      e = chain_run(cl, 0, 4 * n, st);
      if (e != cudaSuccess) return cuda(e, "chain");
      continue;
    }
    cudaError_t e = chain_clear(cl, ws, st);
    if (e != cudaSuccess) return cuda(e, "clear");
    e = chain_run(cl, 0, 1, st);   // QKV of the group's first layer
    if (e != cudaSuccess) return cuda(e, "chain");
    for (int l = 0; l < n; ++l) {
      float* kc = kv->k_caches[g0 + l];
      float* vc = kv->v_caches[g0 + l];
      const KvFuse fuse{cl.p.q, cl.p.k, cl.p.v, kc, vc, kv->pos, kv->rot_dim, kv->rope_base};
      e = launch_kv_attention(nullptr, kc, vc, nullptr, nq, nkv, hd, kv->max_seq, kv->pos + 1,
                              kv->attn_scale, kv->softcap, part, st, att,
                              static_cast<unsigned>(4 * l + 1), &fuse);
      if (e != cudaSuccess) return cuda(e, "attention");
      e = chain_run(cl, 4 * l + 1, std::min(4 * l + 5, 4 * n), st);
      if (e != cudaSuccess) return cuda(e, "chain");
    }
  }
  return QWS_OK;
}
