// engine.cuh -- the weight-streaming pipeline shared by every kernel.
//
// One CTA = one producer warp + one reducer warp + C consumer threads
// (C <= kMaxConsumers), specialised and linked only by mbarriers:
//
//  producer (one lane)  : walks the CTA's tiles in order; for each tile waits
//                         for a free ring stage, then issues 1-D bulk copies
//                         (cp.async.bulk, TMA) of the tile's packed rows from
//                         HBM into that stage; completion is counted in bytes
//                         on the stage's "full" mbarrier.  Weights never depend
//                         on activations, so the producer runs ahead of the
//                         consumers by up to the ring depth.
//  consumers            : each thread owns one 64-column lane unit of the row
//                         and one row slot g; its activations live in
//                         registers for the whole phase (formats.cuh).  For a
//                         landed stage, slot g computes rows g, g+G, ...; every
//                         thread writes one partial per row into the stage's
//                         partial buffer, then each warp arrives on the stage's
//                         "ready" mbarrier.  Consumers never wait for each other.
//  reducer (one warp)   : waits for "ready", sums each row's U partials in a
//                         fixed order (deterministic), runs the epilogue
//                         (store / GEGLU), then frees the stage ("empty").
//
// A tile is T consecutive rows of one matrix segment (QKV stacks three
// segments) or, for the gated FFN, T rows of the gate matrix followed by the
// same T rows of the up matrix in one stage.  Every wait is bounded
// (device_common.cuh); a timeout seen by any consumer ends all consumers at the
// next named barrier.
#pragma once

#include <cstdint>

#include "device_common.cuh"
#include "formats.cuh"

namespace qws {

constexpr int kMaxSeg = 3;
constexpr int kMaxConsumers = 320;
constexpr int kProducerThreads = 32;
constexpr int kReducerThreads = 32;
constexpr int kRoleThreads = kProducerThreads + kReducerThreads;  // consumers start here
constexpr int kConsumerBar = 1;     // named barrier id used by the consumer threads

enum : int { EPI_STORE = 0, EPI_GEGLU = 1, EPI_SWIGLU = 2 };   // GLU kinds read row pairs

struct Seg {
  const uint8_t* W;   // packed rows of this segment
  float* y;           // one output per row
  int64_t rows;
  int tiles;          // ceil(rows / T)
};

struct Phase {
  int fmt;            // 2 (Q4_0), 12 (Q4_K), 14 (Q6_K)
  int epi;            // EPI_STORE, or a gated pair: EPI_GEGLU / EPI_SWIGLU
  int nseg;
  Seg seg[kMaxSeg];
  const uint8_t* W2;  // gated pair: up matrix, same shape as seg[0] (the gate)
  int64_t K;          // columns (weights per row)
  int64_t row_bytes;
  int B;              // activation vectors (batch); x is [B][K], y is [B][rows]
  int U;              // lane units per row = K / 64
  int G;              // row slots per activation vector (B * G * U <= consumers)
  int T;              // rows per tile (per matrix for EPI_GEGLU)
  int T2;             // rows per tile from tile n1 on (T2 <= T): tiles [0, n1) hold
  int n1;             // T rows each, later tiles T2 rows from row n1 * T (one segment)
  int n_tiles;
  int64_t row_stride; // bytes between consecutive rows in global memory
                      // (> row_bytes when the phase covers a column slice)
  int cta0, ncta;     // CTAs [cta0, cta0 + ncta) of the grid serve this phase
};

struct TileRef {
  const uint8_t* W;   // segment's weights (row 0 of the segment)
  float* y;           // segment's outputs
  int64_t seg_rows;
  int64_t r0;         // first row of the tile within the segment
  int nrows;
};

// Segment lookup with constant indices only, so a Phase never needs to live
// in local memory.
__device__ __forceinline__ TileRef tile_ref(const Phase& P, int t) {
  TileRef tr;
  tr.W = P.seg[0].W;
  tr.y = P.seg[0].y;
  tr.seg_rows = P.seg[0].rows;
  int prev_tiles = P.seg[0].tiles;
  bool more = P.nseg > 1;
#pragma unroll
  for (int i = 1; i < kMaxSeg; ++i) {
    if (more && i < P.nseg && t >= prev_tiles) {
      t -= prev_tiles;
      tr.W = P.seg[i].W;
      tr.y = P.seg[i].y;
      tr.seg_rows = P.seg[i].rows;
      prev_tiles = P.seg[i].tiles;
    } else {
      more = false;
    }
  }
  int lim = P.T;
  if (t >= P.n1) {
    // the last round of a balanced phase: smaller tiles
    tr.r0 = static_cast<int64_t>(P.n1) * P.T + static_cast<int64_t>(t - P.n1) * P.T2;
    lim = P.T2;
  } else {
    tr.r0 = static_cast<int64_t>(t) * P.T;
  }
  const int64_t rem = tr.seg_rows - tr.r0;
  tr.nrows = static_cast<int>(rem < lim ? rem : lim);
  return tr;
}

// Shared-memory ring.  Layout: full[S], ready[S], empty[S] mbarriers, S
// partial buffers of red_floats floats (one per stage), the activation
// staging buffer (xs_floats), then S stages of stage_bytes (128-B aligned,
// each with >= 16 B of slack after the largest tile for the 2-byte-aligned
// Q6_K word loads).
// Staging row stride: U rounded up to an odd number of floats, so lanes
// walking units (or columns) hit distinct banks.
__host__ __device__ constexpr int red_stride(int U) { return U | 1; }
// Partial-buffer row pitch: U rounded up to a multiple of 4 floats (rows start
// on 16-byte boundaries, so the reducer reads them as float4) with an odd
// number of float4s, so eight lanes reading eight rows cover all 32 banks.
__host__ __device__ constexpr int red_pitch(int U) {
  return (((U + 3) & ~3) >> 2) % 2 == 0 ? ((U + 3) & ~3) + 4 : ((U + 3) & ~3);
}

struct Ring {
  uint64_t* full;
  uint64_t* ready;
  uint64_t* empty;
  int* rows;          // rows of the tile in each stage (set by the producer)
  float* red;
  float* xs;          // activation staging, transposed [64][U | 1]
  uint8_t* stages;
  uint32_t S;
  uint32_t stage_bytes;
  uint32_t red_floats;
  uint32_t xs_floats;
  __device__ __forceinline__ uint8_t* stage(uint32_t s) const {
    return stages + static_cast<size_t>(s) * stage_bytes;
  }
};

// mbarriers and the stages' row counts first (28 B per stage, rounded up to
// 16 B so the partial buffers start 16-byte aligned), then the partials, then
// the staging buffer.
__host__ __device__ constexpr uint32_t ring_bar_bytes(uint32_t S) { return (28u * S + 15u) & ~15u; }

__host__ __device__ constexpr size_t ring_header_bytes(uint32_t S, uint32_t red_floats,
                                                       uint32_t xs_floats) {
  return ((ring_bar_bytes(S) + 4u * S * red_floats + 4u * xs_floats + 127u) / 128u) * 128u;
}

__host__ __device__ constexpr size_t ring_smem_bytes(uint32_t S, uint32_t stage_bytes,
                                                    uint32_t red_floats, uint32_t xs_floats) {
  return ring_header_bytes(S, red_floats, xs_floats) + static_cast<size_t>(S) * stage_bytes;
}

__device__ __forceinline__ Ring make_ring(uint8_t* smem, uint32_t S, uint32_t stage_bytes,
                                          uint32_t red_floats, uint32_t xs_floats) {
  Ring R;
  R.full = reinterpret_cast<uint64_t*>(smem);
  R.ready = R.full + S;
  R.empty = R.ready + S;
  R.rows = reinterpret_cast<int*>(R.empty + S);
  R.red = reinterpret_cast<float*>(smem + ring_bar_bytes(S));
  R.xs = R.red + static_cast<size_t>(S) * red_floats;
  R.stages = smem + ring_header_bytes(S, red_floats, xs_floats);
  R.S = S;
  R.stage_bytes = stage_bytes;
  R.red_floats = red_floats;
  R.xs_floats = xs_floats;
  return R;
}

// Position in the ring: stage index and phase parity, advanced per tile
// (no division in the loops).
struct RingPos {
  uint32_t s = 0, ph = 0, n = 0;  // n = tiles passed so far
  __device__ __forceinline__ void advance(uint32_t S) {
    ++n;
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Called by one thread before the role split (followed by __syncthreads()).
__device__ __forceinline__ void ring_init(const Ring& R, int consumer_warps) {
  for (uint32_t s = 0; s < R.S; ++s) {
    mbar_init(&R.full[s], 1);
    mbar_init(&R.ready[s], static_cast<uint32_t>(consumer_warps));
    mbar_init(&R.empty[s], 1);
  }
  fence_barrier_init();
}

// ------------------------------------------------------------------ producer
// Fills stage s for tile t of phase P.  Rows are contiguous, so a tile is one
// copy (two for the gated pair).  A copy's start is 16-byte aligned because T
// is a multiple of the rows needed to make T * row_bytes a multiple of 16; only
// the last tile of a matrix can end off a 16-byte boundary, and those < 16 tail
// bytes are moved with plain loads/stores before the arrive (release) that
// publishes the stage.
__device__ __forceinline__ void copy_tail(uint8_t* dst, const uint8_t* src, uint32_t from,
                                          uint32_t to) {
  for (uint32_t i = from; i < to; ++i) dst[i] = src[i];
}

__device__ __forceinline__ void fill_stage(const Phase& P, int t, const Ring& R, uint32_t s,
                                           uint64_t pol) {
  const TileRef tr = tile_ref(P, t);
  uint8_t* dst = R.stage(s);
  const uint32_t bytes = static_cast<uint32_t>(tr.nrows * P.row_bytes);
  const uint32_t bulk = bytes & ~15u;
  const uint8_t* g = tr.W + tr.r0 * P.row_bytes;
  const bool pair = P.epi != EPI_STORE;
  const uint8_t* up = pair ? P.W2 + tr.r0 * P.row_bytes : nullptr;
  uint8_t* dst_up = dst + static_cast<size_t>(P.T) * P.row_bytes;
  // the tile's row count for the consumers, published by the arrive below
  R.rows[s] = tr.nrows;
  if (P.row_stride != P.row_bytes) {
    // column slice (split-K): one copy per row; row_bytes and row_stride are
    // multiples of 16 here (checked on the host)
    mbar_arrive_expect_tx(&R.full[s], bytes);
    const uint8_t* src = tr.W + tr.r0 * P.row_stride;
    for (int i = 0; i < tr.nrows; ++i)
      bulk_copy_g2s(dst + static_cast<size_t>(i) * P.row_bytes, src + i * P.row_stride,
                    static_cast<uint32_t>(P.row_bytes), &R.full[s], pol);
    return;
  }
  copy_tail(dst, g, bulk, bytes);
  if (pair) copy_tail(dst_up, up, bulk, bytes);
  mbar_arrive_expect_tx(&R.full[s], pair ? 2u * bulk : bulk);
  if (bulk) {
    bulk_copy_g2s(dst, g, bulk, &R.full[s], pol);
    if (pair) bulk_copy_g2s(dst_up, up, bulk, &R.full[s], pol);
  }
}

// Producer gate: gate(p, j) is asked before tile j (in this CTA's order) of
// phase p is copied, and may hold the copy back (bounded; false on timeout).
struct NoGate {
  __device__ __forceinline__ bool operator()(int, int) const { return true; }
};

// PhaseList: count() and get(i) -> Phase, evaluated identically by producer
// and consumers.
template <class PhaseList, class Gate = NoGate>
__device__ void run_producer(const PhaseList& L, const Ring& R, unsigned* err,
                             const Gate& gate = Gate()) {
  const uint64_t pol = l2_policy_evict_first();
  RingPos pos;
  bool ok = true;
  const int nph = L.count();
  for (int p = 0; p < nph && ok; ++p) {
    const Phase P = L.get(p);
    const int c = static_cast<int>(blockIdx.x) - P.cta0;
    if (c < 0 || c >= P.ncta) continue;
    for (int t = c, j = 0; t < P.n_tiles; t += P.ncta, ++j) {
      if (!gate(p, j) || !mbar_wait(&R.empty[pos.s], pos.ph ^ 1u)) {
        atomicOr(err, kErrEmptyWait);
        ok = false;
        break;
      }
      fill_stage(P, t, R, pos.s, pol);
      pos.advance(R.S);
    }
  }
  // Do not leave while copies into this CTA's shared memory are in flight.
  const uint32_t k = pos.n;
  const uint32_t first = k > R.S ? k - R.S : 0u;
  for (uint32_t i = first; i < k; ++i) {
    if (!mbar_wait(&R.full[i % R.S], (i / R.S) & 1u)) atomicOr(err, kErrDrain);
  }
}

// ------------------------------------------------------------------ consumers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Activation loaders: x(col) for the phase's input vector.
struct XPlain {            // global, written before this launch
  const float* p;
  __device__ __forceinline__ float operator()(int64_t i) const { return p[i]; }
};
struct XCoherent {         // global, written by other CTAs of this launch
  const float* p;
  __device__ __forceinline__ float operator()(int64_t i) const { return ld_cg(p + i); }
};
struct XShared {           // shared memory, prepared by this CTA
  const float* p;
  __device__ __forceinline__ float operator()(int64_t i) const { return p[i]; }
};

// Unit-local activation loader over the transposed staging buffer:
// element l of unit u lives at xs[l * US + u] (US odd: conflict-free reads
// for consecutive u, and conflict-free writes for consecutive l).
struct XUnit {
  const float* xs;
  int US;
  int u;
  __device__ __forceinline__ float operator()(int l) const { return xs[l * US + u]; }
};

// Copies activation vector `src` (K columns) into the transposed staging
// buffer with coalesced reads.  Called by all C consumer threads.  Loads are
// issued in chunks of 8 before any is used, so a thread waits for one memory
// latency per chunk rather than per element.
template <class Unit, class Src, int kChunk = 8>
__device__ __forceinline__ void stage_x(float* xs, int US, const Src& src, int64_t K, int ctid,
                                        int C) {
  for (int64_t base = ctid; base < K; base += static_cast<int64_t>(kChunk) * C) {
    float v[kChunk];
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int64_t col = base + static_cast<int64_t>(j) * C;
      v[j] = col < K ? src(col) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
      const int64_t col = base + static_cast<int64_t>(j) * C;
      if (col < K) {
        int u, l;
        Unit::unit_of(col, u, l);
        xs[l * US + u] = v[j];
      }
    }
  }
}

// Consume all tiles of phase P assigned to this CTA.  `k` is the CTA's running
// tile counter (producer and reducer walk the same order).  Thread ctid owns
// unit u = ctid % U and slot g = ctid / U; slot g serves activation vector
// b = g / G and rows gg, gg + G, ... of each tile (gg = g % G).  x_of(b)
// returns a column loader of vector b; vectors are staged one at a time
// through shared memory.  With STAGED = false the caller has already written
// the single vector (B = 1) into R.xs.  A unit with kDirect reads its own
// activations from x_of(b) instead (no staging).  Returns false on a timeout.
template <class Unit, bool STAGED = true, bool PIPE = true, class XOf>
__device__ __forceinline__ bool consume_phase(const Phase& Pref, const Ring& Rref, RingPos& pos,
                                              const XOf& x_of, int ctid, int C, unsigned* err) {
  // private copies: the loop stores through generic pointers, which could
  // otherwise alias a referenced Phase and force reloads
  const Phase P = Pref;
  const Ring R = Rref;
  const int cta = static_cast<int>(blockIdx.x) - P.cta0;
  if (cta < 0 || cta >= P.ncta) return true;
  const int U = P.U, G = P.G, US = red_stride(P.U);
  const int u = ctid % U, g = ctid / U;
  const int b = g / G, gg = g % G;
  const bool active = b < P.B;
  const int lane = ctid & 31;
  const bool pair = P.epi != EPI_STORE;
  const int slots = pair ? 2 * P.T : P.T;      // partial rows per vector
  const size_t rb = static_cast<size_t>(P.row_bytes);
  Unit unit;
  if constexpr (Unit::kMixed) unit.q6 = P.fmt == 14;
  if constexpr (Unit::kDirect) {
    // the unit reads its activation bytes of vector b itself
    if (active) unit.setup(u, x_of(b));
  } else if constexpr (STAGED) {
    for (int bb = 0; bb < P.B; ++bb) {
      if (bb) bar_sync(kConsumerBar, C);       // previous vector fully read
      // one round of loads per thread when K allows (every CTA reads the same
      // vector at the same moment: each extra round costs a loaded L2 trip)
      if (P.K > 8 * static_cast<int64_t>(C))
        stage_x<Unit, decltype(x_of(bb)), 16>(R.xs, US, x_of(bb), P.K, ctid, C);
      else
        stage_x<Unit>(R.xs, US, x_of(bb), P.K, ctid, C);
      bar_sync(kConsumerBar, C);
      if (active && b == bb) unit.setup(u, XUnit{R.xs, US, u});
    }
  } else {
    if (active) unit.setup(u, XUnit{R.xs, US, u});
  }
  const int UP = red_pitch(U);
  float* const red_b = R.red + static_cast<size_t>(b * slots) * UP + u;
  for (int t = cta; t < P.n_tiles; t += P.ncta) {
    if (!mbar_wait(&R.full[pos.s], pos.ph)) {
      atomicOr(err, kErrFullWait);
      return false;
    }
    // the tile's row count as the producer wrote it (a shared-memory load in
    // place of the segment / balanced-round arithmetic of tile_ref)
    const int nrows = R.rows[pos.s];
    const uint8_t* st = R.stage(pos.s);
    float* red = red_b + static_cast<size_t>(pos.s) * R.red_floats;
    const int nr = pair ? 2 * nrows : nrows;
    // row r of the tile lives at slot(r) rows into the stage; rows are taken
    // two at a time so that the two independent decode chains interleave
    auto slot_of = [&](int r) { return (pair && r >= nrows) ? P.T + (r - nrows) : r; };
    if constexpr (!PIPE) {
      if (active) {
        int r = gg;
        for (; r + G < nr; r += 2 * G) {
          const int s0 = slot_of(r), s1 = slot_of(r + G);
          float y0, y1;
          unit.row2(st + s0 * rb, st + s1 * rb, y0, y1);
          red[s0 * UP] = y0;
          red[s1 * UP] = y1;
        }
        if (r < nr) red[slot_of(r) * UP] = unit.row(st + slot_of(r) * rb);
      }
    } else if (active) {
      int r = gg;
      for (; r + G < nr; r += 2 * G) {
        const int s0 = slot_of(r), s1 = slot_of(r + G);
        typename Unit::Frag f0, f1;
        unit.load(st + s0 * rb, f0);
        unit.load(st + s1 * rb, f1);
        const float y0 = unit.compute(f0);
        const float y1 = unit.compute(f1);
        red[s0 * UP] = y0;
        red[s1 * UP] = y1;
      }
      if (r < nr) {
        typename Unit::Frag f;
        unit.load(st + slot_of(r) * rb, f);
        red[slot_of(r) * UP] = unit.compute(f);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.ready[pos.s]);
    pos.advance(R.S);
  }
  return true;
}

// sum of p[0 .. n) taken by lane group member c0 of step members, in a fixed
// order: float4 chunks c0, c0 + step, ... of the row (p 16-byte aligned),
// summed lane-wise, then ((s0 + s1) + (s2 + s3)), then the member's share of
// the n % 4 tail entries.
// Chunks are loaded four at a time before they are added (the adds keep the
// chunk order), so one shared-memory latency covers four chunks.
__device__ __forceinline__ float quad_sum(const float* p, int c0, int n, int step) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  const int nq = n >> 2;
  auto add = [&](const float4 v) {
    s0 += v.x;
    s1 += v.y;
    s2 += v.z;
    s3 += v.w;
  };
  int k = c0;
  for (; k + 3 * step < nq; k += 4 * step) {
    const float4 a = *reinterpret_cast<const float4*>(p + 4 * k);
    const float4 b = *reinterpret_cast<const float4*>(p + 4 * (k + step));
    const float4 c = *reinterpret_cast<const float4*>(p + 4 * (k + 2 * step));
    const float4 d = *reinterpret_cast<const float4*>(p + 4 * (k + 3 * step));
    add(a);
    add(b);
    add(c);
    add(d);
  }
  for (; k < nq; k += step) add(*reinterpret_cast<const float4*>(p + 4 * k));
  float t = (s0 + s1) + (s2 + s3);
  for (int c = 4 * nq + c0; c < n; c += step) t += p[c];
  return t;
}

// sum of p[c] for c = c0, c0 + step, ... < n, in a fixed order: four
// interleaved partial sums (independent loads), then ((s0 + s1) + (s2 + s3)).
__device__ __forceinline__ float strided_sum(const float* p, int c0, int n, int step) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  int c = c0;
  for (; c + 3 * step < n; c += 4 * step) {
    s0 += p[c];
    s1 += p[c + step];
    s2 += p[c + 2 * step];
    s3 += p[c + 3 * step];
  }
  for (; c < n; c += step) s0 += p[c];
  return (s0 + s1) + (s2 + s3);
}

// Reduce all tiles of phase P for this CTA (one warp).  Output i of a tile is
// (vector b, row o), i = b * nrows + o.  Lanes form groups of gsz lanes per
// output (gsz = 32 when the tile has one output, 1 when it has >= 32); each
// lane adds a fixed strided subset of the row's partials, then the group adds
// its lanes with a fixed xor tree: the order never changes between runs.
// epi(P, tr, b, o, v, v2) stores the result (v2 = the up row for GEGLU).
template <class Epi>
__device__ __forceinline__ bool reduce_phase(const Phase& Pref, const Ring& Rref, RingPos& pos,
                                             const Epi& epi, unsigned* err) {
  const Phase P = Pref;
  const Ring R = Rref;
  const int cta = static_cast<int>(blockIdx.x) - P.cta0;
  if (cta < 0 || cta >= P.ncta) return true;
  const int lane = threadIdx.x & 31;
  const int U = P.U, UP = red_pitch(P.U);
  const bool pair = P.epi != EPI_STORE;
  const int slots = pair ? 2 * P.T : P.T;
  int cached_n_out = -1, lg = 5;
  for (int t = cta; t < P.n_tiles; t += P.ncta) {
    const uint32_t s = pos.s;
    if (!mbar_wait(&R.ready[s], pos.ph)) {
      atomicOr(err, kErrFullWait);
      return false;
    }
    const TileRef tr = tile_ref(P, t);
    const float* red = R.red + static_cast<size_t>(s) * R.red_floats;
    const int n_out = P.B * tr.nrows;
    // lane grouping: recomputed only when the tile's row count changes (the
    // balanced last round, a segment's end); the reducer's code is a serial
    // chain of dependent instructions, on the critical path at a phase's end
    if (n_out != cached_n_out) {
      cached_n_out = n_out;
      lg = 5;
      while (lg > 0 && (n_out << lg) > 32) --lg;
    }
    const int per_pass = 32 >> lg;
    const int sub = lane & ((1 << lg) - 1);
    for (int base = 0; base < n_out; base += per_pass) {
      const int oi = base + (lane >> lg);
      const bool valid = oi < n_out;
      const int ob = (valid && P.B > 1) ? oi / tr.nrows : 0;
      const int o = valid ? oi - ob * tr.nrows : 0;
      const float* rr = red + (ob * slots + o) * UP;
      float v = 0.f, v2 = 0.f;
      const int gsz = 1 << lg;
      if (valid) {
        v = quad_sum(rr, sub, U, gsz);
        if (pair) v2 = quad_sum(rr + P.T * UP, sub, U, gsz);
      }
      for (int w = gsz >> 1; w > 0; w >>= 1) {
        v += __shfl_xor_sync(0xFFFFFFFFu, v, w);
        v2 += __shfl_xor_sync(0xFFFFFFFFu, v2, w);
      }
      if (valid && sub == 0) epi(P, tr, ob, o, v, v2);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[s]);
    pos.advance(R.S);
  }
  return true;
}

// GELU, tanh form: 0.5 t (1 + tanh(sqrt(2/pi) (t + 0.044715 t^3)))
// (infer-compute README §Shaders, geglu_gelu_tanh).
__device__ __forceinline__ float gelu_tanh(float t) {
  const float k = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * t * (1.0f + tanhf(k * fmaf(0.044715f * t, t * t, t)));
}

struct EpiStore {
  __device__ __forceinline__ void operator()(const Phase& P, const TileRef& tr, int b, int o,
                                             float v, float) const {
    tr.y[b * tr.seg_rows + tr.r0 + o] = v;
  }
};

struct EpiGeglu {
  __device__ __forceinline__ void operator()(const Phase& P, const TileRef& tr, int b, int o,
                                             float g, float u) const {
    tr.y[b * tr.seg_rows + tr.r0 + o] = gelu_tanh(g) * u;
  }
};

// SiLU, the logistic-gated variant for SiLU models (infer-compute README
// §Shaders, the SiLU-gated down variant): silu(t) = t / (1 + exp(-t)).
__device__ __forceinline__ float silu(float t) { return t / (1.0f + expf(-t)); }

struct EpiSwiglu {
  __device__ __forceinline__ void operator()(const Phase& P, const TileRef& tr, int b, int o,
                                             float g, float u) const {
    tr.y[b * tr.seg_rows + tr.r0 + o] = silu(g) * u;
  }
};

// Loader factories: vector b of a [B][stride] activation array.
struct XOfPlain {
  const float* x;
  int64_t stride;
  __device__ __forceinline__ XPlain operator()(int b) const { return XPlain{x + b * stride}; }
};

// Vector b of [B][stride] bytes of Q8_0 blocks (units with kDirect).
struct XOfQ8 {
  const uint8_t* xq;
  int64_t stride;
  __device__ __forceinline__ const uint8_t* operator()(int b) const { return xq + b * stride; }
};

}  // namespace qws
