/*
 * oracle.c -- plain, slow, f64 CPU reference for the quantized weight-streaming
 * decode path.  TEST INFRASTRUCTURE ONLY: it is used by tests/, by the smoke
 * check and by the benchmark's CPU-baseline leg, never by the product path.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (three pages of the "infer" project, pg_infer 0.1.3-alpha):
 *   [compute]  crates/infer-compute/README.md
 *   [engine]   crates/infer-inference/README.md
 *   [perf]     crates/infer-inference/PERFORMANCE.md
 *
 * The pages name the formats (Q4_0, Q4_K, Q6_K, and Q8_0 for the 8-bit path;
 * "GGUF-compatible -- Q4_K/Q6_K formats match Ollama's quantization", [compute]
 * §Design Principles item 8)
 * but print no byte layout.  The layouts below are the plainest reading of
 * "GGUF-compatible": the public GGUF block formats, restated here in prose and
 * written from that understanding.  Every weight is decoded to an f64 value
 * and every sum is accumulated in f64 in index order.  There is no blocking,
 * no fusion and no reordering beyond what each definition states.
 *
 * Pins: every function here is checked by tests/test_oracle_*.py against
 * hand-decoded byte fixtures, closed forms, library routines on special
 * cases, or brute force (see the test files).  Nothing is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QO_Q4_0 2
#define QO_Q4_K 12
#define QO_ACT_GELU_TANH 0
#define QO_ACT_SILU 1
#define QO_Q6_K 14
#define QO_Q8_0 8

/* ---------------------------------------------------------------------------
 * IEEE-754 binary16 -> double, by bit arithmetic (sign, 5-bit exponent with
 * bias 15, 10-bit fraction; exponent 0 is subnormal, 31 is inf/NaN).
 * ------------------------------------------------------------------------- */
double qo_half(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* frac * 2^-10 * 2^-14 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

void qo_dequant_q8_0(const uint8_t *blk, double out[32]);

/* ---------------------------------------------------------------------------
 * Q4_0 ([compute] §Shaders "Q4_0 matvec"): 32 weights in 18 bytes.
 *   bytes 0..1  d (binary16)
 *   bytes 2..17 qs[16]: weight j (0..15) is the low nibble of qs[j],
 *               weight 16+j is the high nibble of qs[j]
 *   w = d * (q - 8)
 * ------------------------------------------------------------------------- */
void qo_dequant_q4_0(const uint8_t *blk, double out[32])
{
    double d = qo_half(rd16(blk));
    const uint8_t *qs = blk + 2;
    for (int j = 0; j < 16; ++j) {
        int lo = qs[j] & 15;
        int hi = qs[j] >> 4;
        out[j] = d * (double)(lo - 8);
        out[16 + j] = d * (double)(hi - 8);
    }
}

/* ---------------------------------------------------------------------------
 * Q4_K ([compute] §Shaders "Q4_K/Q6_K" row, q4k_matvec): a super-block of 256
 * weights in 144 bytes, eight sub-blocks of 32 weights.
 *   bytes 0..1   d    (binary16)  super-block scale of the sub-block scales
 *   bytes 2..3   dmin (binary16)  super-block scale of the sub-block mins
 *   bytes 4..15  sc[12]: eight 6-bit scales and eight 6-bit mins, packed:
 *       sub-block s < 4 : scale = sc[s] & 63,  min = sc[s+4] & 63
 *       sub-block s >= 4: scale = (sc[s+4] & 15) | ((sc[s-4] >> 6) << 4)
 *                         min   = (sc[s+4] >> 4) | ((sc[s]   >> 6) << 4)
 *   bytes 16..143 qs[128], four chunks of 32 bytes; in chunk c (0..3), byte
 *       qs[32c + l] holds weight 64c + l (sub-block 2c) in its low nibble and
 *       weight 64c + 32 + l (sub-block 2c+1) in its high nibble.
 *   w = d * scale[s] * q - dmin * min[s]
 * ------------------------------------------------------------------------- */
void qo_q4_k_scale_min(const uint8_t *sc, int s, int *scale, int *mn)
{
    if (s < 4) {
        *scale = sc[s] & 63;
        *mn = sc[s + 4] & 63;
    } else {
        *scale = (sc[s + 4] & 15) | ((sc[s - 4] >> 6) << 4);
        *mn = (sc[s + 4] >> 4) | ((sc[s] >> 6) << 4);
    }
}

void qo_dequant_q4_k(const uint8_t *blk, double out[256])
{
    double d = qo_half(rd16(blk));
    double dmin = qo_half(rd16(blk + 2));
    const uint8_t *sc = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int c = 0; c < 4; ++c) {
        int s_lo = 2 * c, s_hi = 2 * c + 1;
        int sc_lo, m_lo, sc_hi, m_hi;
        qo_q4_k_scale_min(sc, s_lo, &sc_lo, &m_lo);
        qo_q4_k_scale_min(sc, s_hi, &sc_hi, &m_hi);
        for (int l = 0; l < 32; ++l) {
            int byte = qs[32 * c + l];
            int q_lo = byte & 15;
            int q_hi = byte >> 4;
            out[64 * c + l] = d * (double)sc_lo * (double)q_lo - dmin * (double)m_lo;
            out[64 * c + 32 + l] = d * (double)sc_hi * (double)q_hi - dmin * (double)m_hi;
        }
    }
}

/* ---------------------------------------------------------------------------
 * Q6_K ([compute] §Shaders, q6k_matvec): 256 weights in 210 bytes.
 *   bytes 0..127   ql[128]  low 4 bits
 *   bytes 128..191 qh[64]   high 2 bits, four per byte
 *   bytes 192..207 sc[16]   signed 8-bit scales, one per 16 weights
 *   bytes 208..209 d        (binary16)
 * For each half h (weights 128h .. 128h+127) and l = 0..31:
 *   weight 128h +      l : low  nibble of ql[64h + l],      bits (qh[32h+l] >> 0) & 3
 *   weight 128h + 32 + l : low  nibble of ql[64h + 32 + l], bits (qh[32h+l] >> 2) & 3
 *   weight 128h + 64 + l : high nibble of ql[64h + l],      bits (qh[32h+l] >> 4) & 3
 *   weight 128h + 96 + l : high nibble of ql[64h + 32 + l], bits (qh[32h+l] >> 6) & 3
 *   q = (nibble | bits << 4) - 32, in [-32, 31];  w = d * sc[i / 16] * q
 * ------------------------------------------------------------------------- */
void qo_dequant_q6_k(const uint8_t *blk, double out[256])
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *sc = (const int8_t *)(blk + 192);
    double d = qo_half(rd16(blk + 208));
    for (int h = 0; h < 2; ++h) {
        for (int l = 0; l < 32; ++l) {
            int a = ql[64 * h + l];
            int b = ql[64 * h + 32 + l];
            int hb = qh[32 * h + l];
            int q[4];
            q[0] = ((a & 15) | (((hb >> 0) & 3) << 4)) - 32;
            q[1] = ((b & 15) | (((hb >> 2) & 3) << 4)) - 32;
            q[2] = ((a >> 4) | (((hb >> 4) & 3) << 4)) - 32;
            q[3] = ((b >> 4) | (((hb >> 6) & 3) << 4)) - 32;
            for (int k = 0; k < 4; ++k) {
                int i = 128 * h + 32 * k + l;
                out[i] = d * (double)sc[i / 16] * (double)q[k];
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * Format table.
 * ------------------------------------------------------------------------- */
int qo_block_weights(int fmt)
{
    switch (fmt) {
    case QO_Q4_0: return 32;
    case QO_Q4_K: return 256;
    case QO_Q6_K: return 256;
    case QO_Q8_0: return 32;
    default: return 0;
    }
}

int qo_block_bytes(int fmt)
{
    switch (fmt) {
    case QO_Q4_0: return 18;
    case QO_Q4_K: return 144;
    case QO_Q6_K: return 210;
    case QO_Q8_0: return 34;
    default: return 0;
    }
}

static void dequant_block(int fmt, const uint8_t *blk, double *out)
{
    if (fmt == QO_Q4_0) qo_dequant_q4_0(blk, out);
    else if (fmt == QO_Q8_0) qo_dequant_q8_0(blk, out);
    else if (fmt == QO_Q4_K) qo_dequant_q4_k(blk, out);
    else qo_dequant_q6_k(blk, out);
}

/* Dense f64 copy of rows [0, rows) of a row-major quantized matrix: row r is a
 * contiguous run of hidden / QK blocks.  Returns 0, or -1 on a bad shape. */
int qo_dequant_rows(int fmt, const uint8_t *W, int64_t rows, int64_t hidden, double *out)
{
    int qk = qo_block_weights(fmt), bb = qo_block_bytes(fmt);
    if (qk == 0 || hidden % qk != 0) return -1;
    int64_t nb = hidden / qk;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            dequant_block(fmt, W + (r * nb + b) * bb, out + r * hidden + b * qk);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Quantized matrix-vector product ([compute] §Quick Start
 * "backend.q4k_matvec(&q4k_data, &x, rows, hidden)").
 *   y[b][r]     = sum_i w[r][i] * x[b][i]          (f64, index order)
 *   bound[b][r] = sum_i |w[r][i] * x[b][i]|
 * x is [batch][hidden]; y and bound are [batch][rows].  Only rows in
 * [row_begin, row_end) are written, so a caller may split the rows.
 * ------------------------------------------------------------------------- */
int qo_matvec(int fmt, const uint8_t *W, int64_t rows, int64_t hidden,
              const double *x, int batch, int64_t row_begin, int64_t row_end,
              double *y, double *bound)
{
    int qk = qo_block_weights(fmt), bb = qo_block_bytes(fmt);
    if (qk == 0 || hidden % qk != 0 || batch < 1) return -1;
    if (row_begin < 0 || row_end > rows || row_begin > row_end) return -1;
    int64_t nb = hidden / qk;
    double *wrow = (double *)malloc(sizeof(double) * (size_t)(hidden > 0 ? hidden : 1));
    if (!wrow) return -2;
    for (int64_t r = row_begin; r < row_end; ++r) {
        for (int64_t b = 0; b < nb; ++b)
            dequant_block(fmt, W + (r * nb + b) * bb, wrow + b * qk);
        for (int bt = 0; bt < batch; ++bt) {
            const double *xb = x + (int64_t)bt * hidden;
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < hidden; ++i) {
                double t = wrow[i] * xb[i];
                acc += t;
                mag += fabs(t);
            }
            y[(int64_t)bt * rows + r] = acc;
            if (bound) bound[(int64_t)bt * rows + r] = mag;
        }
    }
    free(wrow);
    return 0;
}

/* ---------------------------------------------------------------------------
 * float -> IEEE-754 binary16 bits, round to nearest, ties to even (the
 * standard conversion), by arithmetic on the value: the magnitude is split
 * into an exponent E and a significand counted in units of the binary16
 * spacing at that exponent (2^(E-10) for normals, 2^-24 below 2^-14); the
 * count is rounded with rint() in the default ties-to-even mode.  A count
 * that rounds up to 2048 carries into the next exponent; magnitudes that
 * round above 65504 become infinity.
 * ------------------------------------------------------------------------- */
uint16_t qo_half_bits(float f)
{
    double v = (double)f;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7E00u);
    v = fabs(v);
    if (isinf(v)) return (uint16_t)(sign | 0x7C00u);
    if (v < ldexp(1.0, -14)) {
        double m = rint(v / ldexp(1.0, -24));       /* subnormal count, 0..1024 */
        return (uint16_t)(sign | (uint16_t)m);    /* 1024 is the smallest normal */
    }
    int e;
    frexp(v, &e);                                  /* v = f * 2^e, f in [0.5, 1) */
    int E = e - 1;                                 /* v in [2^E, 2^(E+1)) */
    double m = rint(v / ldexp(1.0, E - 10));       /* 1024..2048 */
    if (m == 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(m - 1024.0));
}

/* ---------------------------------------------------------------------------
 * Q8_0 ([compute] §Shaders rows "Q8" (q8_matvec) and "Element-wise"
 * (quantize_q8); the GGUF-compatible 8-bit format of the same README's format
 * list): 32 values in 34 bytes.
 *   bytes 0..1   d (binary16)
 *   bytes 2..33  qs[32], int8 (two's complement)
 *   w = d * q
 * ------------------------------------------------------------------------- */
void qo_dequant_q8_0(const uint8_t *blk, double out[32])
{
    double d = qo_half(rd16(blk));
    for (int j = 0; j < 32; ++j) {
        int q = blk[2 + j];
        if (q >= 128) q -= 256;
        out[j] = d * (double)q;
    }
}

/* ---------------------------------------------------------------------------
 * quantize_q8 ([compute] §Shaders "Element-wise", quantize_q8; the Q4_0 FFN
 * goes "through legacy Q8 path", §Architecture): activations -> Q8_0 blocks.
 * The pages give no rounding rule; this is symmetric absmax quantization, the
 * plainest reading of the 8-bit block format, with every decision in f32:
 *   amax = max_j |x_j|,  d = amax / 127,  id = d != 0 ? 1 / d : 0,
 *   q_j  = round(x_j * id)  (nearest, halves away from zero: C roundf)
 * and the stored scale is d rounded to binary16 (the codes use the f32 d).
 * n must be a multiple of 32; block k of x goes to out[34k .. 34k + 33].
 * ------------------------------------------------------------------------- */
int qo_quantize_q8_0(const float *x, int64_t n, uint8_t *out)
{
    if (n < 0 || n % 32 != 0) return -1;
    for (int64_t k = 0; k < n / 32; ++k) {
        const float *xb = x + 32 * k;
        uint8_t *blk = out + 34 * k;
        float amax = 0.0f;
        for (int j = 0; j < 32; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        float id = d != 0.0f ? 1.0f / d : 0.0f;
        uint16_t h = qo_half_bits(d);
        blk[0] = (uint8_t)(h & 0xFF);
        blk[1] = (uint8_t)(h >> 8);
        for (int j = 0; j < 32; ++j) {
            float t = xb[j] * id;
            int q = (int)roundf(t);
            blk[2 + j] = (uint8_t)(q & 0xFF);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Matvec over Q8_0 activations ([compute] §Architecture "Q4_0 through legacy
 * Q8 path"; §Shaders "Q8" row, q8_matvec): weights in Q4_0 or Q8_0 times the
 * quantized activation xq.  Per 32-weight block the integer codes multiply
 * exactly, then the two scales apply:
 *   y[b][r]     = sum_k dw[r][k] * dx[b][k] * sum_j qw[r][k][j] * qx[b][k][j]
 *   bound[b][r] = sum_k |dw * dx| * sum_j |qw * qx|
 * where qw = q - 8 for Q4_0 and qw = q for Q8_0; the integer sums are exact,
 * the rest is f64 in block order.  xq is [batch][hidden / 32] blocks of 34 B;
 * y and bound are [batch][rows], written for rows in [row_begin, row_end).
 * ------------------------------------------------------------------------- */
int qo_matvec_q8(int wfmt, const uint8_t *W, int64_t rows, int64_t hidden,
                 const uint8_t *xq, int batch, int64_t row_begin, int64_t row_end,
                 double *y, double *bound)
{
    if ((wfmt != QO_Q4_0 && wfmt != QO_Q8_0) || hidden % 32 != 0 || batch < 1) return -1;
    if (row_begin < 0 || row_end > rows || row_begin > row_end) return -1;
    int64_t nb = hidden / 32;
    int bb = wfmt == QO_Q4_0 ? 18 : 34;
    for (int bt = 0; bt < batch; ++bt) {
        for (int64_t r = row_begin; r < row_end; ++r) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < nb; ++k) {
                const uint8_t *wb = W + (r * nb + k) * bb;
                const uint8_t *xb = xq + ((int64_t)bt * nb + k) * 34;
                int qw[32];
                if (wfmt == QO_Q4_0) {
                    for (int j = 0; j < 16; ++j) {
                        qw[j] = (wb[2 + j] & 15) - 8;
                        qw[16 + j] = (wb[2 + j] >> 4) - 8;
                    }
                } else {
                    for (int j = 0; j < 32; ++j) qw[j] = wb[2 + j] >= 128 ? wb[2 + j] - 256 : wb[2 + j];
                }
                int64_t isum = 0, iabs = 0;
                for (int j = 0; j < 32; ++j) {
                    int qx = xb[2 + j] >= 128 ? xb[2 + j] - 256 : xb[2 + j];
                    isum += (int64_t)qw[j] * qx;
                    iabs += llabs((int64_t)qw[j] * qx);
                }
                double s = qo_half(rd16(wb)) * qo_half(rd16(xb));
                acc += s * (double)isum;
                mag += fabs(s) * (double)iabs;
            }
            y[(int64_t)bt * rows + r] = acc;
            if (bound) bound[(int64_t)bt * rows + r] = mag;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * GELU, tanh form ([compute] §Shaders "geglu_gelu_tanh"; [perf] §Activation
 * Function Support, Gemma rows).  The pages name it and print no formula; this
 * is the standard tanh approximation of GELU:
 *   gelu(t) = 0.5 t (1 + tanh( sqrt(2/pi) (t + 0.044715 t^3) ))
 * ------------------------------------------------------------------------- */
double qo_gelu_tanh(double t)
{
    const double k = sqrt(2.0 / M_PI);
    return 0.5 * t * (1.0 + tanh(k * (t + 0.044715 * t * t * t)));
}

/* ---------------------------------------------------------------------------
 * SiLU ([compute] §Shaders: the SiLU-gated down variant for SiLU models;
 * [perf] §Activation Function Support): silu(t) = t * sigmoid(t)
 *   = t / (1 + exp(-t)).
 * ------------------------------------------------------------------------- */
double qo_silu(double t)
{
    return t / (1.0 + exp(-t));
}

/* ---------------------------------------------------------------------------
 * RMS norm ([compute] §Shaders "rms_norm"; [engine] §Key Components
 * residual.rs): y_i = x_i / sqrt(mean_j x_j^2 + eps) * w_i.
 * The weight multiplies as given (no 1 + w offset).
 * ------------------------------------------------------------------------- */
void qo_rms_norm(const double *x, const double *w, int64_t n, double eps, double *y)
{
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; ++i) y[i] = x[i] * inv * w[i];
}

/* residual_add ([compute] §Shaders "Element-wise"): h_i <- h_i + y_i. */
void qo_residual_add(double *h, const double *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] += y[i];
}

/* residual_norm ([compute] §Shaders "residual_norm"): the residual add
 * followed by the RMS norm of its result, h <- h + y, x = rms_norm(h, w). */
void qo_residual_rms_norm(double *h, const double *y, const double *w, int64_t n, double eps,
                          double *x)
{
    qo_residual_add(h, y, n);
    qo_rms_norm(h, w, n, eps, x);
}

/* ---------------------------------------------------------------------------
 * Attention at sequence length 1 ([compute] §Architecture, decode.rs
 * "norm -> QKV -> attend -> O").  With one key, the softmax over one score is
 * exactly 1, so each query head's output is the value vector of the KV head it
 * reads.  Query head h reads KV head h / (n_q_heads / n_kv_heads) (contiguous
 * grouped-query grouping).  q and k do not enter the result.
 *   attn[h * head_dim + i] = v[(h / group) * head_dim + i]
 * ------------------------------------------------------------------------- */
int qo_attn_seq1(const double *v, int n_q_heads, int n_kv_heads, int head_dim, double *attn)
{
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
    int group = n_q_heads / n_kv_heads;
    for (int h = 0; h < n_q_heads; ++h)
        for (int i = 0; i < head_dim; ++i)
            attn[h * head_dim + i] = v[(h / group) * head_dim + i];
    return 0;
}

/* ---------------------------------------------------------------------------
 * RoPE at one position ([compute] §Shaders "RoPE" row: rope_at_pos,
 * rope_at_pos_batched; the README's test list names partial RoPE; [perf]
 * §RoPE comparison: full and 25 % rotary dimensions).  The pages give no
 * formula; this is the standard rotary embedding in its half-split form:
 * with r = rot_dim (even, <= head_dim), for i < r/2
 *   theta_i = pos * base^(-2i / r)
 *   (x_i, x_{i+r/2}) <- (x_i cos theta_i - x_{i+r/2} sin theta_i,
 *                        x_i sin theta_i + x_{i+r/2} cos theta_i)
 * and dimensions r .. head_dim-1 are left as they are.  x is [n_heads][head_dim],
 * every head rotated the same way.
 * ------------------------------------------------------------------------- */
int qo_rope(double *x, int n_heads, int head_dim, int rot_dim, int64_t pos, double base)
{
    if (rot_dim < 0 || rot_dim % 2 || rot_dim > head_dim || base <= 0.0) return -1;
    int half = rot_dim / 2;
    for (int h = 0; h < n_heads; ++h) {
        double *xh = x + (int64_t)h * head_dim;
        for (int i = 0; i < half; ++i) {
            double theta = (double)pos * pow(base, -2.0 * (double)i / (double)rot_dim);
            double c = cos(theta), s = sin(theta);
            double a = xh[i], b = xh[i + half];
            xh[i] = a * c - b * s;
            xh[i + half] = a * s + b * c;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * kv_append ([compute] §Shaders "Attention" row): the new token's k and v
 * ([n_kv_heads][head_dim] each) are written at position pos of the caches
 * ([n_kv_heads][max_seq][head_dim] each).
 * ------------------------------------------------------------------------- */
int qo_kv_append(double *kc, double *vc, const double *k, const double *v, int n_kv_heads,
                 int head_dim, int64_t max_seq, int64_t pos)
{
    if (pos < 0 || pos >= max_seq) return -1;
    for (int g = 0; g < n_kv_heads; ++g)
        for (int i = 0; i < head_dim; ++i) {
            kc[((int64_t)g * max_seq + pos) * head_dim + i] = k[(int64_t)g * head_dim + i];
            vc[((int64_t)g * max_seq + pos) * head_dim + i] = v[(int64_t)g * head_dim + i];
        }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Attention of one query token over the KV cache ([compute] §Shaders
 * "Attention" row: kv_attention, GQA, softcap; [engine] §BLAS-Fused
 * Attention steps 1-3: scores = K q, scale and optional softcap, softmax,
 * output = V^T p).  For query head h (kv head g = h / (n_q / n_kv), the
 * contiguous GQA grouping):
 *   s_t = scale * (q_h . k_{g,t})                 t = 0 .. n_ctx-1
 *   s_t <- softcap * tanh(s_t / softcap)          only if softcap > 0
 *   p_t = exp(s_t - max s) / sum_u exp(s_u - max s)
 *   out_h = sum_t p_t v_{g,t}
 * also returns bound_h[i] = sum_t p_t |v_{g,t,i}| and smax_h = max_t
 * sum_i |scale q_h,i k_{g,t,i}| (the magnitude the score rounding scales with).
 * q is [n_q][hd]; caches [n_kv][max_seq][hd]; out and bound [n_q][hd].
 * ------------------------------------------------------------------------- */
int qo_kv_attention(const double *q, const double *kc, const double *vc, int n_q_heads,
                    int n_kv_heads, int head_dim, int64_t max_seq, int64_t n_ctx,
                    double scale, double softcap, double *out, double *bound, double *smax)
{
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
    if (n_ctx < 1 || n_ctx > max_seq) return -1;
    int group = n_q_heads / n_kv_heads;
    double *s = (double *)malloc(sizeof(double) * (size_t)n_ctx);
    if (!s) return -2;
    for (int h = 0; h < n_q_heads; ++h) {
        int g = h / group;
        const double *qh = q + (int64_t)h * head_dim;
        const double *kg = kc + (int64_t)g * max_seq * head_dim;
        const double *vg = vc + (int64_t)g * max_seq * head_dim;
        double mx = -INFINITY, mag = 0.0;
        for (int64_t t = 0; t < n_ctx; ++t) {
            double acc = 0.0, a = 0.0;
            for (int i = 0; i < head_dim; ++i) {
                acc += qh[i] * kg[t * head_dim + i];
                a += fabs(scale * qh[i] * kg[t * head_dim + i]);
            }
            acc *= scale;
            if (softcap > 0.0) acc = softcap * tanh(acc / softcap);
            s[t] = acc;
            if (acc > mx) mx = acc;
            if (a > mag) mag = a;
        }
        double den = 0.0;
        for (int64_t t = 0; t < n_ctx; ++t) {
            s[t] = exp(s[t] - mx);
            den += s[t];
        }
        for (int i = 0; i < head_dim; ++i) {
            double acc = 0.0, b = 0.0;
            for (int64_t t = 0; t < n_ctx; ++t) {
                double p = s[t] / den;
                acc += p * vg[t * head_dim + i];
                b += p * fabs(vg[t * head_dim + i]);
            }
            out[(int64_t)h * head_dim + i] = acc;
            if (bound) bound[(int64_t)h * head_dim + i] = b;
        }
        if (smax) smax[h] = mag;
    }
    free(s);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Gated FFN ([compute] §Shaders "Q4_K fused FFN": q4k_ffn_gate_up then
 * q4k_geglu_gelu_tanh_down, or the SiLU-gated variant; [engine] §WalkFfn
 * steps 1-3: gate and up projections, the gated activation, then the down
 * projection).
 *   g = Wg x,  u = Wu x            (inter rows, hidden columns)
 *   m_j = act(g_j) * u_j           (the gate takes the activation: gelu_tanh
 *                                   for act = QO_ACT_GELU_TANH, silu for
 *                                   QO_ACT_SILU)
 *   y = Wd m                       (hidden rows, inter columns)
 *   bound_y[i] = sum_j |wd[i][j] * m_j|
 * Any of the outputs except y may be NULL.
 * ------------------------------------------------------------------------- */
int qo_ffn_act(int act, int fmt_gu, const uint8_t *Wg, const uint8_t *Wu, int fmt_d,
               const uint8_t *Wd, int64_t hidden, int64_t inter, const double *x,
               double *g, double *u, double *m, double *y, double *bound_y)
{
    double *gg = (double *)malloc(sizeof(double) * (size_t)inter);
    double *uu = (double *)malloc(sizeof(double) * (size_t)inter);
    double *mm = (double *)malloc(sizeof(double) * (size_t)inter);
    int rc = -2;
    if (!gg || !uu || !mm) goto done;
    rc = qo_matvec(fmt_gu, Wg, inter, hidden, x, 1, 0, inter, gg, NULL);
    if (rc) goto done;
    rc = qo_matvec(fmt_gu, Wu, inter, hidden, x, 1, 0, inter, uu, NULL);
    if (rc) goto done;
    for (int64_t j = 0; j < inter; ++j)
        mm[j] = (act == QO_ACT_SILU ? qo_silu(gg[j]) : qo_gelu_tanh(gg[j])) * uu[j];
    rc = qo_matvec(fmt_d, Wd, hidden, inter, mm, 1, 0, hidden, y, bound_y);
    if (rc) goto done;
    if (g) memcpy(g, gg, sizeof(double) * (size_t)inter);
    if (u) memcpy(u, uu, sizeof(double) * (size_t)inter);
    if (m) memcpy(m, mm, sizeof(double) * (size_t)inter);
done:
    free(gg);
    free(uu);
    free(mm);
    return rc;
}

/* The GELU-gated FFN of the Gemma chain. */
int qo_ffn(int fmt_gu, const uint8_t *Wg, const uint8_t *Wu, int fmt_d, const uint8_t *Wd,
           int64_t hidden, int64_t inter, const double *x,
           double *g, double *u, double *m, double *y, double *bound_y)
{
    return qo_ffn_act(QO_ACT_GELU_TANH, fmt_gu, Wg, Wu, fmt_d, Wd, hidden, inter, x, g, u, m, y,
                      bound_y);
}

/* ---------------------------------------------------------------------------
 * One decoder layer of the single-token chain ([compute] §Architecture and
 * §Quick Start decode_token; [perf] §Post-Norm Architecture: Gemma-3 applies
 * a norm after attention and after the FFN as well as before them).
 *
 * post_norms = 1 (Gemma-3 sandwich):
 *   n1 = rms_norm(h, w_in)
 *   q, k, v = Wq n1, Wk n1, Wv n1
 *   a  = attention at seq 1 (value broadcast, see qo_attn_seq1)
 *   o  = Wo a
 *   h1 = h + rms_norm(o, w_post_attn)
 *   n2 = rms_norm(h1, w_pre_ffn)
 *   f  = FFN(n2)
 *   h' = h1 + rms_norm(f, w_post_ffn)
 * post_norms = 0 (pre-norm only): h1 = h + o, h' = h1 + f; w_post_* unused.
 * ------------------------------------------------------------------------- */
typedef struct {
    int fmt_qkv, fmt_o, fmt_gu, fmt_down;
    const uint8_t *Wq, *Wk, *Wv, *Wo, *Wg, *Wu, *Wd;
    const double *w_in, *w_post_attn, *w_pre_ffn, *w_post_ffn;
} qo_layer;

typedef struct {
    int64_t hidden, inter;
    int n_q_heads, n_kv_heads, head_dim;
    double eps;
    int post_norms;
} qo_dims;

/* Optional per-layer trace; any pointer may be NULL. */
typedef struct {
    double *n1, *q, *k, *v, *attn, *o, *h1, *n2, *g, *u, *m, *f, *bound_f;
} qo_trace;

int qo_layer_forward(const qo_layer *L, const qo_dims *D, const double *h, double *h_out,
                     qo_trace *T)
{
    int64_t H = D->hidden, I = D->inter;
    int64_t qd = (int64_t)D->n_q_heads * D->head_dim;
    int64_t kd = (int64_t)D->n_kv_heads * D->head_dim;
    size_t need = (size_t)(H * 6 + qd * 2 + kd * 2 + I * 3);
    double *buf = (double *)malloc(sizeof(double) * need);
    if (!buf) return -2;
    double *n1 = buf, *q = n1 + H, *k = q + qd, *v = k + kd, *a = v + kd, *o = a + qd;
    double *h1 = o + H, *n2 = h1 + H, *t = n2 + H, *f = t + H;
    double *g = f + H, *u = g + I, *m = u + I;
    int rc;

    qo_rms_norm(h, L->w_in, H, D->eps, n1);
    rc = qo_matvec(L->fmt_qkv, L->Wq, qd, H, n1, 1, 0, qd, q, NULL);
    if (!rc) rc = qo_matvec(L->fmt_qkv, L->Wk, kd, H, n1, 1, 0, kd, k, NULL);
    if (!rc) rc = qo_matvec(L->fmt_qkv, L->Wv, kd, H, n1, 1, 0, kd, v, NULL);
    if (!rc) rc = qo_attn_seq1(v, D->n_q_heads, D->n_kv_heads, D->head_dim, a);
    if (!rc) rc = qo_matvec(L->fmt_o, L->Wo, H, qd, a, 1, 0, H, o, NULL);
    if (rc) { free(buf); return rc; }

    memcpy(h1, h, sizeof(double) * (size_t)H);
    if (D->post_norms) {
        qo_rms_norm(o, L->w_post_attn, H, D->eps, t);
        qo_residual_add(h1, t, H);
    } else {
        qo_residual_add(h1, o, H);
    }
    qo_rms_norm(h1, L->w_pre_ffn, H, D->eps, n2);
    rc = qo_ffn(L->fmt_gu, L->Wg, L->Wu, L->fmt_down, L->Wd, H, I, n2, g, u, m, f,
                T ? T->bound_f : NULL);
    if (rc) { free(buf); return rc; }
    memcpy(h_out, h1, sizeof(double) * (size_t)H);
    if (D->post_norms) {
        qo_rms_norm(f, L->w_post_ffn, H, D->eps, t);
        qo_residual_add(h_out, t, H);
    } else {
        qo_residual_add(h_out, f, H);
    }

    if (T) {
        if (T->n1) memcpy(T->n1, n1, sizeof(double) * (size_t)H);
        if (T->q) memcpy(T->q, q, sizeof(double) * (size_t)qd);
        if (T->k) memcpy(T->k, k, sizeof(double) * (size_t)kd);
        if (T->v) memcpy(T->v, v, sizeof(double) * (size_t)kd);
        if (T->attn) memcpy(T->attn, a, sizeof(double) * (size_t)qd);
        if (T->o) memcpy(T->o, o, sizeof(double) * (size_t)H);
        if (T->h1) memcpy(T->h1, h1, sizeof(double) * (size_t)H);
        if (T->n2) memcpy(T->n2, n2, sizeof(double) * (size_t)H);
        if (T->g) memcpy(T->g, g, sizeof(double) * (size_t)I);
        if (T->u) memcpy(T->u, u, sizeof(double) * (size_t)I);
        if (T->m) memcpy(T->m, m, sizeof(double) * (size_t)I);
        if (T->f) memcpy(T->f, f, sizeof(double) * (size_t)H);
    }
    free(buf);
    return 0;
}

/* ---------------------------------------------------------------------------
 * One decoder layer at sequence position pos with a KV cache ([compute]
 * §Architecture decode: norm -> QKV -> attend -> O -> FFN, and §Shaders rows
 * "RoPE" (rope_at_pos) and "Attention" (kv_append, kv_attention); [engine]
 * §BLAS-Fused Attention).  The same steps as qo_layer_forward with the
 * attention of a real decode step in place of the sequence-1 broadcast:
 *   n1 = rms_norm(h, w_in)
 *   q, k, v = Wq n1, Wk n1, Wv n1
 *   q <- rope(q, pos), k <- rope(k, pos)        (qo_rope, rot_dim, base)
 *   caches[pos] <- k, v                          (qo_kv_append)
 *   a  = attention of q over positions 0..pos    (qo_kv_attention, scale,
 *                                                 softcap)
 *   o  = Wo a, then the post-attention part of qo_layer_forward unchanged.
 * At pos = 0 the rotation angle is 0 (q and k unchanged) and the softmax is
 * over one key (weight exactly 1), so the result equals qo_layer_forward's.
 * The caches are [n_kv_heads][max_seq][head_dim] and are updated in place.
 * ------------------------------------------------------------------------- */
typedef struct {
    double *k_cache, *v_cache;
    int64_t max_seq, pos;
    int rot_dim;
    double rope_base, scale, softcap;
} qo_kv;

int qo_layer_forward_kv(const qo_layer *L, const qo_dims *D, qo_kv *KV, const double *h,
                        double *h_out, qo_trace *T)
{
    int64_t H = D->hidden, I = D->inter;
    int64_t qd = (int64_t)D->n_q_heads * D->head_dim;
    int64_t kd = (int64_t)D->n_kv_heads * D->head_dim;
    if (KV->pos < 0 || KV->pos >= KV->max_seq) return -1;
    size_t need = (size_t)(H * 6 + qd * 2 + kd * 2 + I * 3);
    double *buf = (double *)malloc(sizeof(double) * need);
    if (!buf) return -2;
    double *n1 = buf, *q = n1 + H, *k = q + qd, *v = k + kd, *a = v + kd, *o = a + qd;
    double *h1 = o + H, *n2 = h1 + H, *t = n2 + H, *f = t + H;
    double *g = f + H, *u = g + I, *m = u + I;
    int rc;

    qo_rms_norm(h, L->w_in, H, D->eps, n1);
    rc = qo_matvec(L->fmt_qkv, L->Wq, qd, H, n1, 1, 0, qd, q, NULL);
    if (!rc) rc = qo_matvec(L->fmt_qkv, L->Wk, kd, H, n1, 1, 0, kd, k, NULL);
    if (!rc) rc = qo_matvec(L->fmt_qkv, L->Wv, kd, H, n1, 1, 0, kd, v, NULL);
    if (!rc) rc = qo_rope(q, D->n_q_heads, D->head_dim, KV->rot_dim, KV->pos, KV->rope_base);
    if (!rc) rc = qo_rope(k, D->n_kv_heads, D->head_dim, KV->rot_dim, KV->pos, KV->rope_base);
    if (!rc) rc = qo_kv_append(KV->k_cache, KV->v_cache, k, v, D->n_kv_heads, D->head_dim,
                               KV->max_seq, KV->pos);
    if (!rc) rc = qo_kv_attention(q, KV->k_cache, KV->v_cache, D->n_q_heads, D->n_kv_heads,
                                  D->head_dim, KV->max_seq, KV->pos + 1, KV->scale, KV->softcap,
                                  a, NULL, NULL);
    if (!rc) rc = qo_matvec(L->fmt_o, L->Wo, H, qd, a, 1, 0, H, o, NULL);
    if (rc) { free(buf); return rc; }

    memcpy(h1, h, sizeof(double) * (size_t)H);
    if (D->post_norms) {
        qo_rms_norm(o, L->w_post_attn, H, D->eps, t);
        qo_residual_add(h1, t, H);
    } else {
        qo_residual_add(h1, o, H);
    }
    qo_rms_norm(h1, L->w_pre_ffn, H, D->eps, n2);
    rc = qo_ffn(L->fmt_gu, L->Wg, L->Wu, L->fmt_down, L->Wd, H, I, n2, g, u, m, f,
                T ? T->bound_f : NULL);
    if (rc) { free(buf); return rc; }
    memcpy(h_out, h1, sizeof(double) * (size_t)H);
    if (D->post_norms) {
        qo_rms_norm(f, L->w_post_ffn, H, D->eps, t);
        qo_residual_add(h_out, t, H);
    } else {
        qo_residual_add(h_out, f, H);
    }

    if (T) {
        if (T->n1) memcpy(T->n1, n1, sizeof(double) * (size_t)H);
        if (T->q) memcpy(T->q, q, sizeof(double) * (size_t)qd);
        if (T->k) memcpy(T->k, k, sizeof(double) * (size_t)kd);
        if (T->v) memcpy(T->v, v, sizeof(double) * (size_t)kd);
        if (T->attn) memcpy(T->attn, a, sizeof(double) * (size_t)qd);
        if (T->o) memcpy(T->o, o, sizeof(double) * (size_t)H);
        if (T->h1) memcpy(T->h1, h1, sizeof(double) * (size_t)H);
        if (T->n2) memcpy(T->n2, n2, sizeof(double) * (size_t)H);
        if (T->g) memcpy(T->g, g, sizeof(double) * (size_t)I);
        if (T->u) memcpy(T->u, u, sizeof(double) * (size_t)I);
        if (T->m) memcpy(T->m, m, sizeof(double) * (size_t)I);
        if (T->f) memcpy(T->f, f, sizeof(double) * (size_t)H);
    }
    free(buf);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Top-k indices of v by value, descending; equal values keep the lower index
 * first ([perf] §Production Benchmark "top 5" predictions).  Plain repeated
 * selection: k passes over v.
 * ------------------------------------------------------------------------- */
int qo_topk(const double *v, int64_t n, int k, int64_t *idx)
{
    if (k < 0 || k > n) return -1;
    for (int j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t i = 0; i < n; ++i) {
            int taken = 0;
            for (int p = 0; p < j; ++p)
                if (idx[p] == i) { taken = 1; break; }
            if (taken) continue;
            if (best < 0 || v[i] > v[best]) best = i;
        }
        idx[j] = best;
    }
    return 0;
}
