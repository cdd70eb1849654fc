/*
 * kvs oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU model of what the streamed paged
 * attention path computes.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library; the product
 * (the CUDA library under host_streamed_paged_gb300/) never calls it and
 * shares no code, header or table with it.
 *
 * What is modelled, with the passage each part follows:
 *
 *  - Each layer attends over all of its history; streaming changes only
 *    where pages live and when they are copied (Adaptive KV
 *    Streaming for llama.cpp, section "Adaptive KV streaming"; the V2 README,
 *    section "KV data movement and attention").  Streaming therefore does not
 *    enter the mathematics: the oracle is dense softmax attention over the
 *    dequantised history, written out as its definition in fp64
 *    (kvs_oracle_attend).  Row r of a span sits at position pos0 + r and sees
 *    keys 0 .. pos0 + r (inclusive causal convention, the new rows' K/V are
 *    written before they attend).  Query head h reads kv head h / (Hq / Hk).
 *
 *  - K is cached as Q8_0 and V as Q4_0 (V2 README, "Results and quick start"
 *    and its server example's cache-type options).  Both
 *    are 32-element blocks with one fp16 scale.  Q8_0: d = max|x| / 127,
 *    code = round-half-away(x / d) as int8.  Q4_0: m = the element of largest
 *    magnitude (first one on ties) with its sign, d = m / -8,
 *    code = min(15, trunc(x / d + 8.5)); the nibble of element i < 16 is the
 *    low half of byte i, element i + 16 the high half.  Both encoders do
 *    their arithmetic in IEEE fp32 (1/d as a correctly rounded fp32
 *    reciprocal, products in fp32), because fp32 is where the code decision
 *    is taken; decoding is code * fp16(d) (Q8_0) and (code - 8) * fp16(d)
 *    (Q4_0), evaluated in fp64.
 *
 *  - The page layout (V2 README, "KV data movement and attention": pages of
 *    256 tokens each, whose K/V byte sizes follow the quant
 *    types).  The byte order inside a page is this library's own choice and
 *    is spelled out at kvs_oracle_encode_page; the oracle writes it from that
 *    definition only, to pin the bytes the device path stores.
 *
 *  - The split/combine identity (V2 README, "Keep the stock attention order":
 *    one ordered history, then the stock-style final reduction; PR "port
 *    adaptive KV streaming", review: the chunk-normalisation step must guard
 *    a zero denominator): kvs_oracle_attend_partial gives (m, l, o) over a
 *    key range and kvs_oracle_combine merges them with the log-sum-exp rule
 *    M = max m_s, L = sum l_s e^(m_s - M), o = sum o_s e^(m_s - M) / L.
 *
 * Compile without -ffast-math and with -ffp-contract=off so that the fp32
 * quantiser steps are single IEEE operations on every host architecture.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ fp16 */

/* Round-to-nearest-even right shift of an unsigned integer. */
static uint32_t rne_shift(uint32_t v, int s) {
    if (s <= 0) return v;
    if (s > 31) return 0;
    uint32_t q = v >> s;
    uint32_t rem = v & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return q;
}

/* IEEE binary32 -> binary16, round to nearest even (IEEE 754-2008 s. 4.3.1). */
uint16_t kvs_oracle_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ex = (x >> 23) & 0xffu;
    uint32_t man = x & 0x7fffffu;
    if (ex == 0xffu) return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0u));
    if (ex == 0) return (uint16_t)sign; /* fp32 zero/subnormal: far below 2^-25 */
    int e = (int)ex - 127;
    uint32_t full = man | 0x800000u; /* 24-bit significand, value = full * 2^(e-23) */
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    if (e >= -14) {
        uint32_t r = rne_shift(full, 13); /* 11-bit significand */
        if (r == 0x800u) { r >>= 1; e += 1; }
        if (e > 15) return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | ((uint32_t)(e + 15) << 10) | (r & 0x3ffu));
    }
    /* subnormal half: units of 2^-24; value/2^-24 = full * 2^(e+1) */
    uint32_t r = rne_shift(full, -(e + 1));
    return (uint16_t)(sign | r); /* r == 0x400 encodes the smallest normal */
}

/* IEEE binary16 -> binary32 (exact). */
float kvs_oracle_f16_to_f32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t ex = ((uint32_t)h >> 10) & 0x1fu;
    uint32_t man = (uint32_t)h & 0x3ffu;
    uint32_t x;
    if (ex == 0x1fu) {
        x = sign | 0x7f800000u | (man << 13);
    } else if (ex == 0) {
        if (man == 0) {
            x = sign;
        } else { /* subnormal: man * 2^-24, exact in fp32 */
            float v = (float)man * (1.0f / 16777216.0f);
            memcpy(&x, &v, 4);
            x |= sign;
        }
    } else {
        x = sign | ((ex - 15u + 127u) << 23) | (man << 13);
    }
    float f;
    memcpy(&f, &x, 4);
    return f;
}

/* ---------------------------------------------------------- quantisers */

/* Q8_0 block: 32 fp32 values -> 32 int8 codes + fp16 scale. */
void kvs_oracle_q8_0_block(const float *x, int8_t *q, uint16_t *d16) {
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < 32; ++j) {
        float t = x[j] * id;
        q[j] = (int8_t)roundf(t);
    }
    *d16 = kvs_oracle_f32_to_f16(d);
}

/* Q4_0 block: 32 fp32 values -> 32 codes in 0..15 (unpacked) + fp16 scale. */
void kvs_oracle_q4_0_block(const float *x, uint8_t *q, uint16_t *d16) {
    float amax = 0.0f, mx = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float a = fabsf(x[j]);
        if (amax < a) { amax = a; mx = x[j]; }
    }
    float d = mx / -8.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < 32; ++j) {
        float t = x[j] * id;
        float u = t + 8.5f;
        int c = (int)u; /* truncation; u >= 0.5 for finite inputs */
        if (c > 15) c = 15;
        if (c < 0) c = 0;
        q[j] = (uint8_t)c;
    }
    *d16 = kvs_oracle_f32_to_f16(d);
}

/*
 * Quantise a whole history.  k, v: fp32 [T][Hk][D].  Outputs:
 *   kq int8 [T][Hk][D], kd fp16 bits [T][Hk][D/32],
 *   vq uint8 codes 0..15 [T][Hk][D] (unpacked), vd fp16 bits [T][Hk][D/32].
 */
void kvs_oracle_quantize_kv(int64_t T, int Hk, int D, const float *k, const float *v,
                            int8_t *kq, uint16_t *kd, uint8_t *vq, uint16_t *vd) {
    const int64_t nb = (int64_t)T * Hk * (D / 32);
    #pragma omp parallel for schedule(static) if (nb > 4096)
    for (int64_t b = 0; b < nb; ++b) {
        kvs_oracle_q8_0_block(k + b * 32, kq + b * 32, kd + b);
        kvs_oracle_q4_0_block(v + b * 32, vq + b * 32, vd + b);
    }
}

/*
 * Page bytes of page `page` (tokens page*P .. page*P+P-1) of a history of T
 * tokens.  The page is Hk consecutive head sections; head section g holds,
 * at these byte offsets (HS = P*D*13/8 bytes per section, NB = D/32):
 *   Kq  int8  at 0               byte of (token t, dim d):
 *                                ((t/16 * NB + d/32) * 16 + t%16) * 32 + d%32
 *                                (16-token groups; inside a group, one
 *                                32-byte line per (block, token))
 *   Ks  fp16  [P][NB]   at P*D   (token-major K scales)
 *   Vq  uint8 at P*D + P*D/16    byte of (byte row i = b*16 + c, token t):
 *                                ((t/32 * NB + b) * 16 + c) * 32 + t%32;
 *                                byte row b*16 + c holds the codes of dims
 *                                b*32+c (low nibble) and b*32+c+16 (high)
 *   Vs  fp16  [NB][P]   at P*D + P*D/16 + P*D/2 (dim-major V scales)
 * fp16 values are little-endian.  Token slots at or beyond T are zero bytes.
 */
static int64_t kq_at(int64_t t, int d, int NB) {
    return ((t / 16 * NB + d / 32) * 16 + t % 16) * 32 + d % 32;
}

static int64_t vq_at(int64_t t, int row, int NB) {
    return ((t / 32 * NB + row / 16) * 16 + row % 16) * 32 + t % 32;
}

void kvs_oracle_encode_page(int P, int Hk, int D, int64_t T, int64_t page,
                            const int8_t *kq, const uint16_t *kd, const uint8_t *vq,
                            const uint16_t *vd, uint8_t *out) {
    const int nbk = D / 32;
    const int64_t HS = (int64_t)P * D * 13 / 8;
    const int64_t ks_off = (int64_t)P * D;
    const int64_t vq_off = ks_off + (int64_t)P * D / 16;
    const int64_t vs_off = vq_off + (int64_t)P * D / 2;
    memset(out, 0, (size_t)(HS * Hk));
    for (int g = 0; g < Hk; ++g) {
        uint8_t *sec = out + g * HS;
        for (int t = 0; t < P; ++t) {
            int64_t tok = page * P + t;
            if (tok >= T) break;
            const int64_t row = tok * Hk + g;
            for (int d = 0; d < D; ++d) sec[kq_at(t, d, nbk)] = (uint8_t)kq[row * D + d];
            for (int b = 0; b < nbk; ++b) {
                uint16_t s = kd[row * nbk + b];
                sec[ks_off + ((int64_t)t * nbk + b) * 2 + 0] = (uint8_t)(s & 0xff);
                sec[ks_off + ((int64_t)t * nbk + b) * 2 + 1] = (uint8_t)(s >> 8);
                uint16_t sv = vd[row * nbk + b];
                sec[vs_off + ((int64_t)b * P + t) * 2 + 0] = (uint8_t)(sv & 0xff);
                sec[vs_off + ((int64_t)b * P + t) * 2 + 1] = (uint8_t)(sv >> 8);
                for (int c = 0; c < 16; ++c) {
                    uint8_t lo = vq[row * D + b * 32 + c];
                    uint8_t hi = vq[row * D + b * 32 + c + 16];
                    sec[vq_off + vq_at(t, b * 16 + c, nbk)] = (uint8_t)(lo | (hi << 4));
                }
            }
        }
    }
}

/* ----------------------------------------------------------- attention */

static double deq_k(const int8_t *kq, const uint16_t *kd, int64_t row, int D, int d) {
    return (double)kq[row * D + d] * (double)kvs_oracle_f16_to_f32(kd[row * (D / 32) + d / 32]);
}

static double deq_v(const uint8_t *vq, const uint16_t *vd, int64_t row, int D, int d) {
    return ((double)vq[row * D + d] - 8.0) * (double)kvs_oracle_f16_to_f32(vd[row * (D / 32) + d / 32]);
}

/*
 * Partial attention of one (row, head) over keys [k0, k1) clipped to the
 * row's causal limit: m = max score (-inf if no key), l = sum e^(s - m),
 * o[D] = sum e^(s - m) * v (unnormalised).  All fp64.
 */
static void partial_one(int Hk, int D, const int8_t *kq, const uint16_t *kd, const uint8_t *vq,
                        const uint16_t *vd, int G, const float *qrow, int h, int64_t k0,
                        int64_t k1, double scale, double *m_out, double *l_out, double *o) {
    const int g = h / G;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (k1 <= k0) { *m_out = -INFINITY; *l_out = 0.0; return; }
    double *s = (double *)malloc((size_t)(k1 - k0) * sizeof(double));
    double m = -INFINITY;
    for (int64_t j = k0; j < k1; ++j) {
        const int64_t row = j * Hk + g;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += (double)qrow[d] * deq_k(kq, kd, row, D, d);
        s[j - k0] = scale * acc;
        if (s[j - k0] > m) m = s[j - k0];
    }
    double l = 0.0;
    for (int64_t j = k0; j < k1; ++j) {
        const int64_t row = j * Hk + g;
        double w = exp(s[j - k0] - m);
        l += w;
        for (int d = 0; d < D; ++d) o[d] += w * deq_v(vq, vd, row, D, d);
    }
    free(s);
    *m_out = m;
    *l_out = l;
}

/*
 * Causal attention of R rows at positions pos0 .. pos0+R-1 over the
 * quantised history (T tokens; pos0 + R <= T).  q fp32 [R][Hq][D];
 * o fp64 [R][Hq][D] (normalised); lse fp64 [R][Hq] (natural log).
 * Returns 0, or -1 on invalid arguments.  n_threads <= 0: OpenMP default.
 */
int kvs_oracle_attend(int64_t T, int Hk, int D, const int8_t *kq, const uint16_t *kd,
                      const uint8_t *vq, const uint16_t *vd, int R, int Hq, const float *q,
                      int64_t pos0, double scale, double *o, double *lse, int n_threads) {
    if (Hk <= 0 || Hq % Hk != 0 || D % 32 != 0 || pos0 < 0 || pos0 + R > T) return -1;
    const int G = Hq / Hk;
    const int n = R * Hq;
    const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
    #pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int i = 0; i < n; ++i) {
        const int r = i / Hq, h = i % Hq;
        double m, l;
        double *orow = o + (int64_t)i * D;
        partial_one(Hk, D, kq, kd, vq, vd, G, q + (int64_t)i * D, h, 0, pos0 + r + 1, scale, &m,
                    &l, orow);
        for (int d = 0; d < D; ++d) orow[d] /= l;
        lse[i] = m + log(l);
    }
    return 0;
}

/*
 * Partial attention over keys [k0, k1) for every (row, head):
 * m, l fp64 [R][Hq]; o fp64 [R][Hq][D] unnormalised.
 */
int kvs_oracle_attend_partial(int64_t T, int Hk, int D, const int8_t *kq, const uint16_t *kd,
                              const uint8_t *vq, const uint16_t *vd, int R, int Hq, const float *q,
                              int64_t pos0, double scale, int64_t k0, int64_t k1, double *m,
                              double *l, double *o) {
    if (Hk <= 0 || Hq % Hk != 0 || D % 32 != 0 || pos0 < 0 || pos0 + R > T || k0 < 0) return -1;
    const int G = Hq / Hk;
    for (int i = 0; i < R * Hq; ++i) {
        const int r = i / Hq, h = i % Hq;
        int64_t hi = k1 < pos0 + r + 1 ? k1 : pos0 + r + 1;
        partial_one(Hk, D, kq, kd, vq, vd, G, q + (int64_t)i * D, h, k0, hi, scale, m + i, l + i,
                    o + (int64_t)i * D);
    }
    return 0;
}

/*
 * Log-sum-exp combine of n_splits partials of one (row, head), in split
 * order.  m, l [n_splits]; o_part [n_splits][D].  Splits with l == 0 (or
 * m == -inf) contribute nothing; if every split is empty, o = 0 and
 * lse = -inf.
 */
void kvs_oracle_combine(int n_splits, int D, const double *m, const double *l,
                        const double *o_part, double *o, double *lse) {
    double M = -INFINITY;
    for (int s = 0; s < n_splits; ++s)
        if (l[s] > 0.0 && m[s] > M) M = m[s];
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (M == -INFINITY) { *lse = -INFINITY; return; }
    double L = 0.0;
    for (int s = 0; s < n_splits; ++s) {
        if (!(l[s] > 0.0)) continue;
        double w = exp(m[s] - M);
        L += l[s] * w;
        for (int d = 0; d < D; ++d) o[d] += o_part[(int64_t)s * D + d] * w;
    }
    for (int d = 0; d < D; ++d) o[d] /= L;
    *lse = M + log(L);
}

/* Number of threads kvs_oracle_attend uses for a given n_threads argument. */
int kvs_oracle_threads(int n_threads) { return n_threads > 0 ? n_threads : omp_get_max_threads(); }

/* Array forms of the fp16 conversions (for exhaustive checks). */
void kvs_oracle_f32_to_f16_n(int64_t n, const float *in, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvs_oracle_f32_to_f16(in[i]);
}

void kvs_oracle_f16_to_f32_n(int64_t n, const uint16_t *in, float *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvs_oracle_f16_to_f32(in[i]);
}
