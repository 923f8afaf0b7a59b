/*
 * orc.c -- the ORACLE for the speculative-decoding verify pass.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's smoke
 * check and the CPU-baseline leg of the benchmark may load this library.  It shares no
 * source, header, table or helper with the CUDA library and includes none of its files.
 *
 * Everything here is the plainest possible CPU restatement, in IEEE double precision,
 * of what the verify pass computes.  Sources (cited by page title and section):
 *
 *   [P1] "100 tokens per second from a 27B model on a 24 GB AMD card" (curriculo.me),
 *        sections "The wall" and "How speculative decoding gets past a per-token wall".
 *   [P2] "Decode is memory-bound: the ~59 tok/s ceiling on an RTX 4090, and how
 *        speculative decoding gets past it" (trefon.com), sections "The ceiling",
 *        "Speculative decoding" and "Two things the math says to do".
 *   [P3] Hacker News thread on speculative decoding (hn.shard-db.dev, item 49596054),
 *        the comments explaining parallel verification ("D E F" example and the
 *        [4, vocabulary_size] output tensor).
 *
 * Readings taken where the pages are silent are marked READING and listed in the
 * design notes of the repository.
 *
 * Pins (what ties this file to something other than itself) live in tests/: brute
 * force against a dense numpy matmul, closed forms of special cases, the worked greedy
 * example of [P3], Monte-Carlo exactness of the sampled output distribution, the
 * E[tokens per pass] table of [P2] and the Philox known-answer vectors.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------ */
/* Number formats, decoded from their definitions.                                      */
/* ------------------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32 (8 exponent bits, bias 127, 7 fraction). */
double orc_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1, e = (b >> 7) & 0xff, m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);                /* m * 2^-126 * 2^-7 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134);     /* (1 + m/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* ------------------------------------------------------------------------------------ */
/* Verify linear: one read of a block-quantised 4-bit weight matrix applied to the K+1  */
/* activation columns of a verify window ([P1] "How speculative decoding gets past a     */
/* per-token wall": the weights are read once and applied to a K-wide batch;            */
/* [P3]: every layer runs once over all window positions).                              */
/*                                                                                      */
/* Weight format: 4-bit code c in 0..15 with value s * (c - 8), one fp16 scale s per 32 */
/* consecutive inputs of an output row.  Storage (READING: the pages fix none):         */
/*   codes [out][in/2] bytes, input 2t in the low nibble and 2t+1 in the high nibble;   */
/*   scales[out][in/32] fp16 bit patterns.                                              */
/* Activations x[C][in] are bfloat16 bit patterns; the result is                        */
/*   y[c][j] = sum_i s[j][i/32] * (code[j][i] - 8) * x[c][i]                            */
/* and a[c][j] = sum_i |s * (code - 8) * x| (the scale of the parity tolerance).        */
/* ------------------------------------------------------------------------------------ */
void orc_verify_linear(const uint8_t *codes, const uint16_t *scales, int64_t in_f,
                       int64_t out_f, const uint16_t *x_bf16, int64_t C, double *y,
                       double *a, int nthreads)
{
    double *x = (double *)malloc(sizeof(double) * (size_t)(C * in_f));
    for (int64_t t = 0; t < C * in_f; ++t)
        x[t] = orc_bf16_to_f64(x_bf16[t]);
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)(2 * C));
#pragma omp for schedule(static)
        for (int64_t j = 0; j < out_f; ++j) {
            for (int64_t c = 0; c < 2 * C; ++c) acc[c] = 0.0;
            for (int64_t i = 0; i < in_f; ++i) {
                uint8_t byte = codes[j * (in_f / 2) + i / 2];
                int code = (i & 1) ? (byte >> 4) : (byte & 15);
                double w = orc_f16_to_f64(scales[j * (in_f / 32) + i / 32]) * (double)(code - 8);
                for (int64_t c = 0; c < C; ++c) {
                    double t = w * x[c * in_f + i];
                    acc[c] += t;
                    acc[C + c] += fabs(t);
                }
            }
            for (int64_t c = 0; c < C; ++c) {
                y[c * out_f + j] = acc[c];
                if (a) a[c * out_f + j] = acc[C + c];
            }
        }
        free(acc);
    }
    free(x);
}

/* ------------------------------------------------------------------------------------ */
/* Sampler: temperature, min-p and top-p ([P2] "Two things the math says to do": the    */
/* production settings temperature 0.6, top-p 0.95, min-p 0.05; [P1] "The last mile":   */
/* the sampled path at temperature 0.6 and top-p 0.95).                                 */
/*                                                                                      */
/* READING (the pages give only the constants):                                         */
/*   1. z = logit / T, p = softmax(z) in double;                                        */
/*   2. min-p keeps v iff p[v] >= min_p * max(p);                                       */
/*   3. top-p orders tokens by (p descending, id ascending) and keeps the shortest      */
/*      prefix whose mass reaches top_p, the crossing token included; top_p >= 1 keeps  */
/*      everything;                                                                     */
/*   4. both filters read the same un-renormalised p; the kept set is their             */
/*      intersection, which is again a prefix of that order;                            */
/*   5. the kept probabilities are renormalised to sum to one.                          */
/* greedy != 0 returns the one-hot distribution of the argmax (lowest id on ties).      */
/* The returned flags mark decisions that sit within a rounding tolerance of their      */
/* boundary (bit 0: min-p, relative 1e-6; bit 1: top-p, 1e-5 of the mass), where an     */
/* implementation in another precision may legitimately decide the other way.           */
/* ------------------------------------------------------------------------------------ */
typedef struct { double p; int64_t id; } orc_rank_t;

static int orc_rank_cmp(const void *A, const void *B)
{
    const orc_rank_t *a = (const orc_rank_t *)A, *b = (const orc_rank_t *)B;
    if (a->p > b->p) return -1;
    if (a->p < b->p) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

int orc_sampler_row(const float *logits, int64_t V, double T, double top_p, double min_p,
                    int greedy, double *probs, int32_t *argmax_out, int64_t *n_kept_out)
{
    int flags = 0;
    int64_t am = 0;
    for (int64_t v = 1; v < V; ++v)
        if (logits[v] > logits[am]) am = v;          /* strict: lowest id wins ties */
    if (argmax_out) *argmax_out = (int32_t)am;
    if (greedy) {
        for (int64_t v = 0; v < V; ++v) probs[v] = (v == am) ? 1.0 : 0.0;
        if (n_kept_out) *n_kept_out = 1;
        return 0;
    }
    double zmax = (double)logits[am] / T, Z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        probs[v] = exp((double)logits[v] / T - zmax);
        Z += probs[v];
    }
    for (int64_t v = 0; v < V; ++v) probs[v] /= Z;
    double pmax = probs[am];

    char *keep = (char *)calloc((size_t)V, 1);
    for (int64_t v = 0; v < V; ++v) {
        double thr = min_p * pmax;
        keep[v] = probs[v] >= thr;
        if (min_p > 0.0 && fabs(probs[v] - thr) <= 1e-6 * thr) flags |= 1;
    }
    if (top_p < 1.0) {
        orc_rank_t *r = (orc_rank_t *)malloc(sizeof(orc_rank_t) * (size_t)V);
        for (int64_t v = 0; v < V; ++v) { r[v].p = probs[v]; r[v].id = v; }
        qsort(r, (size_t)V, sizeof(orc_rank_t), orc_rank_cmp);
        double cum = 0.0;
        int64_t cut = V;                              /* number of ranks top-p keeps */
        for (int64_t t = 0; t < V; ++t) {
            double before = cum;
            cum += r[t].p;
            if (cum >= top_p) {
                cut = t + 1;
                if (fabs(cum - top_p) < 1e-5 || fabs(before - top_p) < 1e-5) flags |= 2;
                break;
            }
        }
        for (int64_t t = cut; t < V; ++t) keep[r[t].id] = 0;
        free(r);
    }
    double S = 0.0;
    int64_t nk = 0;
    for (int64_t v = 0; v < V; ++v)
        if (keep[v]) { S += probs[v]; ++nk; }
    for (int64_t v = 0; v < V; ++v) probs[v] = keep[v] ? probs[v] / S : 0.0;
    free(keep);
    if (n_kept_out) *n_kept_out = nk;
    return flags;
}

void orc_sampler(const float *logits, int64_t rows, int64_t V, double T, double top_p,
                 double min_p, int greedy, double *probs, int32_t *argmax, int64_t *n_kept,
                 int32_t *flags, int nthreads)
{
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r)
        flags[r] = orc_sampler_row(logits + r * V, V, T, top_p, min_p, greedy, probs + r * V,
                                   argmax ? argmax + r : NULL, n_kept ? n_kept + r : NULL);
}

/* ------------------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1,   */
/* 2, 3", SC'11), written from the paper's definition: a 4-word counter, a 2-word key,  */
/* ten rounds of two 32x32->64 multiplications with the round constants, the key        */
/* advanced by the Weyl constants between rounds.                                       */
/* ------------------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniforms of window w (absolute index) and position i (READING: the pages name no
 * generator): key = seed, counter = (w low, w high, i, 0).  Word 0 gives the acceptance
 * uniform u, word 1 the resampling uniform u'; each is (word >> 8) * 2^-24 in [0, 1). */
void orc_uniforms(uint64_t seed, uint64_t window, uint32_t pos, double *u, double *u2)
{
    uint32_t ctr[4] = {(uint32_t)window, (uint32_t)(window >> 32), pos, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    orc_philox4x32_10(ctr, key, r);
    *u = ldexp((double)(r[0] >> 8), -24);
    *u2 = ldexp((double)(r[1] >> 8), -24);
}

/* ------------------------------------------------------------------------------------ */
/* Acceptance ([P1] "How speculative decoding gets past a per-token wall"; [P2]         */
/* "Speculative decoding"; [P3] the "D E F" example).                                   */
/*                                                                                      */
/* Greedy (q == NULL): emit x_i while x_i equals the target's argmax at position i; at  */
/* the first mismatch j emit argmax_j; if all k drafts match emit argmax_k.  The        */
/* argmax comes from target_argmax when given, else from p (lowest id on ties).         */
/*                                                                                      */
/* Sampled: for i = 0..k-1 accept x_i iff u_i * q_i(x_i) < p_i(x_i), which is accepting */
/* with probability min(1, p/q); at the first rejection j emit a draw from the          */
/* normalised positive part of p_j - q_j using u'_j; if all k are accepted, the target's */
/* own token caps the window: a draw from p_k using u'_k.                               */
/* A draw from weights r with total R emits the smallest v whose running sum C_v        */
/* exceeds u' * R.                                                                      */
/*                                                                                      */
/* Status bits (READING for inputs the pages do not consider):                          */
/*   1 draft id outside [0, V): that position is rejected;                              */
/*   2 q_i(x_i) == 0 for a drafted token (the test u*q < p still decides);              */
/*   4 a probability read is NaN, infinite, negative or above one (clamped into [0,1]);  */
/*   8 the residual has zero mass (READING: the draw falls back to p_j);                */
/*  16 the distribution drawn from has zero mass: no token is emitted there.            */
/* near[w] is set when a draw's u' lies within 1e-6 of either edge of the chosen        */
/* token's interval [C_{v-1}/R, C_v/R): there another summation order may pick a        */
/* neighbour.  margin[w] (optional) is that distance itself (+inf without a draw).      */
/* ------------------------------------------------------------------------------------ */
static double orc_prob(float f, int *st)
{
    double d = (double)f;
    if (!(d >= 0.0 && d <= 1.0)) {                 /* NaN, negative, infinite or > 1 */
        *st |= 4;
        if (d > 1.0) return 1.0;
        return 0.0;
    }
    return d;
}

static int64_t orc_draw(const float *pr, const float *qr, int64_t V, double u2, int *st,
                        int *near, double *margin)
{
    double *r = (double *)malloc(sizeof(double) * (size_t)V);
    double R = 0.0;
    if (qr) {
        for (int64_t v = 0; v < V; ++v) {
            double d = orc_prob(pr[v], st) - orc_prob(qr[v], st);
            r[v] = d > 0.0 ? d : 0.0;
            R += r[v];
        }
        if (!(R > 0.0)) *st |= 8;
    }
    if (!qr || !(R > 0.0)) {
        R = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            r[v] = orc_prob(pr[v], st);
            R += r[v];
        }
    }
    int64_t tok = -1;
    if (R > 0.0) {
        double t = u2 * R, Cprev = 0.0, Cv = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            Cv = Cprev + r[v];
            if (Cv > t) { tok = v; break; }
            Cprev = Cv;
        }
        if (tok < 0) {                      /* only through rounding: last nonzero weight */
            for (int64_t v = V - 1; v >= 0; --v)
                if (r[v] > 0.0) { tok = v; break; }
            Cprev = R - r[tok];
            Cv = R;
        }
        double m = fmin(fabs(u2 - Cprev / R), fabs(u2 - Cv / R));
        if (m < *margin) *margin = m;
        if (m < 1e-6) *near = 1;
    } else {
        *st |= 16;
    }
    free(r);
    return tok;
}

static int64_t orc_argmax_row(const float *row, int64_t V, int *st)
{
    int64_t am = -1;
    for (int64_t v = 0; v < V; ++v) {
        float f = row[v];
        if (f != f) { *st |= 4; continue; }
        if (am < 0 || f > row[am]) am = v;
    }
    return am;
}

void orc_accept(const float *p, const int64_t *p_rows, const float *q, const int64_t *q_rows,
                const int32_t *target_argmax, const int32_t *draft, int64_t n, int k,
                int64_t V, uint64_t seed, uint64_t window_offset, const float *uniforms,
                int32_t *out_tokens, int32_t *n_emitted, int32_t *status, int32_t *near,
                double *margin, int nthreads)
{
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 16)
    for (int64_t w = 0; w < n; ++w) {
        int st = 0, nr = 0, ne = 0;
        double mg = INFINITY;
        int32_t *tok = out_tokens + w * (k + 1);
        for (int i = 0; i <= k; ++i) tok[i] = -1;
        const float *prow[65], *qrow[65];
        for (int i = 0; i <= k; ++i)
            prow[i] = p + (p_rows ? p_rows[w * (k + 1) + i] : w * (k + 1) + i) * V;
        if (q)
            for (int i = 0; i < k; ++i)
                qrow[i] = q + (q_rows ? q_rows[w * k + i] : w * k + i) * V;
        if (!q) {
            int i = 0;
            for (; i <= k; ++i) {
                int64_t a = target_argmax ? target_argmax[w * (k + 1) + i]
                                          : orc_argmax_row(prow[i], V, &st);
                if (a < 0 || a >= V) { st |= 16; break; }   /* no usable target token */
                if (i < k && draft[w * k + i] == a) { tok[ne++] = (int32_t)a; continue; }
                if (i < k && (draft[w * k + i] < 0 || draft[w * k + i] >= V)) st |= 1;
                tok[ne++] = (int32_t)a;
                break;
            }
        } else {
            int i = 0;
            for (; i < k; ++i) {
                double u, u2;
                if (uniforms) {
                    u = uniforms[(w * (k + 1) + i) * 2];
                    u2 = uniforms[(w * (k + 1) + i) * 2 + 1];
                } else {
                    orc_uniforms(seed, window_offset + (uint64_t)w, (uint32_t)i, &u, &u2);
                }
                int32_t x = draft[w * k + i];
                int accept = 0;
                if (x < 0 || x >= V) {
                    st |= 1;
                } else {
                    double pv = orc_prob(prow[i][x], &st), qv = orc_prob(qrow[i][x], &st);
                    if (qv == 0.0) st |= 2;
                    accept = u * qv < pv;
                }
                if (accept) { tok[ne++] = x; continue; }
                int64_t t = orc_draw(prow[i], qrow[i], V, u2, &st, &nr, &mg);
                if (t >= 0) tok[ne++] = (int32_t)t;
                break;
            }
            if (i == k) {
                double u, u2;
                if (uniforms) {
                    u = uniforms[(w * (k + 1) + k) * 2];
                    u2 = uniforms[(w * (k + 1) + k) * 2 + 1];
                } else {
                    orc_uniforms(seed, window_offset + (uint64_t)w, (uint32_t)k, &u, &u2);
                }
                (void)u;
                int64_t t = orc_draw(prow[k], NULL, V, u2, &st, &nr, &mg);
                if (t >= 0) tok[ne++] = (int32_t)t;
            }
        }
        n_emitted[w] = ne;
        status[w] = st;
        if (near) near[w] = nr;
        if (margin) margin[w] = mg;
    }
}

/* ------------------------------------------------------------------------------------ */
/* KV-read attention of a verify window ([P2] "The ceiling": at long context attention  */
/* reads the whole KV cache on every pass, a second stream beside the weights; [P1]     */
/* "The wall" and "The last mile": the target's cache held as q8_0 keys and q4_0        */
/* values at 32K context).                                                              */
/*                                                                                      */
/* Cache format (READING: the pages name the formats only):                             */
/*   keys:   8-bit code q in -128..127 with value s * q, one fp16 scale s per 32        */
/*           consecutive dimensions of a position;                                      */
/*           k_codes [Hkv][ld][D] int8, k_scales [Hkv][ld][D/32] fp16 bits;             */
/*   values: 4-bit code c in 0..15 with value s * (c - 8), one fp16 scale per 32        */
/*           dimensions; v_codes [Hkv][ld][D/2] bytes (dimension 2t in the low nibble, */
/*           2t+1 in the high one), v_scales [Hkv][ld][D/32] fp16 bits.                 */
/* The window's C positions sit at n_past .. n_past+C-1 of the cache (their keys and    */
/* values already written), and window position c sees cache positions 0 .. n_past+c   */
/* (causal).  Query head h reads kv head h / (Hq/Hkv) (consecutive groups).  Queries   */
/* q [C][Hq][D] are bfloat16 bit patterns.  For every (c, h):                           */
/*   s_j = scale * sum_i q[i] k_j[i],  w_j = exp(s_j - max s),                          */
/*   o[d] = sum_j w_j v_j[d] / sum_j w_j,  a[d] = sum_j w_j |v_j[d]| / sum_j w_j        */
/* (a is the scale of the parity tolerance).  o and a are [C][Hq][D] doubles.           */
/* ------------------------------------------------------------------------------------ */
void orc_kv_attention(const uint16_t *q_bf16, const int8_t *k_codes, const uint16_t *k_scales,
                      const uint8_t *v_codes, const uint16_t *v_scales, int64_t Hq,
                      int64_t Hkv, int64_t D, int64_t ld, int64_t n_past, int64_t C,
                      double scale, double *o, double *a, int nthreads)
{
    int64_t G = Hq / Hkv, nb = D / 32, L = n_past + C;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)D);
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double *k = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t row = 0; row < C * Hq; ++row) {
            int64_t c = row / Hq, h = row % Hq, g = h / G, n = n_past + c + 1;
            for (int64_t i = 0; i < D; ++i) q[i] = orc_bf16_to_f64(q_bf16[row * D + i]);
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                const int8_t *kc = k_codes + (g * ld + j) * D;
                const uint16_t *ks = k_scales + (g * ld + j) * nb;
                for (int64_t i = 0; i < D; ++i)
                    k[i] = orc_f16_to_f64(ks[i / 32]) * (double)kc[i];
                double dot = 0.0;
                for (int64_t i = 0; i < D; ++i) dot += q[i] * k[i];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            for (int64_t d = 0; d < D; ++d) {
                double acc = 0.0, mag = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    uint8_t byte = v_codes[(g * ld + j) * (D / 2) + d / 2];
                    int code = (d & 1) ? (byte >> 4) : (byte & 15);
                    double v = orc_f16_to_f64(v_scales[(g * ld + j) * nb + d / 32]) * (double)(code - 8);
                    acc += s[j] * v;
                    mag += s[j] * fabs(v);
                }
                o[row * D + d] = acc / l;
                if (a) a[row * D + d] = mag / l;
            }
        }
        free(q);
        free(s);
        free(k);
    }
}

/* ------------------------------------------------------------------------------------ */
/* Quantisation of the window's keys and values on their way into the cache ([P1] "The  */
/* wall": the cache is held as q8_0 keys and q4_0 values).  READING: the pages name the  */
/* formats only; their definitions are those of the llama.cpp block types of the same    */
/* names, in fp32 arithmetic, per block of 32 consecutive values:                        */
/*   q8_0: d = max|x| / 127, q = round-half-away(x * (1/d)) (0 when d = 0);               */
/*   q4_0: m = the value of largest magnitude (the first on ties), d = m / -8,            */
/*         c = min(15, trunc(x * (1/d) + 8.5)) (8 when d = 0).                            */
/* d is stored as fp16 (round to nearest even); codes use the fp32 d.                    */
/* ------------------------------------------------------------------------------------ */

/* fp32 -> IEEE binary16 bits, round to nearest even, from the two formats' definitions. */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u, ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) return (uint16_t)(sign | (ax > 0x7f800000u ? 0x7e00u : 0x7c00u));
    if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);       /* >= 65520: infinity */
    if (ax < 0x38800000u) {                                          /* below 2^-14 */
        double m = (double)fabsf(f) * 16777216.0;                    /* units of 2^-24, exact */
        return (uint16_t)(sign | (uint32_t)nearbyint(m));            /* ties to even */
    }
    uint32_t e = (ax >> 23) - 127u + 15u, mant = ax & 0x7fffffu;
    uint32_t h = (e << 10) | (mant >> 13), rem = mant & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;      /* carry may bump e */
    return (uint16_t)(sign | h);
}

/* rows x D fp32 keys and values (D a multiple of 32) -> k codes [rows][D], k scales
 * [rows][D/32], v codes [rows][D/2] (dimension 2t in the low nibble), v scales [rows][D/32]. */
void orc_kv_quantize(const float *k, const float *v, int64_t rows, int64_t D, int8_t *kc,
                     uint16_t *ks, uint8_t *vc, uint16_t *vs)
{
    int64_t nb = D / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xk = k + r * D + 32 * b, *xv = v + r * D + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i)
                if (fabsf(xk[i]) > amax) amax = fabsf(xk[i]);
            float d = amax / 127.0f, id = d != 0.0f ? 1.0f / d : 0.0f;
            ks[r * nb + b] = orc_f32_to_f16(d);
            for (int i = 0; i < 32; ++i) {
                float t = xk[i] * id;
                kc[r * D + 32 * b + i] = (int8_t)roundf(t);
            }
            float mabs = 0.0f, m = 0.0f;
            for (int i = 0; i < 32; ++i)
                if (fabsf(xv[i]) > mabs) {
                    mabs = fabsf(xv[i]);
                    m = xv[i];
                }
            float dv = m / -8.0f, idv = dv != 0.0f ? 1.0f / dv : 0.0f;
            vs[r * nb + b] = orc_f32_to_f16(dv);
            for (int i = 0; i < 32; ++i) {
                float t = xv[i] * idv;
                t = t + 8.5f;
                int c = (int)t;
                if (c > 15) c = 15;
                int dim = (int)(32 * b + i);
                uint8_t *byte = vc + r * (D / 2) + dim / 2;
                if (dim & 1)
                    *byte = (uint8_t)((*byte & 0x0f) | (c << 4));
                else
                    *byte = (uint8_t)((*byte & 0xf0) | c);
            }
        }
    }
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
