/*
 * CSA2 decode hot path -- the ORACLE.  Test infrastructure only.
 *
 * A plain, slow, obviously correct CPU restatement of what the CSA2 decode
 * path computes, in fp64 wherever the pages leave the precision open.  Only the
 * tests, the package's smoke check and the benchmark's CPU-baseline leg load
 * it; the product path (the CUDA library) never does, and the two share no
 * code, header, table or constant generator.
 *
 * Sources (web pages on the DeepSeek-V4.1-Flash technical report):
 *   [A] "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression"
 *       (en.mycoding.id), sections 2.3.2, 2.3.4 (HSI), 2.4.4 (FP4 Main KV
 *       Cache), 3.1 (890 B), 3.3.1-3.3.3 (readout, modes).
 *   [N] "DeepSeek-V4.1-Flash - Architecture" (notes.nimendra.online),
 *       section 2 (CSA2 modes table, layer schedule, main attention settings),
 *       section 3 (Hierarchical Sparse Indexer), section 4 (KV cache formats).
 *
 * Readings of points the pages leave open are marked READING below.
 * Functions whose arithmetic is a convention, not fixed by the pages, are
 * marked "parity unpinned": the RoPE pairing/base and the m=2 pooling form.
 *
 * bf16 inputs arrive as their uint16 bit patterns and are widened exactly.
 * Build: plain C11, -O2 -ffp-contract=off (no fused multiply-add anywhere),
 * optional OpenMP over independent outer loops.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define O_D 512        /* latent dim, key = value = latent          [N] sec.2 */
#define O_ROPE 64      /* RoPE'd tail channels (448 NoPE + 64 RoPE)  [A] 3.1  */
#define O_H 64         /* query heads                                 [N] sec.2 */
#define O_HI 32        /* indexer heads                               [N] sec.2 */
#define O_DI 128       /* indexer head dim                            [N] sec.2 */
#define O_GROUP 16     /* channels per E4M3 scale                     [N] sec.4 */
#define O_ENTRY 288    /* 256 B of E2M1 codes + 32 B of E4M3 scales            */

/* ---------------------------------------------------------------- codecs */

static float bf16_to_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* OCP FP8 E4M3 (e4m3fn): bias 7, 3 mantissa bits, subnormal step 2^-9,
 * largest finite 448, no infinities, S.1111.111 is NaN. */
double csa2o_e4m3_decode(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* subnormal: m * 2^-9 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Encode to E4M3 by round-to-nearest-even with saturation to +-448
 * ("satfinite"); the sign of a zero result is kept. */
uint8_t csa2o_e4m3_encode(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (isnan(x)) return 0x7F;
    if (a >= 448.0) return sign | 0x7E;
    /* grid spacing of the binade holding a */
    double step;
    if (a < ldexp(1.0, -6)) step = ldexp(1.0, -9);
    else {
        int e;
        frexp(a, &e);                    /* a = f * 2^e, f in [0.5, 1) */
        step = ldexp(1.0, (e - 1) - 3);  /* 3 mantissa bits below 2^(e-1) */
    }
    double r = rint(a / step);           /* ties to even (default rounding mode) */
    double v = r * step;
    if (v > 448.0) v = 448.0;
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9));
    int e;
    double f = frexp(v, &e);             /* v = f * 2^e, f in [0.5,1) -> 1.m * 2^(e-1) */
    int ee = (e - 1) + 7;
    int mm = (int)((f * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(ee << 3) | (uint8_t)mm;
}

/* E2M1 (OCP MX FP4): values 0, 0.5, 1, 1.5, 2, 3, 4, 6; code = S.EE.M */
double csa2o_e2m1_decode(uint8_t c) {
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[c & 7];
    return (c & 8) ? -v : v;
}

/* Round-to-nearest-even onto the E2M1 grid, saturating at +-6.  READING: a
 * nonzero value that rounds to zero keeps its sign (code 0x8 when negative). */
uint8_t csa2o_e2m1_encode(float x) {
    uint8_t sign = signbit(x) ? 8 : 0;
    double a = fabs((double)x);
    if (a >= 6.0) return sign | 7;
    double step = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double v = rint(a / step) * step;
    uint8_t code;
    if (v < 2.0) code = (uint8_t)(v * 2.0);          /* 0,0.5,1,1.5 -> 0..3; 2.0 -> 4 */
    else if (v < 4.0) code = (uint8_t)(2 + v);       /* 2 -> 4, 3 -> 5 */
    else code = (v < 6.0) ? 6 : 7;                   /* 4 -> 6, 6 -> 7 */
    return sign | code;
}

/* ------------------------------------------------------------------ RoPE */

/* RoPE on the tail 64 channels of a 512-d latent ("quantized after RoPE",
 * [A] 2.4.4; RoPE acts on the tail channels only, [A] 3.3.2).
 * parity unpinned -- READING: interleaved pairs (448+2i, 449+2i), i=0..31,
 * inverse frequency fl32(base^(-2i/64)), angle = pos * inv_freq (exact in
 * double), c,s = fl32(cos/sin(angle)), y0 = x0 c - x1 s, y1 = x0 s + x1 c, each
 * product and the sum rounded to fp32 separately (no fused multiply-add). */
void csa2o_rope_tail(const float *x, int64_t pos, double base, float *y) {
    for (int i = 0; i < O_D; ++i) y[i] = x[i];
    for (int i = 0; i < O_ROPE / 2; ++i) {
        float inv = (float)pow(base, -(2.0 * i) / (double)O_ROPE);
        double ang = (double)pos * (double)inv;
        float c = (float)cos(ang), s = (float)sin(ang);
        float x0 = x[O_D - O_ROPE + 2 * i], x1 = x[O_D - O_ROPE + 2 * i + 1];
        float p0 = x0 * c, p1 = x1 * s, p2 = x0 * s, p3 = x1 * c;
        y[O_D - O_ROPE + 2 * i] = p0 - p1;
        y[O_D - O_ROPE + 2 * i + 1] = p2 + p3;
    }
}

/* --------------------------------------------------------- compressor m=2 */

/* Gated pooling of m source positions into one entry with channel-wise
 * softmax weights over the positions ([A] 2.3.1/3.3.2: "gated pooling",
 * degenerating to a per-token projection at m=1).  parity unpinned --
 * READING: e[c] = sum_j softmax_j(Z[j][c]) * x[j][c], computed in double and
 * rounded once to fp32 (w_j = exp(Z_j - max_j Z) / sum). */
void csa2o_compress(const uint16_t *x, const uint16_t *z, int m, float *e) {
    for (int c = 0; c < O_D; ++c) {
        if (m == 1) { e[c] = bf16_to_f32(x[c]); continue; }
        double zmax = -INFINITY;
        for (int j = 0; j < m; ++j) {
            double zj = bf16_to_f32(z[j * O_D + c]);
            if (zj > zmax) zmax = zj;
        }
        double den = 0.0, num = 0.0;
        for (int j = 0; j < m; ++j) den += exp((double)bf16_to_f32(z[j * O_D + c]) - zmax);
        for (int j = 0; j < m; ++j) {
            double wj = exp((double)bf16_to_f32(z[j * O_D + c]) - zmax) / den;
            num += wj * (double)bf16_to_f32(x[j * O_D + c]);
        }
        e[c] = (float)num;
    }
}

/* ------------------------------------------------------------ FP4 entry */

/* FP4 main-KV format ([N] sec.4, [A] 2.4.4): E2M1 codes, one E4M3 scale per
 * 16 channels, no second-level global scale.  READING (NVFP4 convention the
 * pages point to): scale = E4M3_rne_satfinite(amax/6) with an fp32 divide;
 * code = E2M1_rne_satfinite(fl32(x / decoded_scale)); a zero scale gives
 * all-zero codes.  Layout: bytes 0..255 codes, channel 2j in the low nibble
 * of byte j, channel 2j+1 in the high nibble; bytes 256..287 the 32 scales. */
void csa2o_fp4_quantise(const float *x, uint8_t *entry) {
    memset(entry, 0, O_ENTRY);
    for (int g = 0; g < O_D / O_GROUP; ++g) {
        float amax = 0.0f;
        for (int i = 0; i < O_GROUP; ++i) {
            float a = fabsf(x[g * O_GROUP + i]);
            if (a > amax) amax = a;
        }
        float q = amax / 6.0f;
        uint8_t s = csa2o_e4m3_encode(q);
        float sd = (float)csa2o_e4m3_decode(s);
        entry[256 + g] = s;
        for (int i = 0; i < O_GROUP; ++i) {
            int ch = g * O_GROUP + i;
            uint8_t code = 0;
            if (sd != 0.0f) {
                float t = x[ch] / sd;
                code = csa2o_e2m1_encode(t);
            }
            entry[ch / 2] |= (uint8_t)((ch & 1) ? (code << 4) : code);
        }
    }
}

/* Dequantised latent: value = e2m1(code) * e4m3(scale), exact in double. */
void csa2o_fp4_dequant(const uint8_t *entry, double *out) {
    for (int ch = 0; ch < O_D; ++ch) {
        uint8_t code = (ch & 1) ? (entry[ch / 2] >> 4) : (entry[ch / 2] & 15);
        out[ch] = csa2o_e2m1_decode(code) * csa2o_e4m3_decode(entry[256 + ch / O_GROUP]);
    }
}

/* One main-KV entry as written by a Full layer: compress (m=2) or take the
 * latent (m=1), RoPE the tail, then quantise -- quantisation after RoPE. */
void csa2o_kv_entry(const uint16_t *latent, const uint16_t *z, int m, int64_t pos,
                    double rope_base, uint8_t *entry) {
    float e[O_D], r[O_D];
    csa2o_compress(latent, z, m, e);
    csa2o_rope_tail(e, pos, rope_base, r);
    csa2o_fp4_quantise(r, entry);
}

void csa2o_kv_entries(const uint16_t *latent, const uint16_t *z, int m, int64_t n,
                      const int64_t *pos, double rope_base, uint8_t *entries) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        csa2o_kv_entry(latent + i * m * O_D, z ? z + i * m * O_D : NULL, m, pos[i], rope_base,
                       entries + i * O_ENTRY);
}

/* A real number rounded to the nearest bf16 (ties to even), as its bits:
 * 8 significant bits, quantum 2^-133 below the normal range, overflow to inf. */
static uint16_t f64_to_bf16_rne(double v) {
    if (v != v) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int e;
    frexp(fabs(v), &e);                     /* |v| in [2^(e-1), 2^e) */
    int qexp = e - 8;
    if (qexp < -133) qexp = -133;
    double r = ldexp(rint(ldexp(fabs(v), -qexp)), qexp);
    float rf = r > 3.3895313892515355e38 ? INFINITY : (float)r;   /* exact when finite */
    if (signbit(v)) rf = -rf;
    uint32_t u;
    memcpy(&u, &rf, 4);
    return (uint16_t)(u >> 16);
}

/* The Full layer's indexer key of an entry ("DeepSeek-v4.1 Flash: Pushing
 * the Limits of KV Cache Compression", section 2.3.1: CSA2 obtains the Indexer
 * K by projecting the main KV entry).  READING: the projected entry is the
 * main-KV entry as written, before its FP4 quantisation (compressed at m = 2,
 * RoPE on the tail channels, fp32); k = W e with W bf16 [128][512], in fp64,
 * rounded once to bf16. */
void csa2o_indexer_k_project(const uint16_t *latent, const uint16_t *z, int m, int64_t n, const int64_t *pos,
                             double rope_base, const uint16_t *w, uint16_t *k) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float e[O_D], r[O_D];
        csa2o_compress(latent + i * m * O_D, z ? z + i * m * O_D : NULL, m, e);
        csa2o_rope_tail(e, pos[i], rope_base, r);
        for (int o = 0; o < O_DI; ++o) {
            double acc = 0.0;
            for (int c = 0; c < O_D; ++c) acc += (double)bf16_to_f32(w[o * O_D + c]) * (double)r[c];
            k[i * O_DI + o] = f64_to_bf16_rne(acc);
        }
    }
}

/* -------------------------------------------------------------- indexer */

/* Lightning-indexer score of each key row: s_n = sum_h w_h * ReLU(q_h . k_n)
 * over 32 heads x 128 dims ([N] sec.2 main attention settings; the score form
 * is the plain weighted ReLU sum of head dot products, no extra scale).  fp64. */
void csa2o_index_scores(const uint16_t *q, const float *w, const uint16_t *k, int64_t n,
                        double *s) {
    double qd[O_HI * O_DI];
    for (int i = 0; i < O_HI * O_DI; ++i) qd[i] = bf16_to_f32(q[i]);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        double kd[O_DI];
        for (int d = 0; d < O_DI; ++d) kd[d] = bf16_to_f32(k[r * O_DI + d]);
        double acc = 0.0;
        for (int h = 0; h < O_HI; ++h) {
            double dot = 0.0;
            for (int d = 0; d < O_DI; ++d) dot += qd[h * O_DI + d] * kd[d];
            acc += (double)w[h] * (dot > 0.0 ? dot : 0.0);
        }
        s[r] = acc;
    }
}

/* --------------------------------------------------- MXFP4 indexer cache */

/* MXFP4 (OCP Microscaling v1.0): a block of 32 elements shares one UE8M0
 * scale 2^E; elements are E2M1.  The indexer Q and K are FP4 ([A] 2.4.4: QAT
 * "for the FP4 Indexer Q and K"; [A] 3.1: a 128-dimensional MXFP4 indexer-K
 * entry is 68 B = 64 B of codes + 4 scale bytes).
 * READING (the OCP conversion rule): E = floor(log2(max |x|)) - 2 (2 = the
 * largest E2M1 exponent), clamped to [-127, 127]; an all-zero block takes
 * E = -127; code_i = E2M1_RNE_satfinite(x_i / 2^E) (the quotient is exact).
 * Scale byte = E + 127.  READING (layout): element 2j in the low nibble of
 * code byte j; the 4 scale bytes cover dims 0-31, 32-63, 64-95, 96-127. */
void csa2o_mxfp4_quantise(const float *x, uint8_t *codes, uint8_t *scales) {
    for (int b = 0; b < O_DI / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double a = fabs((double)x[b * 32 + i]);
            if (a > amax) amax = a;
        }
        int E = -127;
        if (amax > 0.0) {
            int e;
            frexp(amax, &e);          /* amax = f 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
            E = e - 1 - 2;
            if (E < -127) E = -127;
            if (E > 127) E = 127;
        }
        scales[b] = (uint8_t)(E + 127);
        for (int i = 0; i < 32; i += 2) {
            uint8_t lo = csa2o_e2m1_encode((float)ldexp((double)x[b * 32 + i], -E));
            uint8_t hi = csa2o_e2m1_encode((float)ldexp((double)x[b * 32 + i + 1], -E));
            codes[(b * 32 + i) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* Rows of bf16 -> MXFP4 (codes [n][64], scales [n][4]). */
void csa2o_mxfp4_quantise_rows(const uint16_t *x, int64_t n, uint8_t *codes, uint8_t *scales) {
    for (int64_t r = 0; r < n; ++r) {
        float xf[O_DI];
        for (int d = 0; d < O_DI; ++d) xf[d] = bf16_to_f32(x[r * O_DI + d]);
        csa2o_mxfp4_quantise(xf, codes + r * (O_DI / 2), scales + r * (O_DI / 32));
    }
}

/* code x 2^E, exact in double */
void csa2o_mxfp4_dequant(const uint8_t *codes, const uint8_t *scales, double *out) {
    for (int d = 0; d < O_DI; ++d) {
        uint8_t c = (uint8_t)((codes[d / 2] >> (4 * (d & 1))) & 15);
        out[d] = ldexp(csa2o_e2m1_decode(c), (int)scales[d / 32] - 127);
    }
}

/* The indexer score with FP4 operands: the query rows (bf16) are quantised
 * to MXFP4 like the keys; s_n = sum_h w_h ReLU(dq(q_h) . dq(k_n)) in fp64. */
void csa2o_index_scores_mxfp4(const uint16_t *q, const float *w, const uint8_t *k_codes,
                              const uint8_t *k_scales, int64_t n, double *s) {
    double qd[O_HI * O_DI];
    for (int h = 0; h < O_HI; ++h) {
        uint8_t qc[O_DI / 2], qs[O_DI / 32];
        csa2o_mxfp4_quantise_rows(q + h * O_DI, 1, qc, qs);
        csa2o_mxfp4_dequant(qc, qs, qd + h * O_DI);
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        double kd[O_DI];
        csa2o_mxfp4_dequant(k_codes + r * (O_DI / 2), k_scales + r * (O_DI / 32), kd);
        double acc = 0.0;
        for (int h = 0; h < O_HI; ++h) {
            double dot = 0.0;
            for (int d = 0; d < O_DI; ++d) dot += qd[h * O_DI + d] * kd[d];
            acc += (double)w[h] * (dot > 0.0 ? dot : 0.0);
        }
        s[r] = acc;
    }
}

/* ---------------------------------------------------------------- top-K */

typedef struct { double s; int64_t i; } scored;

static int by_score_desc_index_asc(const void *a, const void *b) {
    const scored *x = (const scored *)a, *y = (const scored *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

static int by_index_asc(const void *a, const void *b) {
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x < y) ? -1 : (x > y);
}

/* The k highest scores (ties toward the lower index), by a full sort.
 * READING: output ascending by index, -1 padding when fewer than k.
 * Entries whose valid flag is 0 (or all, when valid == NULL) are candidates
 * only if valid.  Returns the number selected. */
int64_t csa2o_topk(const double *s, const uint8_t *valid, int64_t n, int64_t k, int64_t *out) {
    scored *v = (scored *)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i)
        if (!valid || valid[i]) { v[m].s = s[i]; v[m].i = i; ++m; }
    qsort(v, (size_t)m, sizeof(scored), by_score_desc_index_asc);
    int64_t take = m < k ? m : k;
    for (int64_t j = 0; j < take; ++j) out[j] = v[j].i;
    qsort(out, (size_t)take, sizeof(int64_t), by_index_asc);
    for (int64_t j = take; j < k; ++j) out[j] = -1;
    free(v);
    return take;
}

/* ------------------------------------------------------------------ HSI */

/* Block scores of the HSI ([A] 2.3.4): pad the score row with -inf up to a
 * multiple of the block width, view it as [n_blocks, block], reduce each row
 * (max per the pages; READING: "sum" adds the valid positions, padding
 * contributes nothing). */
void csa2o_block_scores(const double *s, int64_t n_vis, int bs, int reduce_sum, double *out) {
    int64_t nb = (n_vis + bs - 1) / bs;
    for (int64_t b = 0; b < nb; ++b) {
        double acc = reduce_sum ? 0.0 : -INFINITY;
        for (int i = 0; i < bs; ++i) {
            int64_t p = b * bs + i;
            double v = (p < n_vis) ? s[p] : -INFINITY;       /* the -inf padding */
            if (reduce_sum) { if (p < n_vis) acc += v; }
            else if (v > acc) acc = v;
        }
        out[b] = acc;
    }
}

/* HSI candidate pool ([A] 2.3.4, [N] sec.3): block scores as above, the block
 * holding the latest visible position forced into the selection (READING:
 * its score set to +inf), the top candidate_topk_blocks blocks by (score desc,
 * block asc).  Output: selected block ids ascending, -1 padded; returns how
 * many.  The pool is those blocks' positions truncated to [0, n_vis). */
int64_t csa2o_hsi_pool(const double *s, int64_t n_vis, int bs, int64_t n_pool_blocks,
                       int reduce_sum, int64_t *blocks_out) {
    int64_t nb = (n_vis + bs - 1) / bs;
    double *b = (double *)malloc(sizeof(double) * (size_t)(nb > 0 ? nb : 1));
    csa2o_block_scores(s, n_vis, bs, reduce_sum, b);
    if (nb > 0) b[(n_vis - 1) / bs] = INFINITY;
    int64_t r = csa2o_topk(b, NULL, nb, n_pool_blocks, blocks_out);
    free(b);
    return r;
}

/* ------------------------------------------------------------ attention */

/* Sparse-attention readout of one query token ([A] 3.3.1-3.3.2, [N] sec.2):
 * one softmax over the selected main-KV entries together with the local SWA
 * entries; key = value = the dequantised 512-d latent (RoPE channels
 * included); logits q_h . k_j / sqrt(512); output the convex combination.
 * READING: no sink, no bias; idx < 0 entries are skipped; SWA rows are E4M3
 * codes times a per-row fp32 scale.  fp64 throughout.
 * out[64][512]; lse[64] = log sum_j exp(logit) (natural log, -inf if no key);
 * weights (optional) [64][k + W] in input order, 0 for skipped slots. */
void csa2o_sparse_attn(const uint16_t *q, const uint8_t *kv, const int64_t *idx, int64_t k,
                       const uint8_t *swa, const float *swa_scale, int64_t swa_len,
                       double *out, double *lse, double *weights) {
    int64_t nk = k + swa_len;
    double *keys = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * O_D);
    uint8_t *ok = (uint8_t *)calloc((size_t)(nk > 0 ? nk : 1), 1);
    for (int64_t j = 0; j < k; ++j) {
        if (idx[j] < 0) continue;
        csa2o_fp4_dequant(kv + idx[j] * O_ENTRY, keys + j * O_D);
        ok[j] = 1;
    }
    for (int64_t t = 0; t < swa_len; ++t) {
        for (int c = 0; c < O_D; ++c)
            keys[(k + t) * O_D + c] = csa2o_e4m3_decode(swa[t * O_D + c]) * (double)swa_scale[t];
        ok[k + t] = 1;
    }
    const double scale = 1.0 / sqrt((double)O_D);
#pragma omp parallel for schedule(static)
    for (int h = 0; h < O_H; ++h) {
        double qh[O_D];
        for (int c = 0; c < O_D; ++c) qh[c] = bf16_to_f32(q[h * O_D + c]);
        double *lg = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        double mx = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
            if (!ok[j]) continue;
            double dot = 0.0;
            for (int c = 0; c < O_D; ++c) dot += qh[c] * keys[j * O_D + c];
            lg[j] = dot * scale;
            if (lg[j] > mx) mx = lg[j];
        }
        double z = 0.0;
        for (int64_t j = 0; j < nk; ++j) if (ok[j]) z += exp(lg[j] - mx);
        for (int c = 0; c < O_D; ++c) out[h * O_D + c] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            double p = ok[j] ? exp(lg[j] - mx) / z : 0.0;
            if (weights) weights[h * nk + j] = p;
            if (!ok[j]) continue;
            for (int c = 0; c < O_D; ++c) out[h * O_D + c] += p * keys[j * O_D + c];
        }
        if (lse) lse[h] = (z > 0.0) ? mx + log(z) : -INFINITY;
        free(lg);
    }
    free(keys);
    free(ok);
}

int csa2o_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
