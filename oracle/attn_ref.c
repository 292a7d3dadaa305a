/*
 * attn_ref.c -- fp64 CPU oracle for the exact attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * with the CUDA library; the two meet only in the seeded inputs they are given.
 *
 * What it computes (the plain definition, no tiling, no online rescale):
 *   for every batch b, query head h and query row i, with kv head h / (Hq/Hkv),
 *     s_j  = scale * sum_d q[i,d] k[j,d]            for the allowed keys j
 *     m    = max_j s_j
 *     l    = sum_j exp(s_j - m)
 *     P_j  = exp(s_j - m) / l
 *     O[i] = sum_j P_j v[j]
 *     LSE  = m + ln l                                 (natural log, scale included)
 *   Softmax attention is the normaliser whose log-sum-exp has a closed form
 *   (page "AdaSplash-2: Faster Differentiable Sparse Attention", technical
 *   summary section 1, problem statement); the fused FlashAttention-style
 *   kernel (same section) reaches this same result up to rounding order.
 *   The kernels the article "L'agent a questions depasse l'agent a outils :
 *   113% contre 50% de la vitesse de FlashAttention-3" reports (section
 *   "Ce que cela a donne") are attention *forward* kernels checked against an
 *   fp32 reference (section "Comment une question change la tache"); this
 *   oracle plays that reference's role, in fp64.
 *
 * Readings where the pages say nothing (each listed in the design notes):
 *   - layout: q,o [B][Hq][Sq][D]; k,v [B][Hkv][Sk][D]; lse [B][Hq][Sq]; contiguous.
 *   - GQA: query head h reads kv head h / (Hq/Hkv) (contiguous groups).
 *   - causal = 0: every key allowed; 1: bottom-right aligned, key j allowed for
 *     row i iff j <= i + (Sk - Sq); 2: top-left aligned, j <= i.
 *   - a row with no allowed key has O = 0 and LSE = -inf.
 *   - inputs arrive as raw bf16 bit patterns and are widened exactly; scale is
 *     the fp32 value the GPU receives, widened exactly to fp64.
 *   - block mask (attn_ref_fwd_masked): the keys a row may attend to are further
 *     restricted to the key blocks its query block's bit-packed mask row marks
 *     (page "AdaSplash-2: Faster Differentiable Sparse Attention", technical
 *     summary section 2, bit-packed block masking: one bit per (query block,
 *     key block), 32 blocks per 32-bit word).  Layout
 *     mask[b][hm][i / block_q][w], hm = 0 when one mask serves every head else
 *     h; bit (kb % 32) of word kb / 32 marks key block kb = j / block_k.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC attn_ref.c -o libattn_ref.so -lm
 * Portable C99: no intrinsics, no architecture flags (runs on x86_64 and aarch64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
static double bf16_bits_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of keys row i may attend to (keys 0 .. n-1), per the causal reading above. */
static int64_t allowed_keys(int64_t i, int64_t Sq, int64_t Sk, int causal) {
    int64_t last;
    if (causal == 0) return Sk;
    last = (causal == 1) ? (i + Sk - Sq) : i;
    if (last >= Sk) last = Sk - 1;
    return last < 0 ? 0 : last + 1;
}

/* Whether key j passes the row's block-mask words (NULL: no block mask). */
static int block_visible(const uint32_t* mask_row, int64_t j, int block_k) {
    int64_t kb;
    if (!mask_row) return 1;
    kb = j / block_k;
    return (int)((mask_row[kb / 32] >> (kb % 32)) & 1u);
}

/*
 * One query row.  s (scratch) and p (optional output) hold at least Sk doubles.
 * q_row: D bf16; kh, vh: the kv head's [Sk][D] bf16; mask_row: the row's block-mask
 * words or NULL.  Writes o_row[D] and *lse.
 */
static void ref_row(const uint16_t* q_row, const uint16_t* kh, const uint16_t* vh,
                    int64_t i, int64_t Sq, int64_t Sk, int64_t D, int causal, double scale,
                    const uint32_t* mask_row, int block_k,
                    double* s, double* p, double* o_row, double* lse) {
    int64_t n = allowed_keys(i, Sq, Sk, causal);
    int64_t j, d, seen = 0;
    double m = -INFINITY, l;

    for (d = 0; d < D; ++d) o_row[d] = 0.0;
    if (p) for (j = 0; j < Sk; ++j) p[j] = 0.0;
    /* logits of the allowed keys, and their maximum */
    for (j = 0; j < n; ++j) {
        double acc = 0.0;
        if (!block_visible(mask_row, j, block_k)) continue;
        for (d = 0; d < D; ++d)
            acc += bf16_bits_to_f64(q_row[d]) * bf16_bits_to_f64(kh[j * D + d]);
        s[j] = scale * acc;
        if (seen == 0 || s[j] > m) m = s[j];
        ++seen;
    }
    if (seen == 0) {
        *lse = -INFINITY;
        return;
    }
    /* normaliser */
    l = 0.0;
    for (j = 0; j < n; ++j)
        if (block_visible(mask_row, j, block_k)) l += exp(s[j] - m);
    /* probabilities, then the weighted sum of value rows */
    for (j = 0; j < n; ++j) {
        double pj;
        if (!block_visible(mask_row, j, block_k)) continue;
        pj = exp(s[j] - m) / l;
        if (p) p[j] = pj;
        for (d = 0; d < D; ++d) o_row[d] += pj * bf16_bits_to_f64(vh[j * D + d]);
    }
    *lse = m + log(l);
}

static int check_args(int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return 1;
    if (Hq % Hkv != 0) return 1;
    if (causal < 0 || causal > 2) return 1;
    return 0;
}

static int fwd_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o, double* lse,
                    int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                    const uint32_t* mask, int mask_heads, int block_q, int block_k,
                    const int64_t* rows, int64_t nrows) {
    const int64_t G = (Hkv > 0) ? (int64_t)Hq / Hkv : 1;
    const int64_t total = (int64_t)B * Hq * Sq;
    const int64_t count = rows ? nrows : total;
    const double scale64 = (double)scale;
    const int64_t qblocks = (mask && block_q > 0) ? ((int64_t)Sq + block_q - 1) / block_q : 0;
    const int64_t words = (mask && block_k > 0) ? (((int64_t)Sk + block_k - 1) / block_k + 31) / 32 : 0;
    int failed = 0;
    int64_t t;

    if (check_args(B, Hq, Hkv, Sq, Sk, D, causal)) return 1;
    if (mask && (block_q <= 0 || block_k <= 0 || (mask_heads != 1 && mask_heads != Hq))) return 1;
    if (rows) {
        for (t = 0; t < nrows; ++t)
            if (rows[t] < 0 || rows[t] >= total) return 1;
    }

#pragma omp parallel for schedule(dynamic, 8) reduction(| : failed)
    for (t = 0; t < count; ++t) {
        const int64_t r = rows ? rows[t] : t;
        const int64_t i = r % Sq;
        const int64_t bh = r / Sq;
        const int64_t b = bh / Hq, h = bh % Hq;
        const int64_t kvh = h / G;
        const uint16_t* kh = k + ((b * Hkv + kvh) * (int64_t)Sk) * D;
        const uint16_t* vh = v + ((b * Hkv + kvh) * (int64_t)Sk) * D;
        const uint32_t* mrow = NULL;
        double* s;
        if (mask) {
            const int64_t hm = (mask_heads == 1) ? 0 : h;
            mrow = mask + ((b * mask_heads + hm) * qblocks + i / block_q) * words;
        }
        s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        if (!s) { failed |= 1; continue; }
        ref_row(q + r * D, kh, vh, i, Sq, Sk, D, causal, scale64, mrow, block_k, s, NULL,
                o + t * D, lse + t);
        free(s);
    }
    return failed ? 2 : 0;
}

/*
 * Full or row-subset forward.
 *   rows == NULL: every row; o is [B][Hq][Sq][D], lse is [B][Hq][Sq].
 *   rows != NULL: nrows flat row ids r = (b*Hq + h)*Sq + i; o is [nrows][D],
 *                 lse is [nrows] (compact, in the order given).
 * Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 */
int attn_ref_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                 double* o, double* lse,
                 int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                 const int64_t* rows, int64_t nrows) {
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, NULL, 1, 1, 1, rows, nrows);
}

/*
 * The same with a bit-packed block mask (layout in the header comment; blocks of
 * block_q query rows by block_k keys; mask_heads 1 or Hq).  A row whose allowed
 * keys all fall in unmarked blocks has O = 0 and LSE = -inf.
 */
int attn_ref_fwd_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        double* o, double* lse,
                        int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                        const uint32_t* mask, int mask_heads, int block_q, int block_k,
                        const int64_t* rows, int64_t nrows) {
    if (!mask) return 1;
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mask, mask_heads, block_q, block_k,
                    rows, nrows);
}

/*
 * Probability matrix of one (b, h) slice, for pinning the oracle on tiny shapes:
 * p is [Sq][Sk] (zeros for masked keys), o is [Sq][D], lse is [Sq].  Same row
 * routine as attn_ref_fwd, so the pins see the code path the comparisons use.
 */
int attn_ref_probs(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   double* p, double* o, double* lse,
                   int Sq, int Sk, int D, int causal, float scale) {
    int64_t i;
    double* s;
    if (check_args(1, 1, 1, Sq, Sk, D, causal)) return 1;
    s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
    if (!s) return 2;
    for (i = 0; i < Sq; ++i)
        ref_row(q + i * D, k, v, i, Sq, Sk, D, causal, (double)scale, NULL, 1, s,
                p + i * (int64_t)Sk, o + i * D, lse + i);
    free(s);
    return 0;
}

/* Threads the oracle's parallel loop uses (reported beside its timings). */
int attn_ref_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Backward of the forward above with respect to its output O (the gradient a
 * training step carries; no gradient flows in through the LSE).  With the
 * forward's probabilities P_ij (softmax over the allowed keys of row i) and the
 * upstream gradient dO_i, by the chain rule through O_i = sum_j P_ij v_j and the
 * softmax Jacobian dP_ij/ds_ik = P_ij (delta_jk - P_ik):
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = dO_i . v_j
 *     D_i   = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij k_j
 *     dK_j  = scale * sum_i dS_ij q_i
 * where the sums over i run over every query head that reads the kv head.
 * Inputs are bf16 bit patterns (dout like q); dq is [B][Hq][Sq][D], dk and dv
 * [B][Hkv][Sk][D], all fp64.  Parallel over (batch, kv head), each of which owns
 * its dk and dv rows.  Returns 0, 1 on bad arguments, 2 on allocation failure.
 */
int attn_ref_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                 double* dq, double* dk, double* dv,
                 int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale) {
    const int64_t G = (Hkv > 0) ? (int64_t)Hq / Hkv : 1;
    const double scale64 = (double)scale;
    int failed = 0;
    int64_t bk;

    if (check_args(B, Hq, Hkv, Sq, Sk, D, causal)) return 1;
    memset(dq, 0, sizeof(double) * (size_t)B * Hq * Sq * D);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Sk * D);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Sk * D);

#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (bk = 0; bk < (int64_t)B * Hkv; ++bk) {
        const int64_t b = bk / Hkv, kvh = bk % Hkv;
        const uint16_t* kh = k + bk * (int64_t)Sk * D;
        const uint16_t* vh = v + bk * (int64_t)Sk * D;
        double* dkh = dk + bk * (int64_t)Sk * D;
        double* dvh = dv + bk * (int64_t)Sk * D;
        double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        double* p = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        double* orow = (double*)malloc(sizeof(double) * (size_t)(D > 0 ? D : 1));
        int64_t g, i, j, d;
        if (!s || !p || !orow) {
            failed |= 1;
            free(s); free(p); free(orow);
            continue;
        }
        for (g = 0; g < G; ++g) {
            const int64_t h = kvh * G + g;
            for (i = 0; i < Sq; ++i) {
                const int64_t r = (b * Hq + h) * (int64_t)Sq + i;
                const uint16_t* qrow = q + r * D;
                const uint16_t* dorow = dout + r * D;
                const int64_t n = allowed_keys(i, Sq, Sk, causal);
                double lse, Di = 0.0;
                /* the forward's probabilities of this row (p is zero past the allowed keys) */
                ref_row(qrow, kh, vh, i, Sq, Sk, D, causal, scale64, NULL, 1, s, p, orow, &lse);
                if (n == 0) continue;
                for (j = 0; j < n; ++j) {
                    double dp = 0.0;
                    for (d = 0; d < D; ++d) dp += bf16_bits_to_f64(dorow[d]) * bf16_bits_to_f64(vh[j * D + d]);
                    s[j] = dp;  /* reuse: dP_ij */
                    Di += p[j] * dp;
                }
                for (j = 0; j < n; ++j) {
                    const double ds = p[j] * (s[j] - Di);
                    for (d = 0; d < D; ++d) {
                        dq[r * D + d] += scale64 * ds * bf16_bits_to_f64(kh[j * D + d]);
                        dkh[j * D + d] += scale64 * ds * bf16_bits_to_f64(qrow[d]);
                        dvh[j * D + d] += p[j] * bf16_bits_to_f64(dorow[d]);
                    }
                }
            }
        }
        free(s); free(p); free(orow);
    }
    return failed ? 2 : 0;
}
