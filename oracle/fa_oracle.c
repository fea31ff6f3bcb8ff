/*
 * fa_oracle.c -- plain float64 CPU oracle for exact attention and Flash-Decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only in the seeded input tensors.
 *
 * What it computes, and where each step comes from:
 *
 *  - "Infra: Flash Attention" (pufanyi.com), section "Attention and its scope":
 *    S = Q K^T / sqrt(d), P = row-softmax(S), O = P V, one head at a time.
 *  - same page, "Stable normalisation": the row softmax subtracts the row
 *    maximum m and divides by l = sum_j exp(S_ij - m).
 *  - same page, "Backward and recomputation": the per-row log-sum-exp
 *    L_i = m_i + log l_i = log sum_j exp(S_ij).
 *  - same page, "Symbols and boundary conditions" and the causal figure:
 *    under causal masking query i sees keys j <= i; a query row with no valid
 *    key is left to the operator (reading used here: O = 0, L = -inf).
 *  - same page, "Merging block states" and "Accumulating the weighted sum":
 *    the (m, l) and (m, l, u) merge with alpha = exp(m_A - m), beta = exp(m_B - m).
 *  - "science-depth M4-055" (airsota.com), "Flash-Decoding Algorithm", step 3:
 *    the log-sum-exp reduction of per-chunk partials (m_k, l_k, O_k).
 *  - same page, "Backward and recomputation" and "Blocked gradient computation":
 *    P_ij = exp(S_ij - L_i); dV = P^T dO; dP = dO V^T; dS_ij = P_ij (dP_ij - D_i)
 *    with D_i = sum_j P_ij dP_ij; dQ = scale dS K; dK = scale dS^T Q.
 *    CMU 10-423 Lecture 18 notes, section 5.3: the same gradients, with the
 *    identity D_i = dO_i . O_i (checked by the tests, not used here).
 *  - CMU 10-423 Lecture 18 notes (semidirectx.com), section 2.1: naive, safe
 *    and online softmax; section 2.2 and Exercise 1: the online recurrence
 *    d_j = d_{j-1} exp(m_{j-1} - m_j) + exp(x_j - m_j).
 *
 * FP8 inputs (the e4m3 variant of the forward) are decoded exactly by
 * oracle_e4m3_to_f64, written from the OCP 8-bit floating-point format
 * definition (E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals at exponent 0, no infinities, S.1111.111 = NaN); the
 * attention itself then runs through oracle_sdpa_forward_f64.
 *
 * Everything is float64.  Inputs arrive as bfloat16 bit patterns (the same
 * bits the GPU receives) and are widened exactly: a bfloat16 value is the top
 * 16 bits of an IEEE-754 binary32 value.
 *
 * The forward oracle is the plain definition, one query row at a time: it
 * materialises that row of S, takes the stable softmax to get that row of P,
 * and forms O_i = sum_j P_ij V_j.  It does not tile, fuse or reorder anything.
 * The decode oracle is the same definition with one query and does NOT split
 * the key range; the split/merge identity is checked separately.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bfloat16 -> float64: place the 16 bits on top of a binary32 word. */
static double widen_bf16(uint16_t bits)
{
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------------
 * Softmax forms of Lecture 18, section 2.1 (used by the oracle's own pins).
 * ------------------------------------------------------------------------- */

/* naive softmax: y_j = exp(x_j) / sum_k exp(x_k) (overflows for large x) */
void oracle_softmax_naive(const double *x, int n, double *y)
{
    double den = 0.0;
    for (int k = 0; k < n; ++k) den += exp(x[k]);
    for (int j = 0; j < n; ++j) y[j] = exp(x[j]) / den;
}

/* safe softmax: subtract the maximum first ("Stable normalisation") */
void oracle_softmax_safe(const double *x, int n, double *y)
{
    double m = -INFINITY;
    for (int k = 0; k < n; ++k) m = x[k] > m ? x[k] : m;
    double l = 0.0;
    for (int k = 0; k < n; ++k) l += exp(x[k] - m);
    for (int j = 0; j < n; ++j) y[j] = exp(x[j] - m) / l;
}

/* online softmax, one element at a time (Lecture 18 section 2.2, Exercise 1):
 *   m_j = max(m_{j-1}, x_j)
 *   d_j = d_{j-1} * exp(m_{j-1} - m_j) + exp(x_j - m_j)
 * m_trace[j], d_trace[j] receive the running values after reading x_j. */
void oracle_online_softmax_trace(const double *x, int n, double *m_trace, double *d_trace)
{
    double m = -INFINITY, dsum = 0.0;
    for (int j = 0; j < n; ++j) {
        double m_new = x[j] > m ? x[j] : m;
        double corr = (j == 0) ? 0.0 : exp(m - m_new);
        dsum = dsum * corr + exp(x[j] - m_new);
        m = m_new;
        m_trace[j] = m;
        d_trace[j] = dsum;
    }
}

/* ---------------------------------------------------------------------------
 * Block state (m, l, u) of "Merging block states" / "Accumulating the
 * weighted sum":  m = max_j x_j,  l = sum_j exp(x_j - m),
 *                 u = sum_j exp(x_j - m) V_j     (V_j has dv components).
 * ------------------------------------------------------------------------- */
void oracle_block_state(const double *x, const double *V, int n, int dv,
                        double *m_out, double *l_out, double *u_out)
{
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) m = x[j] > m ? x[j] : m;
    double l = 0.0;
    for (int c = 0; c < dv; ++c) u_out[c] = 0.0;
    if (n > 0) {
        for (int j = 0; j < n; ++j) {
            double w = exp(x[j] - m);
            l += w;
            for (int c = 0; c < dv; ++c) u_out[c] += w * V[(size_t)j * dv + c];
        }
    }
    *m_out = m;
    *l_out = l;
}

/* merge of two block states:
 *   m = max(m_A, m_B), alpha = exp(m_A - m), beta = exp(m_B - m),
 *   l = alpha l_A + beta l_B,  u = alpha u_A + beta u_B.
 * An empty state (m = -inf, l = 0) contributes nothing. */
void oracle_state_merge(double m_a, double l_a, const double *u_a,
                        double m_b, double l_b, const double *u_b, int dv,
                        double *m_out, double *l_out, double *u_out)
{
    double m = m_a > m_b ? m_a : m_b;
    if (m == -INFINITY) {           /* both empty */
        *m_out = m;
        *l_out = 0.0;
        for (int c = 0; c < dv; ++c) u_out[c] = 0.0;
        return;
    }
    double alpha = (m_a == -INFINITY) ? 0.0 : exp(m_a - m);
    double beta = (m_b == -INFINITY) ? 0.0 : exp(m_b - m);
    *m_out = m;
    *l_out = alpha * l_a + beta * l_b;
    for (int c = 0; c < dv; ++c) u_out[c] = alpha * u_a[c] + beta * u_b[c];
}

/* Flash-Decoding log-sum-exp reduction ("science-depth M4-055", step 3):
 *   m_f = max_k m_k,   l_f = sum_k l_k exp(m_k - m_f),
 *   O_f = sum_k O_k * (l_k exp(m_k - m_f) / l_f),
 * with O_k the chunk outputs already divided by their own l_k.  Chunks with
 * l_k = 0 (no keys) are skipped.  Returns L_f = m_f + log l_f in *lse_out. */
void oracle_lse_reduce(const double *m_k, const double *l_k, const double *O_k,
                       int nchunks, int dv, double *O_out, double *lse_out)
{
    double m_f = -INFINITY;
    for (int k = 0; k < nchunks; ++k)
        if (l_k[k] > 0.0 && m_k[k] > m_f) m_f = m_k[k];
    for (int c = 0; c < dv; ++c) O_out[c] = 0.0;
    if (m_f == -INFINITY) {
        *lse_out = -INFINITY;
        return;
    }
    double l_f = 0.0;
    for (int k = 0; k < nchunks; ++k)
        if (l_k[k] > 0.0) l_f += l_k[k] * exp(m_k[k] - m_f);
    for (int k = 0; k < nchunks; ++k) {
        if (!(l_k[k] > 0.0)) continue;
        double w = l_k[k] * exp(m_k[k] - m_f) / l_f;
        for (int c = 0; c < dv; ++c) O_out[c] += O_k[(size_t)k * dv + c] * w;
    }
    *lse_out = m_f + log(l_f);
}

/* ---------------------------------------------------------------------------
 * Attention of one query over an explicit score vector: the stable softmax
 * P_j = exp(x_j - m) / l, then O = sum_j P_j V_j and L = m + log l.
 * n == 0 (no valid key) gives O = 0 and L = -inf.
 * ------------------------------------------------------------------------- */
void oracle_attend_scores(const double *x, const double *V, int n, int dv,
                          double *O_out, double *lse_out)
{
    for (int c = 0; c < dv; ++c) O_out[c] = 0.0;
    if (n <= 0) {
        *lse_out = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) m = x[j] > m ? x[j] : m;
    double l = 0.0;
    for (int j = 0; j < n; ++j) l += exp(x[j] - m);
    for (int j = 0; j < n; ++j) {
        double p = exp(x[j] - m) / l;
        for (int c = 0; c < dv; ++c) O_out[c] += p * V[(size_t)j * dv + c];
    }
    *lse_out = m + log(l);
}

/* ---------------------------------------------------------------------------
 * Exact scaled-dot-product attention, selected query rows.
 *
 * Q: bf16 bits [B, H, Nq, d];  K, V: bf16 bits [B, H, Nk, d]  (row-major).
 * A row is the flat index r = (b * H + h) * Nq + i.  For that row the valid
 * keys are j < key_len[b] (all Nk when key_len is NULL), and, when causal,
 * j <= i (query i and key i are the same position; causal needs Nq == Nk).
 * For each requested row the function forms the explicit score row
 * S_ij = scale * sum_c Q_ic K_jc over the valid keys, its stable softmax,
 * O_i = sum_j P_ij V_j and L_i = m_i + log l_i.
 *
 * O_out is [nrows, d] float64, lse_out is [nrows]; rows == NULL means every
 * row in order (nrows must then be B*H*Nq).  Returns 0, or -1 on bad sizes.
 * ------------------------------------------------------------------------- */
int oracle_sdpa_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     int B, int H, int Nq, int Nk, int d, int causal, double scale,
                     const int32_t *key_len, const int64_t *rows, int64_t nrows,
                     double *O_out, double *lse_out, int nthreads)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0 || nrows < 0) return -1;
    if (causal && Nq != Nk) return -1;
    if (!rows && nrows != (int64_t)B * H * Nq) return -1;
    if (nthreads <= 0) nthreads = 1;
    int bad = 0;

#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *vrows = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1) * (size_t)d);
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !vrows || !q) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t t = 0; t < nrows; ++t) {
            if (!s || !vrows || !q) continue;
            int64_t r = rows ? rows[t] : t;
            if (r < 0 || r >= (int64_t)B * H * Nq) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                bad = 1;
                continue;
            }
            int64_t bh = r / Nq;
            int i = (int)(r % Nq);
            int b = (int)(bh / H);
            int nvalid = Nk;
            if (key_len) nvalid = key_len[b] < nvalid ? key_len[b] : nvalid;
            if (causal && i + 1 < nvalid) nvalid = i + 1;
            if (nvalid < 0) nvalid = 0;

            const uint16_t *qrow = Q + (size_t)r * d;
            const uint16_t *kbase = K + (size_t)bh * Nk * d;
            const uint16_t *vbase = V + (size_t)bh * Nk * d;
            for (int c = 0; c < d; ++c) q[c] = widen_bf16(qrow[c]);
            /* S row: scale * (q . k_j) */
            for (int j = 0; j < nvalid; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += q[c] * widen_bf16(kbase[(size_t)j * d + c]);
                s[j] = scale * acc;
            }
            for (int j = 0; j < nvalid; ++j)
                for (int c = 0; c < d; ++c)
                    vrows[(size_t)j * d + c] = widen_bf16(vbase[(size_t)j * d + c]);
            oracle_attend_scores(s, vrows, nvalid, d, O_out + (size_t)t * d, lse_out + t);
        }
        free(s);
        free(vrows);
        free(q);
    }
    return bad ? -1 : 0;
}

/* Full forward: every row, O [B,H,N,d] and L [B,H,N] in float64. */
int oracle_sdpa_forward(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                        int B, int H, int N, int d, int causal, double scale,
                        const int32_t *key_len, double *O_out, double *lse_out, int nthreads)
{
    return oracle_sdpa_rows(Q, K, V, B, H, N, N, d, causal, scale, key_len, NULL,
                            (int64_t)B * H * N, O_out, lse_out, nthreads);
}

/* Decode: one query per (b, h) over the first seqlens[b] cached keys, no
 * splitting.  q: [B,H,d]; Kc, Vc: [B,H,Lmax,d]; O: [B,H,d]; L: [B,H]. */
int oracle_decode(const uint16_t *q, const uint16_t *Kc, const uint16_t *Vc,
                  const int32_t *seqlens, int B, int H, int Lmax, int d, double scale,
                  double *O_out, double *lse_out, int nthreads)
{
    return oracle_sdpa_rows(q, Kc, Vc, B, H, 1, Lmax, d, 0, scale, seqlens, NULL,
                            (int64_t)B * H, O_out, lse_out, nthreads);
}

/* Paged decode ("CMU 10-423 Lecture 18", section 7.3, PagedAttention): the
 * cache is a pool of fixed-size blocks, and block_table[b * max_blocks + i]
 * names the physical block that holds tokens i*bs .. i*bs+bs-1 of sequence b.
 * Pool layout: [num_blocks][H][bs][d] (bf16 bits).  The keys and values of
 * sequence b are gathered through its table (tokens t < seqlens[b], clamped
 * to max_blocks * bs) and attended exactly as in oracle_decode: one explicit
 * score row, its stable softmax, no split.  Returns -1 on a table entry
 * outside [0, num_blocks). */
int oracle_decode_paged(const uint16_t *q, const uint16_t *Kpool, const uint16_t *Vpool,
                        const int32_t *block_table, int max_blocks, const int32_t *seqlens,
                        int B, int H, int num_blocks, int bs, int d, double scale,
                        double *O_out, double *lse_out, int nthreads)
{
    if (B < 0 || H < 0 || num_blocks <= 0 || bs <= 0 || d <= 0 || max_blocks < 0) return -1;
    if (nthreads <= 0) nthreads = 1;
    const int cap = max_blocks * bs;
    int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        int n = seqlens[b];
        if (n < 0) n = 0;
        if (n > cap) n = cap;
        double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double *vr = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)d);
        double *qv = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !vr || !qv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
            free(s); free(vr); free(qv);
            continue;
        }
        for (int c = 0; c < d; ++c) qv[c] = widen_bf16(q[(size_t)bh * d + c]);
        int ok = 1;
        for (int t = 0; t < n && ok; ++t) {
            const int phys = block_table[(size_t)b * max_blocks + t / bs];
            if (phys < 0 || phys >= num_blocks) { ok = 0; break; }
            const size_t row = (((size_t)phys * H + h) * bs + (size_t)(t % bs)) * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += qv[c] * widen_bf16(Kpool[row + c]);
            s[t] = scale * acc;
            for (int c = 0; c < d; ++c) vr[(size_t)t * d + c] = widen_bf16(Vpool[row + c]);
        }
        if (ok) {
            oracle_attend_scores(s, vr, n, d, O_out + (size_t)bh * d, lse_out + bh);
        } else {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        }
        free(s); free(vr); free(qv);
    }
    return bad ? -1 : 0;
}

/* -------------------------------------------------------------------------
 * Forward on float64 inputs (the same definition as oracle_sdpa_rows, for
 * inputs that are not bfloat16 values: the finite-difference checks of the
 * backward perturb the inputs by amounts bfloat16 cannot represent).
 * Q, K, V: [B,H,N,d] float64; O_out [B,H,N,d], lse_out [B,H,N].
 * ------------------------------------------------------------------------- */
int oracle_sdpa_forward_f64(const double *Q, const double *K, const double *V,
                            int B, int H, int N, int d, int causal, double scale,
                            const int32_t *key_len, double *O_out, double *lse_out)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!s) return -1;
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        const int b = (int)(bh / H);
        const double *kb = K + (size_t)bh * N * d;
        const double *vb = V + (size_t)bh * N * d;
        for (int i = 0; i < N; ++i) {
            int nvalid = N;
            if (key_len) nvalid = key_len[b] < nvalid ? key_len[b] : nvalid;
            if (causal && i + 1 < nvalid) nvalid = i + 1;
            if (nvalid < 0) nvalid = 0;
            const double *q = Q + ((size_t)bh * N + i) * d;
            for (int j = 0; j < nvalid; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += q[c] * kb[(size_t)j * d + c];
                s[j] = scale * acc;
            }
            oracle_attend_scores(s, vb, nvalid, d, O_out + ((size_t)bh * N + i) * d, lse_out + (size_t)bh * N + i);
        }
    }
    free(s);
    return 0;
}

/* -------------------------------------------------------------------------
 * Backward ("Infra: Flash Attention", "Backward and recomputation" and
 * "Blocked gradient computation"; CMU 10-423 Lecture 18 notes, 5.3).
 *
 * For every (b, h) and query row i, over the valid keys j (key_len, causal
 * j <= i), with G = dO the upstream gradient:
 *   S_ij  = scale * Q_i . K_j,   L_i = log sum_j exp(S_ij)
 *   P_ij  = exp(S_ij - L_i)
 *   dP_ij = G_i . V_j             (the page's H = G V^T)
 *   D_i   = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dV_j += P_ij G_i,  dK_j += scale dS_ij Q_i,  dQ_i = scale sum_j dS_ij K_j
 * Rows without a valid key contribute nothing (P = 0).
 *
 * Inputs float64 [B,H,N,d]; outputs dQ, dK, dV [B,H,N,d], D and L [B,H,N].
 * If mag != NULL it receives three arrays [3][B,H,N,d] of term magnitudes
 * used by the GPU parity tests to bound rounding error per element:
 *   M_dV[j,c] = sum_i P_ij |G_ic|
 *   M_dK[j,c] = scale sum_i P_ij (|dP_ij| + A_i) |Q_ic|
 *   M_dQ[i,c] = scale sum_j P_ij (|dP_ij| + A_i) |K_jc|
 * with A_i = |D_i| + sum_c |G_ic| |O_ic| (O_i = sum_j P_ij V_j).
 * Returns 0, or -1 on bad sizes / allocation failure.
 * ------------------------------------------------------------------------- */
int oracle_sdpa_backward(const double *Q, const double *K, const double *V, const double *dO,
                         int B, int H, int N, int d, int causal, double scale, const int32_t *key_len,
                         double *dQ, double *dK, double *dV, double *D_out, double *L_out,
                         double *mag, int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0) return -1;
    if (nthreads <= 0) nthreads = 1;
    const size_t total = (size_t)B * H * N * d;
    memset(dQ, 0, sizeof(double) * total);
    memset(dK, 0, sizeof(double) * total);
    memset(dV, 0, sizeof(double) * total);
    if (mag) memset(mag, 0, sizeof(double) * 3 * total);
    int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        const int b = (int)(bh / H);
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double *pr = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !pr || !dp || !o) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
            free(s); free(pr); free(dp); free(o);
            continue;
        }
        const size_t base = (size_t)bh * N * d;
        const double *kb = K + base, *vb = V + base;
        double *dKb = dK + base, *dVb = dV + base;
        double *MdV = mag ? mag + base : NULL;
        double *MdK = mag ? mag + total + base : NULL;
        double *MdQ = mag ? mag + 2 * total + base : NULL;
        for (int i = 0; i < N; ++i) {
            int nvalid = N;
            if (key_len) nvalid = key_len[b] < nvalid ? key_len[b] : nvalid;
            if (causal && i + 1 < nvalid) nvalid = i + 1;
            if (nvalid < 0) nvalid = 0;
            const double *q = Q + base + (size_t)i * d;
            const double *g = dO + base + (size_t)i * d;
            double *dq = dQ + base + (size_t)i * d;
            if (nvalid == 0) {
                D_out[(size_t)bh * N + i] = 0.0;
                L_out[(size_t)bh * N + i] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int j = 0; j < nvalid; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += q[c] * kb[(size_t)j * d + c];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int j = 0; j < nvalid; ++j) l += exp(s[j] - m);
            const double L = m + log(l);
            L_out[(size_t)bh * N + i] = L;
            double D = 0.0;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            for (int j = 0; j < nvalid; ++j) {
                pr[j] = exp(s[j] - L);
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += g[c] * vb[(size_t)j * d + c];
                dp[j] = acc;
                D += pr[j] * dp[j];
                for (int c = 0; c < d; ++c) o[c] += pr[j] * vb[(size_t)j * d + c];
            }
            D_out[(size_t)bh * N + i] = D;
            double A = fabs(D);
            for (int c = 0; c < d; ++c) A += fabs(g[c]) * fabs(o[c]);
            for (int j = 0; j < nvalid; ++j) {
                const double ds = pr[j] * (dp[j] - D);
                const double w = pr[j] * (fabs(dp[j]) + A);
                for (int c = 0; c < d; ++c) {
                    dVb[(size_t)j * d + c] += pr[j] * g[c];
                    dKb[(size_t)j * d + c] += scale * ds * q[c];
                    dq[c] += scale * ds * kb[(size_t)j * d + c];
                    if (mag) {
                        MdV[(size_t)j * d + c] += pr[j] * fabs(g[c]);
                        MdK[(size_t)j * d + c] += scale * w * fabs(q[c]);
                        MdQ[(size_t)i * d + c] += scale * w * fabs(kb[(size_t)j * d + c]);
                    }
                }
            }
        }
        free(s); free(pr); free(dp); free(o);
    }
    return bad ? -1 : 0;
}

/* E4M3 (OCP 8-bit floating point) to float64, exactly:
 *   exponent field e in 1..15: (-1)^s * 2^(e-7) * (1 + m/8)
 *   e = 0 (subnormal):         (-1)^s * 2^(-6) * (m/8)
 *   e = 15 and m = 7:          NaN (the format has no infinities) */
void oracle_e4m3_to_f64(const uint8_t *x, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) {
        const unsigned b = x[i];
        const int sgn = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
        double v;
        if (e == 15 && m == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)m / 8.0, -6);
        else
            v = ldexp(1.0 + (double)m / 8.0, e - 7);
        out[i] = sgn ? -v : v;
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
