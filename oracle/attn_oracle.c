/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact softmax attention,
 * forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition of attention that the tiled method
 * reproduces exactly ("FlashAttention-2-ICLR24", section 问题与动机: standard
 * attention forms S = QK^T and P = softmax(S); the tiled kernel is exact):
 *
 *   S_ij  = scale * sum_c Q_ic K_jc          (key j hidden when causal and j > i)
 *   m_i   = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
 *   LSE_i = m_i + ln(l_i)                     ("FlashAttention-2-ICLR24", 核心方法 1:
 *                                              only the logsumexp is kept)
 *   P_ij  = exp(S_ij - LSE_i),  O_i = sum_j P_ij V_j
 *   D_i   = sum_c dO_ic O_ic
 *   dP_ij = sum_c dO_ic V_jc,  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij K_j,  dK_j = scale sum_i dS_ij Q_i,  dV_j = sum_i P_ij dO_i
 *
 * The backward pass is the five products named in "FlashAttention-4反向传播优化"
 * section 1.1 (S, dP, dV, dK, dQ), with P recomputed from the stored LSE.
 * For grouped/multi-query attention ("FlashAttention-2-ICLR24", 核心方法 4)
 * query head h reads key/value head g = floor(h * Hkv / Hq), and dK/dV of g are
 * the sums over every query head that maps to g.
 *
 * Softmax is the two-pass exact form (max, then sum); there is no online
 * rescaling here.  S and P are materialised one full row (row routine) or one
 * full column (column routine) at a time, which keeps memory O(N) so that the
 * longest sequences still fit.
 *
 * Layout: packed token-major arrays [T, H, d] (d innermost), sequence b owning
 * tokens cu[b] .. cu[b+1]-1.  lse and D are [Hq, T].  All arithmetic is fp64.
 *
 * Queries and keys may have different lengths (the *_kv entry points: query
 * sequence b owns tokens cu_q[b].., key/value sequence b owns cu_k[b]..).  The
 * pages state the causal mask only for equal lengths; the reading here is that
 * the Lq queries are the LAST Lq positions of the Lk-long key sequence (as when
 * new tokens attend to a cache of earlier ones): under the causal mask query i
 * sees key j iff j <= i + (Lk - Lq).  With Lq = Lk this is j <= i.  A row that
 * sees no key (causal with i < Lq - Lk) gets O = 0, LSE = -inf, D = 0 and
 * contributes nothing to any gradient.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX(t, h, H, d) (((size_t)(t) * (size_t)(H) + (size_t)(h)) * (size_t)(d))

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

static int kv_head(int h, int Hq, int Hkv) { return (int)(((long long)h * Hkv) / Hq); }

/*
 * One query row i (query head h, key/value head g) of a sequence whose keys
 * start at token tk0, Lk keys long, with causal offset off = Lk - Lq: the score
 * row, the exact two-pass softmax, O_i and LSE_i; when doi != NULL also D_i,
 * the dP and dS rows and dQ_i.  row_s and row_p are scratch of length >= Lk.
 * Outputs: oi[d], *lse_i, and (backward) *D_i, dqi[d].
 */
static void row_compute(const double* qi, const double* k, const double* v, const double* doi,
                        int tk0, int Lk, int off, int i, int g, int Hkv, int d, double scale,
                        int causal, double* row_s, double* row_p,
                        double* oi, double* lse_i, double* D_i, double* dqi) {
    int nv = Lk;
    if (causal) {
        nv = i + off + 1;  /* keys j <= i + off are visible */
        if (nv > Lk) nv = Lk;
    }
    for (int c = 0; c < d; ++c) oi[c] = 0.0;
    if (doi)
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
    if (nv <= 0) {
        *lse_i = -INFINITY;
        if (doi) *D_i = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int j = 0; j < nv; ++j) {
        row_s[j] = scale * dot(qi, k + IDX(tk0 + j, g, Hkv, d), d);
        if (row_s[j] > m) m = row_s[j];
    }
    double l = 0.0;
    for (int j = 0; j < nv; ++j) l += exp(row_s[j] - m);
    const double lse = m + log(l);
    *lse_i = lse;
    for (int j = 0; j < nv; ++j) row_p[j] = exp(row_s[j] - lse);
    for (int j = 0; j < nv; ++j) {
        const double* vj = v + IDX(tk0 + j, g, Hkv, d);
        for (int c = 0; c < d; ++c) oi[c] += row_p[j] * vj[c];
    }
    if (!doi) return;
    const double Di = dot(doi, oi, d);
    *D_i = Di;
    for (int j = 0; j < nv; ++j) {
        const double dP = dot(doi, v + IDX(tk0 + j, g, Hkv, d), d);
        const double dS = row_p[j] * (dP - Di);
        const double* kj = k + IDX(tk0 + j, g, Hkv, d);
        for (int c = 0; c < d; ++c) dqi[c] += scale * dS * kj[c];
    }
}

/*
 * One key column j (key/value head g) of a sequence whose queries start at
 * token tq0 (Lq rows) and keys at tk0, causal offset off = Lk - Lq: for every
 * query head h in [h_lo, h_hi) that maps to g (increasing h) and every row
 * i >= i_lo that sees key j (i >= j - off under the causal mask), recompute
 * S_ij and P_ij = exp(S_ij - LSE_i), dP_ij and dS_ij = P_ij (dP_ij - D_i), and
 * accumulate dK_j and dV_j.  LSE_i / D_i of head h are read at
 * [h * ld_head + (i - i_lo)].
 */
static void col_compute(const double* q, const double* k, const double* v, const double* dout,
                        const double* lse, const double* D, size_t ld_head, int i_lo,
                        int tq0, int Lq, int tk0, int off, int j, int g, int h_lo, int h_hi,
                        int Hq, int Hkv, int d, double scale, int causal, double* dkj,
                        double* dvj) {
    const double* kj = k + IDX(tk0 + j, g, Hkv, d);
    const double* vj = v + IDX(tk0 + j, g, Hkv, d);
    for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
    for (int h = h_lo; h < h_hi; ++h) {
        if (kv_head(h, Hq, Hkv) != g) continue;
        int i0 = causal ? j - off : 0;
        if (i0 < i_lo) i0 = i_lo;
        for (int i = i0; i < Lq; ++i) {
            const double* qi = q + IDX(tq0 + i, h, Hq, d);
            const double* doi = dout + IDX(tq0 + i, h, Hq, d);
            const double S = scale * dot(qi, kj, d);
            const double P = exp(S - lse[(size_t)h * ld_head + (size_t)(i - i_lo)]);
            const double dP = dot(doi, vj, d);
            const double dS = P * (dP - D[(size_t)h * ld_head + (size_t)(i - i_lo)]);
            for (int c = 0; c < d; ++c) {
                dvj[c] += P * doi[c];
                dkj[c] += scale * dS * qi[c];
            }
        }
    }
}

static int max_len(int nseq, const int* cu) {
    int mx = 0;
    for (int b = 0; b < nseq; ++b)
        if (cu[b + 1] - cu[b] > mx) mx = cu[b + 1] - cu[b];
    return mx;
}

/*
 * Full oracle over query heads [h_lo, h_hi) of every sequence; queries of
 * sequence b are tokens cu_q[b].. and its keys/values tokens cu_k[b]..
 * Forward outputs o [Tq,Hq,d] and lse [Hq,Tq] are written for those heads.
 * If dout != NULL the backward pass also runs: D [Hq,Tq], dq [Tq,Hq,d], and
 * dk, dv [Tk,Hkv,d] for every kv head that some head in [h_lo, h_hi) maps to
 * (summing only over the heads in range).  Returns 0, or -1 on bad arguments.
 */
int oracle_attention_kv(const double* q, const double* k, const double* v, const double* dout,
                        double* o, double* lse, double* D, double* dq, double* dk, double* dv,
                        int nseq, const int* cu_q, const int* cu_k, int Hq, int Hkv, int d,
                        double scale, int causal, int h_lo, int h_hi) {
    if (nseq < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || h_lo < 0 || h_hi > Hq || h_lo > h_hi)
        return -1;
    const int Tq = cu_q[nseq];
    const int Lkmax = max_len(nseq, cu_k);
    /* rows are independent */
    #pragma omp parallel
    {
        double* row_s = (double*)malloc(sizeof(double) * (size_t)(Lkmax > 0 ? Lkmax : 1));
        double* row_p = (double*)malloc(sizeof(double) * (size_t)(Lkmax > 0 ? Lkmax : 1));
        for (int b = 0; b < nseq; ++b) {
            const int tq0 = cu_q[b], Lq = cu_q[b + 1] - cu_q[b];
            const int tk0 = cu_k[b], Lk = cu_k[b + 1] - cu_k[b];
            for (int h = h_lo; h < h_hi; ++h) {
                const int g = kv_head(h, Hq, Hkv);
                #pragma omp for schedule(dynamic, 4)
                for (int i = 0; i < Lq; ++i) {
                    const size_t at = IDX(tq0 + i, h, Hq, d);
                    const size_t st = (size_t)h * Tq + (size_t)(tq0 + i);
                    row_compute(q + at, k, v, dout ? dout + at : NULL, tk0, Lk, Lk - Lq, i, g,
                                Hkv, d, scale, causal, row_s, row_p, o + at, lse + st,
                                dout ? D + st : NULL, dout ? dq + at : NULL);
                }
            }
        }
        free(row_s);
        free(row_p);
    }
    if (!dout) return 0;
    /* key columns are independent; lse/D of sequence b start at query token tq0 */
    const int g_lo = kv_head(h_lo, Hq, Hkv);
    const int g_hi = h_hi > h_lo ? kv_head(h_hi - 1, Hq, Hkv) + 1 : g_lo;
    for (int b = 0; b < nseq; ++b) {
        const int tq0 = cu_q[b], Lq = cu_q[b + 1] - cu_q[b];
        const int tk0 = cu_k[b], Lk = cu_k[b + 1] - cu_k[b];
        for (int g = g_lo; g < g_hi; ++g) {
            #pragma omp parallel for schedule(dynamic, 4)
            for (int j = 0; j < Lk; ++j)
                col_compute(q, k, v, dout, lse + tq0, D + tq0, (size_t)Tq, 0, tq0, Lq, tk0,
                            Lk - Lq, j, g, h_lo, h_hi, Hq, Hkv, d, scale, causal,
                            dk + IDX(tk0 + j, g, Hkv, d), dv + IDX(tk0 + j, g, Hkv, d));
        }
    }
    return 0;
}

/* Equal query and key lengths: the same sequence boundaries for both. */
int oracle_attention(const double* q, const double* k, const double* v, const double* dout,
                     double* o, double* lse, double* D, double* dq, double* dk, double* dv,
                     int nseq, const int* cu, int Hq, int Hkv, int d, double scale, int causal,
                     int h_lo, int h_hi) {
    return oracle_attention_kv(q, k, v, dout, o, lse, D, dq, dk, dv, nseq, cu, cu, Hq, Hkv, d,
                               scale, causal, h_lo, h_hi);
}

/*
 * Selected rows of one (sequence b, query head h): O_i, LSE_i and, when dout
 * is given, D_i and dQ_i for each row i in rows[0..nrows) (positions within
 * the query sequence).  Every quantity of the row routine depends on row i
 * alone, so this is the full oracle restricted to those rows.  Outputs are
 * compact: o_rows/dq_rows [nrows, d], lse_rows and D_rows [nrows].  Returns 0,
 * or -1 on bad arguments.
 */
int oracle_rows_kv(const double* q, const double* k, const double* v, const double* dout,
                   int nseq, const int* cu_q, const int* cu_k, int Hq, int Hkv, int d,
                   double scale, int causal, int b, int h, const int* rows, int nrows,
                   double* o_rows, double* lse_rows, double* D_rows, double* dq_rows) {
    if (b < 0 || b >= nseq || h < 0 || h >= Hq || nrows < 0) return -1;
    const int tq0 = cu_q[b], Lq = cu_q[b + 1] - cu_q[b];
    const int tk0 = cu_k[b], Lk = cu_k[b + 1] - cu_k[b];
    const int g = kv_head(h, Hq, Hkv);
    for (int r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= Lq) return -1;
    #pragma omp parallel
    {
        double* row_s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double* row_p = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            const int i = rows[r];
            const size_t at = IDX(tq0 + i, h, Hq, d);
            row_compute(q + at, k, v, dout ? dout + at : NULL, tk0, Lk, Lk - Lq, i, g, Hkv, d,
                        scale, causal, row_s, row_p, o_rows + (size_t)r * d, lse_rows + r,
                        dout ? D_rows + r : NULL, dout ? dq_rows + (size_t)r * d : NULL);
        }
        free(row_s);
        free(row_p);
    }
    return 0;
}

int oracle_rows(const double* q, const double* k, const double* v, const double* dout,
                int nseq, const int* cu, int Hq, int Hkv, int d, double scale, int causal,
                int b, int h, const int* rows, int nrows,
                double* o_rows, double* lse_rows, double* D_rows, double* dq_rows) {
    return oracle_rows_kv(q, k, v, dout, nseq, cu, cu, Hq, Hkv, d, scale, causal, b, h, rows,
                          nrows, o_rows, lse_rows, D_rows, dq_rows);
}

/*
 * dK_j and dV_j for selected keys (positions within key sequence b) of one
 * key/value head g, summed over every query head that maps to g.  Only rows
 * i >= min(keys) - (Lk - Lq) can see those keys under the causal mask, so
 * LSE_i and D_i are computed (row routine) for rows i >= i_lo only, where
 * i_lo = (causal ? max(0, min(keys) - (Lk - Lq)) : 0) -- the result is exact,
 * and cheap for keys near the end of a causal sequence.
 * Outputs are compact: dk_rows, dv_rows [nkeys, d].  Returns 0, -1 on bad
 * arguments, -2 if scratch allocation fails.
 */
int oracle_key_grads_kv(const double* q, const double* k, const double* v, const double* dout,
                        int nseq, const int* cu_q, const int* cu_k, int Hq, int Hkv, int d,
                        double scale, int causal, int b, int g, const int* keys, int nkeys,
                        double* dk_rows, double* dv_rows) {
    if (b < 0 || b >= nseq || g < 0 || g >= Hkv || nkeys <= 0) return -1;
    const int tq0 = cu_q[b], Lq = cu_q[b + 1] - cu_q[b];
    const int tk0 = cu_k[b], Lk = cu_k[b + 1] - cu_k[b];
    const int off = Lk - Lq;
    int kmin = Lk;
    for (int r = 0; r < nkeys; ++r) {
        if (keys[r] < 0 || keys[r] >= Lk) return -1;
        if (keys[r] < kmin) kmin = keys[r];
    }
    int i_lo = causal ? kmin - off : 0;
    if (i_lo < 0) i_lo = 0;
    const int nrow = Lq > i_lo ? Lq - i_lo : 0;
    const size_t nalloc = (size_t)Hq * (size_t)(nrow > 0 ? nrow : 1);
    double* lse = (double*)malloc(sizeof(double) * nalloc);
    double* Dv = (double*)malloc(sizeof(double) * nalloc);
    if (!lse || !Dv) { free(lse); free(Dv); return -2; }
    for (int h = 0; h < Hq; ++h) {
        if (kv_head(h, Hq, Hkv) != g) continue;
        #pragma omp parallel
        {
            double* row_s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
            double* row_p = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
            double* o_i = (double*)malloc(sizeof(double) * (size_t)d);
            double* dq_i = (double*)malloc(sizeof(double) * (size_t)d);
            #pragma omp for schedule(dynamic, 4)
            for (int i = i_lo; i < Lq; ++i) {
                const size_t at = IDX(tq0 + i, h, Hq, d);
                row_compute(q + at, k, v, dout + at, tk0, Lk, off, i, g, Hkv, d, scale, causal,
                            row_s, row_p, o_i, lse + (size_t)h * nrow + (i - i_lo),
                            Dv + (size_t)h * nrow + (i - i_lo), dq_i);
            }
            free(row_s);
            free(row_p);
            free(o_i);
            free(dq_i);
        }
    }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < nkeys; ++r)
        col_compute(q, k, v, dout, lse, Dv, (size_t)nrow, i_lo, tq0, Lq, tk0, off, keys[r], g, 0,
                    Hq, Hq, Hkv, d, scale, causal, dk_rows + (size_t)r * d,
                    dv_rows + (size_t)r * d);
    free(lse);
    free(Dv);
    return 0;
}

int oracle_key_grads(const double* q, const double* k, const double* v, const double* dout,
                     int nseq, const int* cu, int Hq, int Hkv, int d, double scale, int causal,
                     int b, int g, const int* keys, int nkeys, double* dk_rows, double* dv_rows) {
    return oracle_key_grads_kv(q, k, v, dout, nseq, cu, cu, Hq, Hkv, d, scale, causal, b, g,
                               keys, nkeys, dk_rows, dv_rows);
}
