/*
 * oracle.c -- plain, slow, fp64 CPU oracle for exact (causal) attention, its
 * analytic gradients, chunk-pair partials, the log-sum-exp merge and the
 * sequence partitions used by ring-style context parallelism.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark load it.  It shares no code, header or constant with the
 * CUDA path.
 *
 * Every function is the plain definition written out, row by row, in double
 * precision, with no tiling, no online rescaling and no fusion:
 *
 *   s_ij  = scale * q_i . k_j                 (masked to -inf where the key is
 *                                              in the query's future)
 *   LSE_i = ln sum_j exp(s_ij)                 (computed as m + ln sum exp(s - m))
 *   P_ij  = exp(s_ij - LSE_i),  O_i = sum_j P_ij v_j
 *
 *   Striped Attention Guide, "The Fatal Flaw: Causal Workload Imbalance" (the
 *   causal score matrix A_ij, j <= i kept, j > i set to -inf) and
 *   "Incremental Online Softmax Rescaling" (m, l and O/l); FlashAttention
 *   glossary entry (exact attention; the backward pass is recomputed from the
 *   softmax statistics, read here as the per-row log-sum-exp).
 *
 * Gradients follow the chain rule of that definition, without the
 * D = rowsum(dO * O) shortcut that fast kernels use:
 *   dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . v_j,
 *   dS_ij = P_ij (dP_ij - sum_l P_il dP_il),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i.
 * The pages print no backward formulas; these are the analytic gradients of
 * the forward definition (pinned by finite differences in the tests).
 *
 * Grouped-query attention: query head h reads key/value head h / (Hq/Hkv)
 * (contiguous groups; the pages do not fix the mapping).  dK and dV of a
 * key/value head are summed over its query heads.
 *
 * Tensors are [B, H, L, d] contiguous; q/k/v/dout are bf16 bit patterns
 * (uint16), widened exactly to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element i of an input tensor: bf16 bit patterns (f64 == 0) widened exactly,
 * or plain doubles (f64 != 0, used by the finite-difference checks). */
static inline double ld(const void* p, int64_t i, int f64)
{
    return f64 ? ((const double*)p)[i] : bf(((const uint16_t*)p)[i]);
}

/* ---------------------------------------------------------------------------
 * Document masking (Striped Attention Guide, "Document Packing and Boundary
 * Alignment": documents concatenated into one sequence must not attend to
 * each other; boundaries by cumulative document indexing).  Reading: the
 * documents are the position ranges [bounds[t], bounds[t+1]), t < ndocs; a
 * key is visible to a query only when both positions lie in the same range
 * (and, when causal, the key's position is not after the query's).  Set once
 * with orc_set_docs (ndocs = 0: no documents); it applies to
 * orc_attn_fwd_rows, orc_attn_bwd and orc_attn_bwd_q_rows.
 * ------------------------------------------------------------------------- */
static int64_t* g_docs = NULL;
static int g_ndocs = 0;

void orc_set_docs(const int64_t* bounds, int ndocs)
{
    free(g_docs);
    g_docs = NULL;
    g_ndocs = 0;
    if (ndocs > 0 && bounds) {
        g_docs = (int64_t*)malloc(sizeof(int64_t) * (size_t)(ndocs + 1));
        memcpy(g_docs, bounds, sizeof(int64_t) * (size_t)(ndocs + 1));
        g_ndocs = ndocs;
    }
}

/* index of the document holding position x (-1 outside every document) */
static int doc_of(int64_t x)
{
    for (int t = 0; t < g_ndocs; ++t)
        if (g_docs[t] <= x && x < g_docs[t + 1])
            return t;
    return -1;
}

static int visible(int causal, int64_t pi, int64_t pj)
{
    if (causal && pj > pi)
        return 0;
    if (g_ndocs > 0 && doc_of(pi) != doc_of(pj))
        return 0;
    return 1;
}

/* ---------------------------------------------------------------------------
 * Sequence partitions.
 *
 * kind 0, contiguous: worker p owns tokens [p*N/P, (p+1)*N/P)
 *   (DistFlashAttn Guide, "The Causal Imbalance Crisis"; Striped Attention
 *   Guide, "Mathematical Formulation of Token Striping", the contiguous
 *   interval I_p).
 * kind 1, folded / load-balanced: the sequence is cut into 2P equal chunks and
 *   worker p owns chunk p followed by chunk 2P-1-p
 *   (DistFlashAttn Guide, "The Folded Chunk Assignment").
 * kind 2, striped with block size s: worker p owns every token whose block
 *   index floor(i/s) is congruent to p mod P, in increasing order; s = 1 is
 *   round-robin token striping, i = m*P + p
 *   (Striped Attention Guide, "Mathematical Formulation of Token Striping",
 *   the block-striped set, and "Preserving Rotary Position Embeddings", the
 *   position m*P + p).
 * Returns the global token index of local row m of worker p, or -1 when the
 * arguments do not describe a valid partition.
 * ------------------------------------------------------------------------- */
int64_t orc_partition_pos(int kind, int64_t N, int P, int stripe, int p, int64_t m)
{
    if (P <= 0 || p < 0 || p >= P || N <= 0 || N % P != 0)
        return -1;
    int64_t n = N / P;
    if (m < 0 || m >= n)
        return -1;
    if (kind == 0) {
        return (int64_t)p * n + m;
    } else if (kind == 1) {
        if (N % (2 * (int64_t)P) != 0)
            return -1;
        int64_t c = N / (2 * (int64_t)P);
        if (m < c)
            return (int64_t)p * c + m;
        return (int64_t)(2 * P - 1 - p) * c + (m - c);
    } else if (kind == 2) {
        int64_t s = stripe;
        if (s <= 0 || N % (s * P) != 0)
            return -1;
        /* walk the blocks of the whole sequence and keep worker p's, in order */
        int64_t local_block = m / s, off = m % s;
        int64_t seen = -1;
        for (int64_t blk = 0; blk < N / s; ++blk) {
            if (blk % P == p) {
                ++seen;
                if (seen == local_block)
                    return blk * s + off;
            }
        }
        return -1;
    }
    return -1;
}

/* Fill pos[0..n) for worker p. */
int orc_partition_fill(int kind, int64_t N, int P, int stripe, int p, int64_t* pos)
{
    int64_t n = N / P;
    for (int64_t m = 0; m < n; ++m) {
        pos[m] = orc_partition_pos(kind, N, P, stripe, p, m);
        if (pos[m] < 0)
            return -1;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Forward attention for selected query rows.
 *
 * q: [B,Hq,Lq,d]; k, v: [B,Hkv,Lk,d] (element type per f64, see ld()).
 * qpos[Lq], kpos[Lk] are global token positions (NULL = 0..L-1).  With
 * causal != 0 key j is visible to query i iff kpos[j] <= qpos[i] (diagonal
 * included); otherwise every key is visible.  rows[r] is a flat index
 * (b*Hq + h)*Lq + i; the outputs are o[r*d + c] and lse[r].  A row that sees
 * no key gets O = 0 and LSE = -inf (the zero-sum convention of the Striped
 * Attention Guide's engine: the normaliser 0 is replaced by 1, leaving O = 0).
 * ------------------------------------------------------------------------- */
void orc_attn_fwd_rows(const void* q, const void* k, const void* v, int f64,
                       int B, int Hq, int Hkv, int64_t Lq, int64_t Lk, int d,
                       int causal, double scale, const int64_t* qpos,
                       const int64_t* kpos, int64_t nrows, const int64_t* rows,
                       double* o, double* lse, int nthreads)
{
    (void)B;
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double* qi = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t flat = rows[r];
            int64_t i = flat % Lq;
            int64_t bh = flat / Lq;
            int64_t b = bh / Hq;
            int h = (int)(bh % Hq);
            int hk = h / G;
            int64_t kb = ((b * Hkv + hk) * Lk) * d; /* element offset of K/V head */
            int64_t pi = qpos ? qpos[i] : i;
            for (int c = 0; c < d; ++c)
                qi[c] = ld(q, flat * d + c, f64);
            double m = -INFINITY;
            for (int64_t j = 0; j < Lk; ++j) {
                int64_t pj = kpos ? kpos[j] : j;
                if (!visible(causal, pi, pj)) {
                    s[j] = -INFINITY;
                    continue;
                }
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += qi[c] * ld(k, kb + j * d + c, f64);
                s[j] = scale * acc;
                if (s[j] > m)
                    m = s[j];
            }
            double* orow = o + r * d;
            for (int c = 0; c < d; ++c)
                orow[c] = 0.0;
            if (m == -INFINITY) {
                lse[r] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int64_t j = 0; j < Lk; ++j)
                if (s[j] != -INFINITY)
                    l += exp(s[j] - m);
            double L = m + log(l);
            lse[r] = L;
            for (int64_t j = 0; j < Lk; ++j) {
                if (s[j] == -INFINITY)
                    continue;
                double pij = exp(s[j] - L);
                for (int c = 0; c < d; ++c)
                    orow[c] += pij * ld(v, kb + j * d + c, f64);
            }
        }
        free(s);
        free(qi);
    }
}

/* ---------------------------------------------------------------------------
 * Full backward for every row, by the chain rule above.
 *
 * dq: [B,Hq,Lq,d]; dk, dv: [B,Hkv,Lk,d] (summed over the G query heads of a
 * key/value head).  Outputs are overwritten.
 *
 * When lse_in / delta_in are non-NULL the softmax is normalised with the given
 * per-row log-sum-exp and the row constant sum_l P_il dP_il is taken from
 * delta_in: this is the contribution of one chunk pair (the keys of the chunk
 * only) to the gradient of the attention over the whole sequence, whose
 * statistics are supplied.  With NULL they are computed from the keys given.
 * ------------------------------------------------------------------------- */
void orc_attn_bwd(const void* q, const void* k, const void* v, const void* dout,
                  int f64, int B, int Hq, int Hkv, int64_t Lq, int64_t Lk, int d,
                  int causal, double scale, const int64_t* qpos,
                  const int64_t* kpos, const double* lse_in,
                  const double* delta_in, double* dq, double* dk, double* dv,
                  int nthreads)
{
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    memset(dq, 0, sizeof(double) * (size_t)B * Hq * Lq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Lk * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Lk * d);
    /* one (b, kv head) group per thread, so that dK/dV sums never race */
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double* dp = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t grp = 0; grp < (int64_t)B * Hkv; ++grp) {
            int64_t b = grp / Hkv;
            int hk = (int)(grp % Hkv);
            int64_t kb = ((b * Hkv + hk) * Lk) * d;
            double* dkb = dk + kb;
            double* dvb = dv + kb;
            for (int g = 0; g < G; ++g) {
                int h = hk * G + g;
                for (int64_t i = 0; i < Lq; ++i) {
                    int64_t flat = (b * Hq + h) * Lq + i;
                    int64_t qr = flat * d;
                    int64_t pi = qpos ? qpos[i] : i;
                    double m = -INFINITY;
                    for (int64_t j = 0; j < Lk; ++j) {
                        int64_t pj = kpos ? kpos[j] : j;
                        if (!visible(causal, pi, pj)) {
                            s[j] = -INFINITY;
                            continue;
                        }
                        double acc = 0.0;
                        for (int c = 0; c < d; ++c)
                            acc += ld(q, qr + c, f64) * ld(k, kb + j * d + c, f64);
                        s[j] = scale * acc;
                        if (s[j] > m)
                            m = s[j];
                    }
                    if (m == -INFINITY)
                        continue; /* no visible key: every gradient term is 0 */
                    double L;
                    if (lse_in) {
                        L = lse_in[flat];
                        if (L == -INFINITY)
                            continue;
                    } else {
                        double l = 0.0;
                        for (int64_t j = 0; j < Lk; ++j)
                            if (s[j] != -INFINITY)
                                l += exp(s[j] - m);
                        L = m + log(l);
                    }
                    /* dP_ij = dO_i . v_j and the row constant sum_l P_il dP_il */
                    double rowc = 0.0;
                    for (int64_t j = 0; j < Lk; ++j) {
                        if (s[j] == -INFINITY) {
                            dp[j] = 0.0;
                            continue;
                        }
                        double acc = 0.0;
                        for (int c = 0; c < d; ++c)
                            acc += ld(dout, qr + c, f64) * ld(v, kb + j * d + c, f64);
                        dp[j] = acc;
                        rowc += exp(s[j] - L) * acc;
                    }
                    if (delta_in)
                        rowc = delta_in[flat];
                    double* dqr = dq + qr;
                    for (int64_t j = 0; j < Lk; ++j) {
                        if (s[j] == -INFINITY)
                            continue;
                        double pij = exp(s[j] - L);
                        double dsij = pij * (dp[j] - rowc);
                        for (int c = 0; c < d; ++c) {
                            dqr[c] += scale * dsij * ld(k, kb + j * d + c, f64);
                            dkb[j * d + c] += scale * dsij * ld(q, qr + c, f64);
                            dvb[j * d + c] += pij * ld(dout, qr + c, f64);
                        }
                    }
                }
            }
        }
        free(s);
        free(dp);
    }
}

/* ---------------------------------------------------------------------------
 * dQ for selected query rows only (the sampled-row check at long sequences),
 * causal or not, natural order.  rows[r] = (b*Hq + h)*Lq + i; dq[r*d + c].
 * Also returns the row's LSE and its row constant sum_l P_il dP_il (the
 * quantity fast kernels call D).
 * ------------------------------------------------------------------------- */
void orc_attn_bwd_q_rows(const void* q, const void* k, const void* v,
                         const void* dout, int f64, int B, int Hq, int Hkv,
                         int64_t Lq, int64_t Lk, int d, int causal, double scale,
                         int64_t nrows, const int64_t* rows, double* dq,
                         double* lse, double* rowconst, int nthreads)
{
    (void)B;
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double* dp = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t flat = rows[r];
            int64_t i = flat % Lq;
            int64_t bh = flat / Lq;
            int64_t b = bh / Hq;
            int h = (int)(bh % Hq);
            int hk = h / G;
            int64_t qr = flat * d;
            int64_t kb = ((b * Hkv + hk) * Lk) * d;
            double* dqr = dq + r * d;
            for (int c = 0; c < d; ++c)
                dqr[c] = 0.0;
            double m = -INFINITY;
            for (int64_t j = 0; j < Lk; ++j) {
                if (!visible(causal, i, j)) {
                    s[j] = -INFINITY;
                    continue;
                }
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += ld(q, qr + c, f64) * ld(k, kb + j * d + c, f64);
                s[j] = scale * acc;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < Lk; ++j)
                if (s[j] != -INFINITY)
                    l += exp(s[j] - m);
            double L = m + log(l);
            double rowc = 0.0;
            for (int64_t j = 0; j < Lk; ++j) {
                if (s[j] == -INFINITY) {
                    dp[j] = 0.0;
                    continue;
                }
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += ld(dout, qr + c, f64) * ld(v, kb + j * d + c, f64);
                dp[j] = acc;
                rowc += exp(s[j] - L) * acc;
            }
            for (int64_t j = 0; j < Lk; ++j) {
                if (s[j] == -INFINITY)
                    continue;
                double dsij = exp(s[j] - L) * (dp[j] - rowc);
                for (int c = 0; c < d; ++c)
                    dqr[c] += scale * dsij * ld(k, kb + j * d + c, f64);
            }
            lse[r] = L;
            rowconst[r] = rowc;
        }
        free(s);
        free(dp);
    }
}

/* ---------------------------------------------------------------------------
 * dK and dV for selected key rows of one (b, kv-head) group, causal, natural
 * order, without documents (orc_set_docs does not apply here).  First the
 * full softmax statistics (LSE_i and sum_l P_il dP_il) of every query row of
 * the group's G heads are computed from the definition; then, for each
 * selected key j, dV_j = sum_{h,i>=j} P_ij dO_i and
 * dK_j = scale sum_{h,i>=j} dS_ij q_i.  krows[r] is the key index j; outputs
 * are dk[r*d + c], dv[r*d + c].  Statistics are computed only for the query
 * rows that can see a selected key (i >= min krows).  Cost: O(G * (N - min
 * krows) * N * d).
 *
 * The group's rows are widened to double once (exactly, as ld() does) and the
 * dot products use four partial sums, so that a check of key rows anywhere
 * in a 128K-token sequence finishes in about a minute on a server's cores;
 * only the rounding order of the sums differs from a single running sum.
 * ------------------------------------------------------------------------- */
static double dot_rows(const double* a, const double* b, int d)
{
    double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
    int c = 0;
    for (; c + 4 <= d; c += 4) {
        s0 += a[c] * b[c];
        s1 += a[c + 1] * b[c + 1];
        s2 += a[c + 2] * b[c + 2];
        s3 += a[c + 3] * b[c + 3];
    }
    for (; c < d; ++c)
        s0 += a[c] * b[c];
    return (s0 + s1) + (s2 + s3);
}

void orc_attn_bwd_kv_rows(const void* q, const void* k, const void* v,
                          const void* dout, int f64, int B, int Hq, int Hkv,
                          int64_t N, int d, double scale, int b, int hk,
                          int64_t nkrows, const int64_t* krows, double* dk,
                          double* dv, int nthreads)
{
    (void)B;
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    /* only query rows i >= min(krows) can see a selected key (causal) */
    int64_t jmin = N;
    for (int64_t r = 0; r < nkrows; ++r)
        if (krows[r] < jmin)
            jmin = krows[r];
    if (nkrows <= 0 || jmin >= N)
        return;
    int64_t nrow = N - jmin;
    double* L = (double*)malloc(sizeof(double) * (size_t)G * nrow);
    double* RC = (double*)malloc(sizeof(double) * (size_t)G * nrow);
    double* Kd = (double*)malloc(sizeof(double) * (size_t)N * d);
    double* Vd = (double*)malloc(sizeof(double) * (size_t)N * d);
    double* Qd = (double*)malloc(sizeof(double) * (size_t)G * nrow * d);
    double* Od = (double*)malloc(sizeof(double) * (size_t)G * nrow * d);
    int64_t kb = (((int64_t)b * Hkv + hk) * N) * d;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int c = 0; c < d; ++c) {
            Kd[j * d + c] = ld(k, kb + j * d + c, f64);
            Vd[j * d + c] = ld(v, kb + j * d + c, f64);
        }
#pragma omp parallel for schedule(static)
    for (int64_t gi = 0; gi < (int64_t)G * nrow; ++gi) {
        int g = (int)(gi / nrow);
        int64_t i = jmin + gi % nrow;
        int64_t qr = ((((int64_t)b * Hq + hk * G + g) * N) + i) * d;
        for (int c = 0; c < d; ++c) {
            Qd[gi * d + c] = ld(q, qr + c, f64);
            Od[gi * d + c] = ld(dout, qr + c, f64);
        }
    }
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 16)
        for (int64_t gi = 0; gi < (int64_t)G * nrow; ++gi) {
            int64_t i = jmin + gi % nrow;
            const double* qi = Qd + gi * d;
            const double* oi = Od + gi * d;
            double m = -INFINITY;
            for (int64_t j = 0; j <= i; ++j) {
                s[j] = scale * dot_rows(qi, Kd + j * d, d);
                if (s[j] > m)
                    m = s[j];
            }
            /* e_j = exp(s_j - m), l = sum e_j, LSE = m + ln l, P_ij = e_j / l */
            double l = 0.0;
            for (int64_t j = 0; j <= i; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            double rowc = 0.0;
            for (int64_t j = 0; j <= i; ++j)
                rowc += (s[j] / l) * dot_rows(oi, Vd + j * d, d);
            L[gi] = m + log(l);
            RC[gi] = rowc;
        }
        free(s);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nkrows; ++r) {
        int64_t j = krows[r];
        double* dkr = dk + r * d;
        double* dvr = dv + r * d;
        for (int c = 0; c < d; ++c) {
            dkr[c] = 0.0;
            dvr[c] = 0.0;
        }
        const double* kj = Kd + j * d;
        const double* vj = Vd + j * d;
        for (int g = 0; g < G; ++g) {
            for (int64_t i = j; i < N; ++i) {
                int64_t gi = (int64_t)g * nrow + (i - jmin);
                const double* qi = Qd + gi * d;
                const double* oi = Od + gi * d;
                double sij = scale * dot_rows(qi, kj, d);
                double dpij = dot_rows(oi, vj, d);
                double pij = exp(sij - L[gi]);
                double dsij = pij * (dpij - RC[gi]);
                for (int c = 0; c < d; ++c) {
                    dvr[c] += pij * oi[c];
                    dkr[c] += scale * dsij * qi[c];
                }
            }
        }
    }
    free(L);
    free(RC);
    free(Kd);
    free(Vd);
    free(Qd);
    free(Od);
}

/* ---------------------------------------------------------------------------
 * Log-sum-exp merge of k partial results of the same query rows.
 *
 * LSE = ln sum_c exp(LSE_c);  O = sum_c exp(LSE_c - LSE) O_c.
 * A row whose partials are all -inf stays (O = 0, LSE = -inf).
 * (Striped Attention Guide, "Incremental Online Softmax Rescaling": the alpha /
 * beta rescaling of two running states, written for normalised partials.)
 * o_parts: [k][rows][d]; lse_parts: [k][rows].
 * ------------------------------------------------------------------------- */
void orc_lse_merge(int64_t rows, int d, int k, const double* o_parts,
                   const double* lse_parts, double* o, double* lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int c = 0; c < k; ++c)
            if (lse_parts[(int64_t)c * rows + r] > m)
                m = lse_parts[(int64_t)c * rows + r];
        double* orow = o + r * d;
        for (int x = 0; x < d; ++x)
            orow[x] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int c = 0; c < k; ++c)
            sum += exp(lse_parts[(int64_t)c * rows + r] - m);
        double L = m + log(sum);
        lse[r] = L;
        for (int c = 0; c < k; ++c) {
            double w = exp(lse_parts[(int64_t)c * rows + r] - L);
            const double* op = o_parts + ((int64_t)c * rows + r) * d;
            for (int x = 0; x < d; ++x)
                orow[x] += w * op[x];
        }
    }
}

/* ---------------------------------------------------------------------------
 * Causal pair counts between workers, by brute force over token pairs.
 *
 * counts[p*P + w] = #{(i, j) : i owned by worker p, j owned by worker w,
 *                             pos(j) <= pos(i)}.
 * At ring step s worker p holds the keys of worker (p - s) mod P (Striped
 * Attention Guide, "Workload Balance Theorem"; DistFlashAttn Guide, the ring
 * steps of "The Causal Imbalance Crisis"), so its step-s load is
 * counts[p*P + (p - s) mod P].
 * ------------------------------------------------------------------------- */
int orc_pair_counts(int kind, int64_t N, int P, int stripe, int64_t* counts)
{
    int64_t n = N / P;
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)N);
    for (int p = 0; p < P; ++p)
        if (orc_partition_fill(kind, N, P, stripe, p, pos + (int64_t)p * n) != 0) {
            free(pos);
            return -1;
        }
    for (int p = 0; p < P; ++p)
        for (int w = 0; w < P; ++w) {
            int64_t c = 0;
            const int64_t* pq = pos + (int64_t)p * n;
            const int64_t* pk = pos + (int64_t)w * n;
            for (int64_t i = 0; i < n; ++i)
                for (int64_t j = 0; j < n; ++j)
                    if (pk[j] <= pq[i])
                        ++c;
            counts[p * P + w] = c;
        }
    free(pos);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Tile classification of one chunk pair, by brute force over token pairs.
 *
 * Query rows of worker p are cut into tiles of tm rows, key rows of worker w
 * into tiles of tn rows (the last tile of each may be short).  For every tile
 * pair: 0 = skip (no visible pair), 1 = full (every pair visible), 2 = partial
 * (an element mask is needed) -- Striped Attention Guide, "Intra-Block vs.
 * Inter-Block Masking Logic".  cls[qt * nkt + kt].
 * ------------------------------------------------------------------------- */
int orc_tile_classes(int kind, int64_t N, int P, int stripe, int p, int w,
                     int tm, int tn, int8_t* cls)
{
    int64_t n = N / P;
    int64_t* pq = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
    int64_t* pk = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
    if (orc_partition_fill(kind, N, P, stripe, p, pq) ||
        orc_partition_fill(kind, N, P, stripe, w, pk)) {
        free(pq);
        free(pk);
        return -1;
    }
    int64_t nqt = (n + tm - 1) / tm, nkt = (n + tn - 1) / tn;
    for (int64_t qt = 0; qt < nqt; ++qt)
        for (int64_t kt = 0; kt < nkt; ++kt) {
            int64_t vis = 0, tot = 0;
            for (int64_t i = qt * tm; i < n && i < (qt + 1) * tm; ++i)
                for (int64_t j = kt * tn; j < n && j < (kt + 1) * tn; ++j) {
                    ++tot;
                    if (pk[j] <= pq[i])
                        ++vis;
                }
            cls[qt * nkt + kt] = (int8_t)(vis == 0 ? 0 : (vis == tot ? 1 : 2));
        }
    free(pq);
    free(pk);
    return 0;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
