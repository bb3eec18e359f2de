/*
 * attention_oracle.c -- plain, slow, fp64 CPU reference for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. The CUDA library never links, loads or calls this file. Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg use it. It shares no code,
 * header, helper, table or constant with the CUDA kernels.
 *
 * What it computes is the plain definition of attention, written out term by term:
 *
 *   s_ij  = scale * <q_i, k_j>                     for allowed pairs (i, j)
 *   m_i   = max_j s_ij,   l_i = sum_j exp(s_ij - m_i)
 *   P_ij  = exp(s_ij - m_i) / l_i                  (0 for masked pairs)
 *   O_i   = sum_j P_ij v_j,   LSE_i = m_i + ln l_i  (natural log)
 *   dP_ij = <dO_i, v_j>,  D_i = <dO_i, O_i>,  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_{query heads of the group} sum_i dS_ij q_i
 *   dV_j  = sum_{query heads of the group} sum_i P_ij dO_i
 *
 * Sources (page title, section, formula):
 *  - Forward: "Attention's hidden recurrence: an introduction to Flash Attention" (mzeromiko blog),
 *    section "standard attention / forward": O = Diag((exp(QK^T) (.) M) 1)^-1 (exp(QK^T) (.) M) V.
 *    Subtracting the row maximum before exp (the stability shift) is from the same page, section
 *    "blocked form with online-softmax rescaling", and from the FlashAttention note
 *    (paweldubiel.com), section "averaging block results is not enough" (state m, l, u; result u/l).
 *  - Mask: FlashAttention DAC'24 reading note (paper.adslab.icu), section "other operators": the
 *    mask acts on each block of QK^T; mzeromiko blog, "blocked recurrence": M is causal or none.
 *    Masked pairs carry weight exactly 0 (M multiplies exp(S) by 0), i.e. -inf before softmax.
 *  - Backward: mzeromiko blog, section "standard attention / backward":
 *    d(exp(QK^T) (.) M) = Diag(E 1)^-1 (dO V^T - diag(dO O^T) 1^T),  dV = E^T Diag(E 1)^-1 dO,
 *    dQ = (dE (.) E) K,  dK = (dE (.) E)^T Q  with E = exp(QK^T) (.) M.  Since dE (.) E equals
 *    P (.) (dP - D 1^T), that is dS above; diag(dO O^T) is D.  The factor `scale` on dQ and dK is
 *    the chain rule through s = scale * q.k (the pages use scale = 1).
 *  - GQA: FlashAttention note (paweldubiel.com), last section: grouped-query attention combines
 *    with the method.  Query head hq reads key/value head hq / (Hq / Hkv) (consecutive groups).
 *
 *  - General masks (the *_masked entry points): the same rule, "the mask acts on each block of
 *    QK^T" (reading note, "other operators"), with the allowed set of a pair (i, j) of head
 *    (b, hq) being the AND of: the causal rule; i < q_len[b] and j < k_len[b] (per-batch valid
 *    lengths of a padded batch, clamped to [0, N]); and block_mask[h][i / block][j / block] != 0
 *    for a 0/1 mask over block x block tiles, h = 0, hq or b * Hq + hq when the mask holds 1,
 *    Hq or B * Hq heads.  A row with no allowed key (every row i >= q_len[b], or one whose tiles
 *    are all masked) gets O = 0 and LSE = -inf, and passes no gradient.
 *
 *  - Dropout (the *_dropout entry points): the reading note ("other operators") lists dropout
 *    among the operations fused per block.  Read as inverted dropout on the normalised P:
 *    P~_ij = P_ij Z_ij / (1 - p) with Z_ij in {0, 1}, O = P~ V; LSE is that of the undropped
 *    P.  Z_ij = 1 ("keep") iff word (j mod 4) of Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
 *    "Parallel random numbers: as easy as 1, 2, 3", SC'11) at counter (j / 4, i, b * Hq + hq,
 *    offset) and key (seed mod 2^32, seed / 2^32) is below floor((1 - p) 2^32).  The backward
 *    follows by the chain rule: dV = P~^T dO, dP~ = dO V^T, dS = P (.) (Z / (1 - p) (.) dP~ - D)
 *    with D_i = <dO_i, O_i> of the dropped O (since sum_j P_ij Z_ij / (1 - p) <dO_i, v_j> =
 *    <dO_i, O_i>), dQ = scale dS K, dK = scale dS^T Q.
 *
 * Layout: every tensor is contiguous [B, H, N, d] fp64 (d fastest); K, V, dK, dV use H = Hkv.
 * LSE is [B, Hq, N].  Causal means key j <= query i (top-left aligned, Nq = Nk = N).
 *
 * Parallelism: OpenMP over independent rows (or key columns); no blocking or reordering of the
 * sums beyond what the definition states.  Every function returns 0 on success, nonzero on
 * invalid arguments or allocation failure.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

/* Which (query i, key j) pairs are allowed; see the header.  NULL members mean "no limit". */
typedef struct {
    int causal;
    const int *q_len, *k_len;          /* [B] */
    const unsigned char *block_mask;   /* [mask_heads, nb, nb] */
    int mask_heads, block, nb;
    int B, Hq, N;
} mask_t;

static mask_t causal_only(int causal, int B, int Hq, int N) {
    mask_t m = {causal, NULL, NULL, NULL, 0, 1, 1, B, Hq, N};
    return m;
}

static i64 clamp_len(int len, int N) { return len < 0 ? 0 : (len > N ? N : len); }

static int allowed(const mask_t *M, i64 b, i64 hq, i64 i, i64 j) {
    if (M->causal && j > i) return 0;
    if (M->q_len && i >= clamp_len(M->q_len[b], M->N)) return 0;
    if (M->k_len && j >= clamp_len(M->k_len[b], M->N)) return 0;
    if (M->block_mask) {
        const i64 h = M->mask_heads == 1 ? 0
                    : (M->mask_heads == M->B * M->Hq ? b * M->Hq + hq : hq);
        if (!M->block_mask[(h * M->nb + i / M->block) * M->nb + j / M->block]) return 0;
    }
    return 1;
}

/* Builds the general mask; returns nonzero for an invalid mask description. */
static int make_mask(mask_t *M, int causal, int B, int Hq, int N, const int *q_len,
                     const int *k_len, const unsigned char *block_mask, int mask_heads, int block) {
    *M = causal_only(causal, B, Hq, N);
    M->q_len = q_len;
    M->k_len = k_len;
    if (block_mask) {
        if (block < 1) return 1;
        if (mask_heads != 1 && mask_heads != Hq && mask_heads != B * Hq) return 1;
        M->block_mask = block_mask;
        M->mask_heads = mask_heads;
        M->block = block;
        M->nb = (N + block - 1) / block;
    }
    return 0;
}

static double dot(const double *a, const double *b, int d) {
    double acc = 0.0;
    for (int k = 0; k < d; ++k) acc += a[k] * b[k];
    return acc;
}

static int check_shape(int B, int Hq, int Hkv, int N, int d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return 1;
    if (Hq % Hkv != 0) return 1;
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * One query row of one head: fills s_row[0..N) with the scores (-INFINITY where masked), turns it
 * into the probability row in place, writes o_row[0..d) and returns LSE_i.
 */
static double softmax_row(const mask_t *M, i64 b, i64 hq, const double *qi, const double *k,
                          const double *v, i64 i, int N, int d, double scale, double *p_row,
                          double *o_row) {
    double m = -INFINITY;
    for (i64 j = 0; j < N; ++j) {
        if (allowed(M, b, hq, i, j)) {
            p_row[j] = scale * dot(qi, k + j * d, d);
            if (p_row[j] > m) m = p_row[j];
        } else {
            p_row[j] = -INFINITY;
        }
    }
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    if (m == -INFINITY) {               /* no allowed key: O = 0, LSE = -inf */
        for (i64 j = 0; j < N; ++j) p_row[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (i64 j = 0; j < N; ++j) {
        double e = allowed(M, b, hq, i, j) ? exp(p_row[j] - m) : 0.0;
        p_row[j] = e;
        l += e;
    }
    for (i64 j = 0; j < N; ++j) {
        p_row[j] /= l;
        if (p_row[j] != 0.0) {
            const double *vj = v + j * d;
            for (int c = 0; c < d; ++c) o_row[c] += p_row[j] * vj[c];
        }
    }
    return m + log(l);
}

/*
 * Forward over a list of heads, materialising S and P (N x N) for each head.
 *   heads[h] = b * Hq + hq.  O_out is [nheads, N, d], LSE_out is [nheads, N].
 *   P_out (optional, may be NULL) receives the probability matrices [nheads, N, N].
 */
static int forward_impl(const mask_t *M, int B, int Hq, int Hkv, int N, int d, double scale,
                        const double *Q, const double *K, const double *V, int nheads,
                        const int *heads, double *O_out, double *LSE_out, double *P_out) {
    if (check_shape(B, Hq, Hkv, N, d) || nheads < 0) return 1;
    const int G = Hq / Hkv;
    const i64 nn = (i64)N * N, nd = (i64)N * d;
    double *P = P_out ? NULL : (double *)malloc(sizeof(double) * nn);
    if (!P_out && !P) return 2;
    for (int h = 0; h < nheads; ++h) {
        const int bh = heads[h];
        if (bh < 0 || bh >= B * Hq) { free(P); return 1; }
        const int b = bh / Hq, hq = bh % Hq, hk = hq / G;
        const double *q = Q + (i64)bh * nd;
        const double *k = K + ((i64)b * Hkv + hk) * nd;
        const double *v = V + ((i64)b * Hkv + hk) * nd;
        double *Ph = P_out ? P_out + (i64)h * nn : P;
#pragma omp parallel for schedule(dynamic, 16)
        for (i64 i = 0; i < N; ++i)
            LSE_out[(i64)h * N + i] = softmax_row(M, b, hq, q + i * d, k, v, i, N, d, scale,
                                                  Ph + i * N, O_out + (i64)h * nd + i * d);
    }
    free(P);
    return 0;
}

int oracle_attention_forward(int B, int Hq, int Hkv, int N, int d, int causal, double scale,
                             const double *Q, const double *K, const double *V, int nheads,
                             const int *heads, double *O_out, double *LSE_out, double *P_out) {
    const mask_t M = causal_only(causal, B, Hq, N);
    return forward_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, nheads, heads, O_out, LSE_out, P_out);
}

/* oracle_attention_forward under the general mask (see the header). */
int oracle_attention_forward_masked(int B, int Hq, int Hkv, int N, int d, int causal,
                                    const int *q_len, const int *k_len,
                                    const unsigned char *block_mask, int mask_heads, int block,
                                    double scale, const double *Q, const double *K,
                                    const double *V, int nheads, const int *heads, double *O_out,
                                    double *LSE_out) {
    mask_t M;
    if (check_shape(B, Hq, Hkv, N, d) ||
        make_mask(&M, causal, B, Hq, N, q_len, k_len, block_mask, mask_heads, block))
        return 1;
    return forward_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, nheads, heads, O_out, LSE_out, NULL);
}

/*
 * Forward restricted to the keys key_begin <= j < key_end (on top of the causal mask), over a
 * list of heads, materialising one score/probability row at a time: the partial result one key
 * range contributes (split-KV).  A row with no allowed key in the range gets O = 0 and
 * LSE = -inf.  O_out is [nheads, N, d], LSE_out [nheads, N].
 */
int oracle_attention_forward_keys(int B, int Hq, int Hkv, int N, int d, int causal, double scale,
                                  const double *Q, const double *K, const double *V, int key_begin,
                                  int key_end, int nheads, const int *heads, double *O_out,
                                  double *LSE_out) {
    if (check_shape(B, Hq, Hkv, N, d) || nheads < 0) return 1;
    if (key_begin < 0 || key_end > N || key_begin > key_end) return 1;
    const int G = Hq / Hkv;
    const i64 nd = (i64)N * d;
    int bad = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * N);
#pragma omp for schedule(dynamic, 16) collapse(2)
        for (int h = 0; h < nheads; ++h)
            for (i64 i = 0; i < N; ++i) {
                const int bh = heads[h];
                if (!p || bh < 0 || bh >= B * Hq) { bad = 1; continue; }
                const int b = bh / Hq, hk = (bh % Hq) / G;
                const double *q = Q + (i64)bh * nd + i * d;
                const double *k = K + ((i64)b * Hkv + hk) * nd, *v = V + ((i64)b * Hkv + hk) * nd;
                double *o = O_out + (i64)h * nd + i * d;
                double m = -INFINITY;
                for (i64 j = 0; j < N; ++j) {
                    const int ok = (!causal || j <= i) && j >= key_begin && j < key_end;
                    p[j] = ok ? scale * dot(q, k + j * d, d) : -INFINITY;
                    if (p[j] > m) m = p[j];
                }
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                if (m == -INFINITY) { LSE_out[(i64)h * N + i] = -INFINITY; continue; }
                double l = 0.0;
                for (i64 j = 0; j < N; ++j) {
                    p[j] = (p[j] == -INFINITY) ? 0.0 : exp(p[j] - m);
                    l += p[j];
                }
                for (i64 j = 0; j < N; ++j)
                    if (p[j] != 0.0)
                        for (int c = 0; c < d; ++c) o[c] += p[j] / l * v[j * d + c];
                LSE_out[(i64)h * N + i] = m + log(l);
            }
        free(p);
    }
    return bad;
}

/*
 * Merge of S partial results over disjoint key sets, in the form of the reading note's update
 * (FlashAttention DAC'24 reading note, Methods): with the running state (m, l, O), each new part
 * with its own normalised output O~ and log-sum-exp L~ = m~ + ln l~ updates
 *   m' = max(m, L~),  l' = e^{m - m'} l + e^{L~ - m'},  O' = (e^{m - m'} l O + e^{L~ - m'} O~) / l'
 * (a part is a block whose l~ is folded into its LSE); the result is O and LSE = m + ln l.
 * Parts with LSE = -inf (no allowed key) contribute nothing.  O_parts is [S, rows, d] and
 * LSE_parts [S, rows]; O_out [rows, d], LSE_out [rows].
 */
int oracle_merge_partials(int S, i64 rows, int d, const double *O_parts, const double *LSE_parts,
                          double *O_out, double *LSE_out) {
    if (S < 1 || rows < 0 || d < 1) return 1;
#pragma omp parallel for schedule(static)
    for (i64 r = 0; r < rows; ++r) {
        double m = -INFINITY, l = 0.0;
        double *o = O_out + r * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int s = 0; s < S; ++s) {
            const double Ls = LSE_parts[(i64)s * rows + r];
            if (Ls == -INFINITY) continue;
            const double *os = O_parts + ((i64)s * rows + r) * d;
            const double mn = m > Ls ? m : Ls;
            const double a = (m == -INFINITY) ? 0.0 : exp(m - mn) * l;   /* old weight */
            const double bw = exp(Ls - mn);                               /* new part's weight */
            const double ln = a + bw;
            for (int c = 0; c < d; ++c) o[c] = (a * o[c] + bw * os[c]) / ln;
            m = mn;
            l = ln;
        }
        LSE_out[r] = (l == 0.0) ? -INFINITY : m + log(l);
    }
    return 0;
}

/*
 * Backward over a list of KV groups, materialising P and dS (N x N) for each query head.
 *   groups[g] = b * Hkv + hk.  dQ_out is [ngroups, G, N, d] (the group's query heads in order),
 *   dK_out and dV_out are [ngroups, N, d].  O and D come from the oracle's own fp64 forward.
 */
static int backward_impl(const mask_t *M, int B, int Hq, int Hkv, int N, int d, double scale,
                         const double *Q, const double *K, const double *V, const double *dO,
                         int ngroups, const int *groups, double *dQ_out, double *dK_out,
                         double *dV_out) {
    if (check_shape(B, Hq, Hkv, N, d) || ngroups < 0) return 1;
    const int G = Hq / Hkv;
    const i64 nn = (i64)N * N, nd = (i64)N * d;
    double *P = (double *)malloc(sizeof(double) * nn);
    double *O = (double *)malloc(sizeof(double) * nd);
    double *D = (double *)malloc(sizeof(double) * N);
    if (!P || !O || !D) { free(P); free(O); free(D); return 2; }
    for (int g = 0; g < ngroups; ++g) {
        const int bk = groups[g];
        if (bk < 0 || bk >= B * Hkv) { free(P); free(O); free(D); return 1; }
        const int b = bk / Hkv, hk = bk % Hkv;
        const double *k = K + (i64)bk * nd, *v = V + (i64)bk * nd;
        double *dk = dK_out + (i64)g * nd, *dv = dV_out + (i64)g * nd;
        memset(dk, 0, sizeof(double) * nd);
        memset(dv, 0, sizeof(double) * nd);
        for (int r = 0; r < G; ++r) {
            const int hq = hk * G + r;
            const double *q = Q + ((i64)b * Hq + hq) * nd;
            const double *dor = dO + ((i64)b * Hq + hq) * nd;
            double *dq = dQ_out + ((i64)g * G + r) * nd;
            /* forward: P, O, then D_i = <dO_i, O_i> */
#pragma omp parallel for schedule(dynamic, 16)
            for (i64 i = 0; i < N; ++i) {
                softmax_row(M, b, hq, q + i * d, k, v, i, N, d, scale, P + i * N, O + i * d);
                D[i] = dot(dor + i * d, O + i * d, d);
            }
            /* dV_j += sum_i P_ij dO_i  (parallel over key columns j) */
#pragma omp parallel for schedule(dynamic, 16)
            for (i64 j = 0; j < N; ++j)
                for (i64 i = 0; i < N; ++i) {
                    const double p = P[i * N + j];
                    if (p != 0.0)
                        for (int c = 0; c < d; ++c) dv[j * d + c] += p * dor[i * d + c];
                }
            /* dS_ij = P_ij (<dO_i, v_j> - D_i), in place over P; dQ_i = scale sum_j dS_ij k_j */
#pragma omp parallel for schedule(dynamic, 16)
            for (i64 i = 0; i < N; ++i) {
                double *row = P + i * N;
                for (int c = 0; c < d; ++c) dq[i * d + c] = 0.0;
                for (i64 j = 0; j < N; ++j) {
                    if (row[j] == 0.0) continue;
                    row[j] = row[j] * (dot(dor + i * d, v + j * d, d) - D[i]);
                    for (int c = 0; c < d; ++c) dq[i * d + c] += row[j] * k[j * d + c];
                }
                for (int c = 0; c < d; ++c) dq[i * d + c] *= scale;
            }
            /* dK_j += scale sum_i dS_ij q_i  (parallel over key columns j) */
#pragma omp parallel for schedule(dynamic, 16)
            for (i64 j = 0; j < N; ++j) {
                for (i64 i = 0; i < N; ++i) {
                    const double ds = P[i * N + j];
                    if (ds != 0.0)
                        for (int c = 0; c < d; ++c) dk[j * d + c] += scale * ds * q[i * d + c];
                }
            }
        }
    }
    free(P); free(O); free(D);
    return 0;
}

int oracle_attention_backward(int B, int Hq, int Hkv, int N, int d, int causal, double scale,
                              const double *Q, const double *K, const double *V, const double *dO,
                              int ngroups, const int *groups, double *dQ_out, double *dK_out,
                              double *dV_out) {
    const mask_t M = causal_only(causal, B, Hq, N);
    return backward_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, dO, ngroups, groups, dQ_out,
                         dK_out, dV_out);
}

/* oracle_attention_backward under the general mask (see the header). */
int oracle_attention_backward_masked(int B, int Hq, int Hkv, int N, int d, int causal,
                                     const int *q_len, const int *k_len,
                                     const unsigned char *block_mask, int mask_heads, int block,
                                     double scale, const double *Q, const double *K,
                                     const double *V, const double *dO, int ngroups,
                                     const int *groups, double *dQ_out, double *dK_out,
                                     double *dV_out) {
    mask_t M;
    if (check_shape(B, Hq, Hkv, N, d) ||
        make_mask(&M, causal, B, Hq, N, q_len, k_len, block_mask, mask_heads, block))
        return 1;
    return backward_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, dO, ngroups, groups, dQ_out,
                         dK_out, dV_out);
}

/*
 * Sampled forward rows: rows[r] = (b * Hq + hq) * N + i.  O_rows is [nrows, d], LSE_rows [nrows].
 * Each row materialises its own score/probability row; cost O(N d) per row.
 */
static int forward_rows_impl(const mask_t *M, int B, int Hq, int Hkv, int N, int d, double scale,
                             const double *Q, const double *K, const double *V, int nrows,
                             const i64 *rows, double *O_rows, double *LSE_rows) {
    if (check_shape(B, Hq, Hkv, N, d) || nrows < 0) return 1;
    const int G = Hq / Hkv;
    const i64 nd = (i64)N * d;
    int bad = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * N);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            const i64 idx = rows[r];
            if (!p || idx < 0 || idx >= (i64)B * Hq * N) { bad = 1; continue; }
            const i64 bh = idx / N, i = idx % N;
            const i64 b = bh / Hq, hq = bh % Hq, hk = hq / G;
            const double *k = K + (b * Hkv + hk) * nd, *v = V + (b * Hkv + hk) * nd;
            LSE_rows[r] = softmax_row(M, b, hq, Q + bh * nd + i * d, k, v, i, N, d, scale, p,
                                      O_rows + (i64)r * d);
        }
        free(p);
    }
    return bad;
}

int oracle_forward_rows(int B, int Hq, int Hkv, int N, int d, int causal, double scale,
                        const double *Q, const double *K, const double *V, int nrows,
                        const i64 *rows, double *O_rows, double *LSE_rows) {
    const mask_t M = causal_only(causal, B, Hq, N);
    return forward_rows_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, nrows, rows, O_rows, LSE_rows);
}

int oracle_forward_rows_masked(int B, int Hq, int Hkv, int N, int d, int causal, const int *q_len,
                               const int *k_len, const unsigned char *block_mask, int mask_heads,
                               int block, double scale, const double *Q, const double *K,
                               const double *V, int nrows, const i64 *rows, double *O_rows,
                               double *LSE_rows) {
    mask_t M;
    if (check_shape(B, Hq, Hkv, N, d) ||
        make_mask(&M, causal, B, Hq, N, q_len, k_len, block_mask, mask_heads, block))
        return 1;
    return forward_rows_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, nrows, rows, O_rows, LSE_rows);
}

/* Sampled dQ rows (same row encoding as oracle_forward_rows). dQ_rows is [nrows, d]. */
static int dq_rows_impl(const mask_t *M, int B, int Hq, int Hkv, int N, int d, double scale,
                        const double *Q, const double *K, const double *V, const double *dO,
                        int nrows, const i64 *rows, double *dQ_rows) {
    if (check_shape(B, Hq, Hkv, N, d) || nrows < 0) return 1;
    const int G = Hq / Hkv;
    const i64 nd = (i64)N * d;
    int bad = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * N);
        double *o = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            const i64 idx = rows[r];
            if (!p || !o || idx < 0 || idx >= (i64)B * Hq * N) { bad = 1; continue; }
            const i64 bh = idx / N, i = idx % N;
            const i64 b = bh / Hq, hq = bh % Hq, hk = hq / G;
            const double *k = K + (b * Hkv + hk) * nd, *v = V + (b * Hkv + hk) * nd;
            const double *doi = dO + bh * nd + i * d;
            softmax_row(M, b, hq, Q + bh * nd + i * d, k, v, i, N, d, scale, p, o);
            const double Di = dot(doi, o, d);
            double *dq = dQ_rows + (i64)r * d;
            for (int c = 0; c < d; ++c) dq[c] = 0.0;
            for (i64 j = 0; j < N; ++j) {
                if (p[j] == 0.0) continue;
                const double ds = p[j] * (dot(doi, v + j * d, d) - Di);
                for (int c = 0; c < d; ++c) dq[c] += ds * k[j * d + c];
            }
            for (int c = 0; c < d; ++c) dq[c] *= scale;
        }
        free(p); free(o);
    }
    return bad;
}

int oracle_backward_dq_rows(int B, int Hq, int Hkv, int N, int d, int causal, double scale,
                            const double *Q, const double *K, const double *V, const double *dO,
                            int nrows, const i64 *rows, double *dQ_rows) {
    const mask_t M = causal_only(causal, B, Hq, N);
    return dq_rows_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, dO, nrows, rows, dQ_rows);
}

int oracle_backward_dq_rows_masked(int B, int Hq, int Hkv, int N, int d, int causal,
                                   const int *q_len, const int *k_len,
                                   const unsigned char *block_mask, int mask_heads, int block,
                                   double scale, const double *Q, const double *K,
                                   const double *V, const double *dO, int nrows, const i64 *rows,
                                   double *dQ_rows) {
    mask_t M;
    if (check_shape(B, Hq, Hkv, N, d) ||
        make_mask(&M, causal, B, Hq, N, q_len, k_len, block_mask, mask_heads, block))
        return 1;
    return dq_rows_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, dO, nrows, rows, dQ_rows);
}

/*
 * Sampled dK / dV rows: cols[r] = (b * Hkv + hk) * N + j.  dK_rows and dV_rows are [ncols, d].
 * First a row pass computes LSE_i and D_i for every query row of each touched KV group (one
 * group at a time), then each key column recomputes P_ij = exp(s_ij - LSE_i) and dS_ij.
 */
static int dkv_cols_impl(const mask_t *M, int B, int Hq, int Hkv, int N, int d, double scale,
                         const double *Q, const double *K, const double *V, const double *dO,
                         int ncols, const i64 *cols, double *dK_rows, double *dV_rows) {
    if (check_shape(B, Hq, Hkv, N, d) || ncols < 0) return 1;
    const int G = Hq / Hkv;
    const i64 nd = (i64)N * d;
    for (int r = 0; r < ncols; ++r)
        if (cols[r] < 0 || cols[r] >= (i64)B * Hkv * N) return 1;
    double *LSE = (double *)malloc(sizeof(double) * (i64)G * N);
    double *D = (double *)malloc(sizeof(double) * (i64)G * N);
    char *done = (char *)calloc(ncols > 0 ? ncols : 1, 1);
    if (!LSE || !D || !done) { free(LSE); free(D); free(done); return 2; }
    int bad = 0;
    for (int r0 = 0; r0 < ncols; ++r0) {
        if (done[r0]) continue;
        const i64 bk = cols[r0] / N, b = bk / Hkv, hk = bk % Hkv;
        const double *k = K + bk * nd, *v = V + bk * nd;
        /* row pass over the group's query heads: LSE_i and D_i */
        for (int g = 0; g < G; ++g) {
            const i64 bh = b * Hq + hk * G + g;
#pragma omp parallel
            {
                double *p = (double *)malloc(sizeof(double) * N);
                double *o = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 16)
                for (i64 i = 0; i < N; ++i) {
                    if (!p || !o) { bad = 2; continue; }
                    LSE[(i64)g * N + i] = softmax_row(M, b, hk * G + g, Q + bh * nd + i * d, k, v,
                                                      i, N, d, scale, p, o);
                    D[(i64)g * N + i] = dot(dO + bh * nd + i * d, o, d);
                }
                free(p); free(o);
            }
        }
        /* column pass for every requested key of this group */
#pragma omp parallel for schedule(dynamic, 1)
        for (int r = r0; r < ncols; ++r) {
            if (cols[r] / N != bk) continue;
            done[r] = 1;
            const i64 j = cols[r] % N;
            double *dk = dK_rows + (i64)r * d, *dv = dV_rows + (i64)r * d;
            for (int c = 0; c < d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
            for (int g = 0; g < G; ++g) {
                const i64 bh = b * Hq + hk * G + g;
                const double *q = Q + bh * nd, *dor = dO + bh * nd;
                for (i64 i = 0; i < N; ++i) {
                    if (!allowed(M, b, hk * G + g, i, j)) continue;
                    const double lse = LSE[(i64)g * N + i];
                    if (lse == -INFINITY) continue;
                    const double pij = exp(scale * dot(q + i * d, k + j * d, d) - lse);
                    const double dsij = pij * (dot(dor + i * d, v + j * d, d) - D[(i64)g * N + i]);
                    for (int c = 0; c < d; ++c) {
                        dv[c] += pij * dor[i * d + c];
                        dk[c] += scale * dsij * q[i * d + c];
                    }
                }
            }
        }
    }
    free(LSE); free(D); free(done);
    return bad;
}

int oracle_backward_dkv_cols(int B, int Hq, int Hkv, int N, int d, int causal, double scale,
                             const double *Q, const double *K, const double *V, const double *dO,
                             int ncols, const i64 *cols, double *dK_rows, double *dV_rows) {
    const mask_t M = causal_only(causal, B, Hq, N);
    return dkv_cols_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, dO, ncols, cols, dK_rows, dV_rows);
}

int oracle_backward_dkv_cols_masked(int B, int Hq, int Hkv, int N, int d, int causal,
                                    const int *q_len, const int *k_len,
                                    const unsigned char *block_mask, int mask_heads, int block,
                                    double scale, const double *Q, const double *K,
                                    const double *V, const double *dO, int ncols, const i64 *cols,
                                    double *dK_rows, double *dV_rows) {
    mask_t M;
    if (check_shape(B, Hq, Hkv, N, d) ||
        make_mask(&M, causal, B, Hq, N, q_len, k_len, block_mask, mask_heads, block))
        return 1;
    return dkv_cols_impl(&M, B, Hq, Hkv, N, d, scale, Q, K, V, dO, ncols, cols, dK_rows, dV_rows);
}

/* ------------------------------------------------------------------------------- dropout */

/*
 * Philox4x32-10 (Salmon et al., SC'11): ten rounds; each multiplies words 0 and 2 by the two
 * round multipliers into 64-bit products, and the new state is
 *   (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)),
 * after which the key is bumped by the two Weyl increments.
 */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint64_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = M0 * (uint64_t)x0, p1 = M1 * (uint64_t)x2;
        const uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
        const uint32_t y1 = (uint32_t)p1;
        const uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
        const uint32_t y3 = (uint32_t)p0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* floor((1 - p) 2^32) for 0 < p < 1 (0 for an invalid p). */
uint32_t oracle_dropout_threshold(double p) {
    if (!(p > 0.0) || !(p < 1.0)) return 0;
    const double t = floor((1.0 - p) * 4294967296.0);
    return t >= 4294967295.0 ? 4294967295u : (uint32_t)t;
}

static int dropout_keep(uint64_t seed, uint32_t offset, uint32_t thresh, i64 bh, i64 i, i64 j) {
    const uint32_t ctr[4] = {(uint32_t)(j >> 2), (uint32_t)i, (uint32_t)bh, offset};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    oracle_philox4x32_10(ctr, key, r);
    return r[j & 3] < thresh;
}

/* The keep decisions Z [BH, N, N] (1 = keep) of every (head, query, key). */
int oracle_dropout_mask(int BH, int N, uint64_t seed, uint32_t offset, double p,
                        unsigned char *Z_out) {
    if (BH < 1 || N < 1) return 1;
    const uint32_t thresh = oracle_dropout_threshold(p);
    if (thresh == 0) return 1;
#pragma omp parallel for schedule(static) collapse(2)
    for (i64 bh = 0; bh < BH; ++bh)
        for (i64 i = 0; i < N; ++i)
            for (i64 j = 0; j < N; ++j)
                Z_out[(bh * N + i) * N + j] = (unsigned char)dropout_keep(seed, offset, thresh, bh, i, j);
    return 0;
}

/* Forward with dropout on every head: O [B, Hq, N, d] = P~ V, LSE [B, Hq, N] of the undropped P. */
int oracle_attention_forward_dropout(int B, int Hq, int Hkv, int N, int d, int causal,
                                     double scale, double p, uint64_t seed, uint32_t offset,
                                     const double *Q, const double *K, const double *V,
                                     double *O_out, double *LSE_out) {
    if (check_shape(B, Hq, Hkv, N, d)) return 1;
    const uint32_t thresh = oracle_dropout_threshold(p);
    if (thresh == 0) return 1;
    const int G = Hq / Hkv;
    const i64 nd = (i64)N * d;
    const mask_t M = causal_only(causal, B, Hq, N);
    int bad = 0;
#pragma omp parallel
    {
        double *prow = (double *)malloc(sizeof(double) * N);
        double *ofull = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 16) collapse(2)
        for (i64 bh = 0; bh < (i64)B * Hq; ++bh)
            for (i64 i = 0; i < N; ++i) {
                if (!prow || !ofull) { bad = 2; continue; }
                const i64 b = bh / Hq, hq = bh % Hq, hk = hq / G;
                const double *k = K + (b * Hkv + hk) * nd, *v = V + (b * Hkv + hk) * nd;
                LSE_out[bh * N + i] = softmax_row(&M, b, hq, Q + bh * nd + i * d, k, v, i, N, d,
                                                  scale, prow, ofull);
                double *o = O_out + bh * nd + i * d;
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                for (i64 j = 0; j < N; ++j) {
                    if (prow[j] == 0.0 || !dropout_keep(seed, offset, thresh, bh, i, j)) continue;
                    const double w = prow[j] / (1.0 - p);
                    for (int c = 0; c < d; ++c) o[c] += w * v[j * d + c];
                }
            }
        free(prow); free(ofull);
    }
    return bad;
}

/* Backward with dropout on every KV group: dQ [B, Hq, N, d], dK and dV [B, Hkv, N, d]. */
int oracle_attention_backward_dropout(int B, int Hq, int Hkv, int N, int d, int causal,
                                      double scale, double p, uint64_t seed, uint32_t offset,
                                      const double *Q, const double *K, const double *V,
                                      const double *dO, double *dQ_out, double *dK_out,
                                      double *dV_out) {
    if (check_shape(B, Hq, Hkv, N, d)) return 1;
    const uint32_t thresh = oracle_dropout_threshold(p);
    if (thresh == 0) return 1;
    const int G = Hq / Hkv;
    const i64 nn = (i64)N * N, nd = (i64)N * d;
    const mask_t M = causal_only(causal, B, Hq, N);
    double *P = (double *)malloc(sizeof(double) * nn);     /* P, then dS */
    double *Mk = (double *)malloc(sizeof(double) * nn);    /* Z / (1 - p) */
    double *O = (double *)malloc(sizeof(double) * nd);
    double *D = (double *)malloc(sizeof(double) * N);
    if (!P || !Mk || !O || !D) { free(P); free(Mk); free(O); free(D); return 2; }
    for (i64 bk = 0; bk < (i64)B * Hkv; ++bk) {
        const i64 b = bk / Hkv, hk = bk % Hkv;
        const double *k = K + bk * nd, *v = V + bk * nd;
        double *dk = dK_out + bk * nd, *dv = dV_out + bk * nd;
        memset(dk, 0, sizeof(double) * nd);
        memset(dv, 0, sizeof(double) * nd);
        for (int r = 0; r < G; ++r) {
            const i64 hq = hk * G + r, bh = b * Hq + hq;
            const double *q = Q + bh * nd, *dor = dO + bh * nd;
            double *dq = dQ_out + bh * nd;
            /* forward: P, Z / (1 - p), the dropped O and D_i = <dO_i, O_i> */
#pragma omp parallel
            {
                double *ofull = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 16)
                for (i64 i = 0; i < N; ++i) {
                    softmax_row(&M, b, hq, q + i * d, k, v, i, N, d, scale, P + i * N,
                                ofull ? ofull : O + i * d);
                    double *o = O + i * d;
                    for (int c = 0; c < d; ++c) o[c] = 0.0;
                    for (i64 j = 0; j < N; ++j) {
                        Mk[i * N + j] = dropout_keep(seed, offset, thresh, bh, i, j) ? 1.0 / (1.0 - p) : 0.0;
                        const double w = P[i * N + j] * Mk[i * N + j];
                        if (w != 0.0)
                            for (int c = 0; c < d; ++c) o[c] += w * v[j * d + c];
                    }
                    D[i] = dot(dor + i * d, o, d);
                }
                free(ofull);
            }
            /* dV_j += sum_i P~_ij dO_i */
#pragma omp parallel for schedule(dynamic, 16)
            for (i64 j = 0; j < N; ++j)
                for (i64 i = 0; i < N; ++i) {
                    const double w = P[i * N + j] * Mk[i * N + j];
                    if (w != 0.0)
                        for (int c = 0; c < d; ++c) dv[j * d + c] += w * dor[i * d + c];
                }
            /* dS_ij = P_ij (Z_ij / (1 - p) <dO_i, v_j> - D_i), over P; dQ_i = scale sum_j dS_ij k_j */
#pragma omp parallel for schedule(dynamic, 16)
            for (i64 i = 0; i < N; ++i) {
                double *row = P + i * N;
                for (int c = 0; c < d; ++c) dq[i * d + c] = 0.0;
                for (i64 j = 0; j < N; ++j) {
                    if (row[j] == 0.0) continue;
                    row[j] = row[j] * (Mk[i * N + j] * dot(dor + i * d, v + j * d, d) - D[i]);
                    for (int c = 0; c < d; ++c) dq[i * d + c] += row[j] * k[j * d + c];
                }
                for (int c = 0; c < d; ++c) dq[i * d + c] *= scale;
            }
            /* dK_j += scale sum_i dS_ij q_i */
#pragma omp parallel for schedule(dynamic, 16)
            for (i64 j = 0; j < N; ++j)
                for (i64 i = 0; i < N; ++i) {
                    const double ds = P[i * N + j];
                    if (ds != 0.0)
                        for (int c = 0; c < d; ++c) dk[j * d + c] += scale * ds * q[i * d + c];
                }
        }
    }
    free(P); free(Mk); free(O); free(D);
    return 0;
}
