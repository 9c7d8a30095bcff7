/*
 * oracle.c -- the plain, slow, double-precision CPU oracle for block-sparse GQA
 * decode attention with learned block selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load the library built from this file.  The product (the CUDA
 * library under block_sparse_long_pool_gb300/csrc) never calls it, and the two
 * share no code, header, table or helper.
 *
 * Every routine is the plain definition of one step, written as loops in double
 * precision over the exact bf16 input values.  Sources (three web pages):
 *   [SparDA] "SparDA: sparse decoupled attention" reading notes,
 *            zhongzhuzhou.org/blog/2026-06-24 (Chinese).
 *   [SSV]    "SSV: sparse speculative verification" reading notes,
 *            zhongzhuzhou.org/blog/2026-07-01 (Chinese).
 *
 *   oracle_pool    [SparDA] background §3 eq.(4): a compressed key is the mean of
 *                  the keys it covers; here one mean per non-overlapping 64-token
 *                  block, over the tokens present (t < len).
 *   oracle_select  [SparDA] §4.1 eq.(6) and §4.2 Alg.1 step 2: score the Forecast
 *                  vector against every compressed key (one head per GQA group,
 *                  §4.3 eq.(9)), take the k best blocks outside the init and local
 *                  blocks, and return init ∪ local ∪ top-k in ascending order.
 *   oracle_select_heads  the InfLLM-V2 multi-head selector that [SparDA] §4.3 (eq.(8),
 *                  Figure 3) compares against: G query heads score, per-head softmax
 *                  over the blocks, summed over heads, then the same top-k.
 *   oracle_attn    [SparDA] §4.1 eq.(7): attention of each query head of the group
 *                  over the tokens of the selected blocks, with the 1/sqrt(d) scale
 *                  of [SSV] "NSA three-branch math" step 3.
 *   oracle_verify  [SSV] mechanism 1, mode A: every (query, head) attends over its
 *                  own block set I_q plus the sliding-window blocks; the group's
 *                  merged union is what a grouped kernel has to load.
 *   oracle_verify_shared  [SSV] mechanism 1, mode B: every query of a group attends
 *                  over the layout of the group's first query (plus the window).
 *   oracle_nsa     [SSV] "NSA three-branch math": compressed, selected and sliding-window
 *                  branches, each its own softmax, combined by per-head gates.
 *   oracle_pool_windows  eq.(4) with an overlapping kernel l and stride s (the pages'
 *                  inference setting l = 32, s = 16): the compressed rows of NSA's
 *                  compressed branch ([SSV] "NSA", branch 1).
 *   oracle_select_windows  NSA routing on those rows: each head's softmax over the
 *                  windows, summed over heads, max-pooled onto the 64-token blocks
 *                  ([SparDA] §4.4: scores on a finer grid are max-pooled onto the
 *                  coarse one), then the top-k of oracle_select.
 *   oracle_nsa_windows  oracle_nsa with the compressed branch over the windows.
 *   oracle_prefill_select  [SparDA] eq.(16): the Forecast selection of every prefill
 *                  position, each over the blocks it can see (causal).
 *   oracle_gather  [SparDA] §4.5: staging selected blocks is a plain copy.
 *
 * Readings where the pages are silent are stated at each routine.
 * Fixed sizes: head dimension D = 128, block size BLK = 64 tokens.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D 128
#define BLK 64

/* bf16 is the upper half of an IEEE-754 binary32: widen the bits, then the value. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of 64-token blocks that hold at least one of the first len tokens. */
static int blocks_of(long long len)
{
    return len <= 0 ? 0 : (int)((len + BLK - 1) / BLK);
}

/* Number of complete compression windows [s*j, s*j + l) within the first len tokens. */
static int windows_of(long long len, int l, int s)
{
    return len < l ? 0 : (int)((len - l) / s + 1);
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Pooling, [SparDA] eq.(4).  K is [n_pairs][pair_stride][D] bf16 bits, len[p] the
 * tokens present for pair p.  ktil is [n_pairs][n_blocks_cap][D]:
 *   ktil[p][j][d] = (1/n_j) * sum_{t = 64j}^{min(64j+64, len)-1} K[p][t][d],
 * n_j the number of those tokens.  Blocks with no token are written as zero.
 */
void oracle_pool(const uint16_t *K, long long pair_stride, int n_pairs,
                 const long long *len, int n_blocks_cap, double *ktil)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < n_pairs; ++p) {
        const uint16_t *Kp = K + (size_t)p * (size_t)pair_stride * D;
        double *out = ktil + (size_t)p * (size_t)n_blocks_cap * D;
        int nb = blocks_of(len[p]);
        for (int j = 0; j < n_blocks_cap; ++j) {
            double sum[D];
            long long n = 0;
            for (int d = 0; d < D; ++d)
                sum[d] = 0.0;
            if (j < nb) {
                long long end = (long long)(j + 1) * BLK;
                if (end > len[p])
                    end = len[p];
                for (long long t = (long long)j * BLK; t < end; ++t) {
                    for (int d = 0; d < D; ++d)
                        sum[d] += bf16_value(Kp[(size_t)t * D + d]);
                    ++n;
                }
            }
            for (int d = 0; d < D; ++d)
                out[(size_t)j * D + d] = n > 0 ? sum[d] / (double)n : 0.0;
        }
    }
}

/*
 * Overlapping compression, [SparDA] eq.(4) with kernel l and stride s ([SparDA] §4.4:
 * l = 32, s = 16 at inference) and [SSV] "NSA" branch 1 (compressed blocks of length
 * l, stride d).  X is [n_pairs][pair_stride][D] bf16 bits; out [n_pairs][n_rows_cap][D]:
 *   out[p][j][d] = (1/l) * sum_{t = s*j}^{s*j + l - 1} X[p][t][d],   j < W = floor((len - l)/s) + 1.
 * Reading: only complete windows are rows (a window is compressed once its last token
 * is present; the most recent tokens are the sliding window's); rows j >= W are zero.
 * Returns -1 when some pair has more than n_rows_cap windows (its rows are clipped).
 */
int oracle_pool_windows(const uint16_t *X, long long pair_stride, int n_pairs, const long long *len, int l, int s,
                        int n_rows_cap, double *out)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int p = 0; p < n_pairs; ++p) {
        const uint16_t *Xp = X + (size_t)p * (size_t)pair_stride * D;
        double *o = out + (size_t)p * (size_t)n_rows_cap * D;
        int W = windows_of(len[p], l, s);
        if (W > n_rows_cap) {
            bad |= 1;
            W = n_rows_cap;
        }
        for (int j = 0; j < n_rows_cap; ++j) {
            double sum[D];
            for (int d = 0; d < D; ++d)
                sum[d] = 0.0;
            if (j < W)
                for (long long t = (long long)s * j; t < (long long)s * j + l; ++t)
                    for (int d = 0; d < D; ++d)
                        sum[d] += bf16_value(Xp[(size_t)t * D + d]);
            for (int d = 0; d < D; ++d)
                o[(size_t)j * D + d] = j < W ? sum[d] / (double)l : 0.0;
        }
    }
    return bad ? -1 : 0;
}

typedef struct {
    double s;
    int j;
} cand_t;

/* Descending score; equal scores keep the lower block index first. */
static int cand_order(const void *a, const void *b)
{
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->s > y->s)
        return -1;
    if (x->s < y->s)
        return 1;
    return (x->j > y->j) - (x->j < y->j);
}

/*
 * Selection, [SparDA] eq.(6) + Alg.1 step 2.
 *   F     [n_pairs][D]  bf16 bits: one Forecast vector per (batch, KV head).
 *   ktil  [n_pairs][n_blocks_cap][D] compressed keys of the layer being selected for.
 *   len   tokens present per pair; N_b = ceil(len / 64).
 * B_init  = blocks [0, n_init); B_local = the last n_local blocks [N_b-n_local, N_b)
 * (the block holding token len-1 and the ones before it).  Candidates are all other
 * blocks; s_j = sum_d F[d] * ktil[j][d]; the k candidates of largest score are taken,
 * a full sort deciding ties towards the lower index (Alg.1 step 2 excludes init and
 * local from the top-k, so the union has min(N_b, n_init+n_local+k) distinct blocks).
 * Output idx[p][0..count) ascending, padded with -1 up to k_tot.  scores (nullable)
 * receives s_j for every block j < N_b (the rest zero).
 * Returns 0, or -1 when a pair needs more than k_tot or n_blocks_cap entries.
 */
/*
 * The selection of one pair from its block scores s[0 .. nb): B_init = [0, n_init),
 * B_local = [nb - n_local, nb), and the k candidates (all other blocks) of largest
 * score, a full sort deciding ties towards the lower index; idx[0 .. count) ascending,
 * padded with -1 up to k_tot.  Returns 1 when the union needs more than k_tot entries.
 */
static int select_from_scores(const double *s, int nb, int n_init, int n_local, int k, int k_tot, int *out,
                              int *count)
{
    char *chosen = (char *)calloc((size_t)nb + 1, 1);
    cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * ((size_t)nb + 1));
    for (int j = 0; j < nb && j < n_init; ++j)
        chosen[j] = 1;
    for (int j = nb - n_local; j < nb; ++j)
        if (j >= 0)
            chosen[j] = 1;
    int nc = 0;
    for (int j = 0; j < nb; ++j) {
        if (!chosen[j]) {
            cand[nc].s = s[j];
            cand[nc].j = j;
            ++nc;
        }
    }
    qsort(cand, (size_t)nc, sizeof(cand_t), cand_order);
    for (int r = 0; r < nc && r < k; ++r)
        chosen[cand[r].j] = 1;
    int c = 0, bad = 0;
    for (int j = 0; j < nb; ++j) {
        if (!chosen[j])
            continue;
        if (c < k_tot)
            out[c] = j;
        ++c;
    }
    if (c > k_tot) {
        bad = 1;
        c = k_tot;
    }
    *count = c;
    for (int r = c; r < k_tot; ++r)
        out[r] = -1;
    free(cand);
    free(chosen);
    return bad;
}

int oracle_select(const uint16_t *F, const double *ktil, int n_blocks_cap, int n_pairs,
                  const long long *len, int n_init, int n_local, int k, int k_tot,
                  int *idx, int *count, double *scores)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int p = 0; p < n_pairs; ++p) {
        int nb = blocks_of(len[p]);
        int *out = idx + (size_t)p * k_tot;
        if (nb > n_blocks_cap) {
            bad |= 1;
            count[p] = 0;
            continue;
        }
        double Fp[D];
        for (int d = 0; d < D; ++d)
            Fp[d] = bf16_value(F[(size_t)p * D + d]);
        double *s = (double *)malloc(sizeof(double) * ((size_t)nb + 1));
        for (int j = 0; j < nb; ++j) {
            const double *kj = ktil + ((size_t)p * n_blocks_cap + j) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += Fp[d] * kj[d];
            s[j] = acc;
        }
        if (scores) {
            for (int j = 0; j < n_blocks_cap; ++j)
                scores[(size_t)p * n_blocks_cap + j] = j < nb ? s[j] : 0.0;
        }
        bad |= select_from_scores(s, nb, n_init, n_local, k, k_tot, out, count + p);
        free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Multi-head selection of InfLLM-V2, the baseline of [SparDA] §4.3 (eq.(8) and its
 * Figure 3): every one of the G query heads of the group scores every compressed key,
 *     a^h_j = scale * <q_h, ktil_j>,   j < N_b,
 * each head's scores pass through a softmax over the pair's blocks, and the G
 * distributions are summed,
 *     s_j = sum_h exp(a^h_j) / sum_i exp(a^h_i);
 * then the k largest s_j outside the init and local blocks are taken as in
 * oracle_select.  Readings: the softmax runs over all N_b blocks (init and local
 * included); the max-pooling of the notes maps overlapping compression windows onto
 * selection blocks and is the identity for non-overlapping 64-token blocks; scale is
 * the attention scale (1/sqrt(d) when 0 is passed).
 *   Q [n_pairs][G][D] bf16 bits.  scores (nullable) receives s_j (the rest zero).
 */
int oracle_select_heads(const uint16_t *Q, int G, const double *ktil, int n_blocks_cap, int n_pairs,
                        const long long *len, double scale, int n_init, int n_local, int k, int k_tot,
                        int *idx, int *count, double *scores)
{
    if (scale == 0.0)
        scale = 1.0 / sqrt((double)D);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int p = 0; p < n_pairs; ++p) {
        int nb = blocks_of(len[p]);
        int *out = idx + (size_t)p * k_tot;
        if (nb > n_blocks_cap) {
            bad |= 1;
            count[p] = 0;
            continue;
        }
        double *a = (double *)malloc(sizeof(double) * ((size_t)nb + 1));
        double *s = (double *)calloc((size_t)nb + 1, sizeof(double));
        for (int h = 0; h < G; ++h) {
            double q[D];
            for (int d = 0; d < D; ++d)
                q[d] = bf16_value(Q[((size_t)p * G + h) * D + d]);
            double m = -INFINITY;
            for (int j = 0; j < nb; ++j) {
                const double *kj = ktil + ((size_t)p * n_blocks_cap + j) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += q[d] * kj[d];
                a[j] = scale * acc;
                if (a[j] > m)
                    m = a[j];
            }
            double z = 0.0;
            for (int j = 0; j < nb; ++j)
                z += exp(a[j] - m);
            for (int j = 0; j < nb; ++j)
                s[j] += exp(a[j] - m) / z;
        }
        if (scores) {
            for (int j = 0; j < n_blocks_cap; ++j)
                scores[(size_t)p * n_blocks_cap + j] = j < nb ? s[j] : 0.0;
        }
        bad |= select_from_scores(s, nb, n_init, n_local, k, k_tot, out, count + p);
        free(s);
        free(a);
    }
    return bad ? -1 : 0;
}

/*
 * NSA routing over overlapping compression windows (rows of oracle_pool_windows):
 *   a^h_j = scale * <q_h, kcmp_j>,  j < W(len) complete windows;
 *   p_j   = sum_h exp(a^h_j) / sum_i exp(a^h_i)    (each head's softmax, summed);
 *   s_b   = max { p_j : window j shares a token with block b }, 0 when none,
 * for the N_b = ceil(len / 64) selection blocks, then the top-k of oracle_select.
 * Readings: "shares a token" = [s*j, s*j + l) meets [64b, 64b + 64) (max-pooling
 * onto the coarse grid, [SparDA] §4.4); a block no complete window reaches (the
 * trailing one) scores 0 (the p_j are positive); scale 0 means 1/sqrt(d).
 *   kcmp [n_pairs][n_rows_cap][D]; scores (nullable) [n_pairs][n_blocks_cap] block scores.
 * Returns -1 when a pair needs more than k_tot entries, more than n_rows_cap windows
 * or more than n_blocks_cap blocks.
 */
int oracle_select_windows(const uint16_t *Q, int G, const double *kcmp, int n_rows_cap, int n_pairs,
                          const long long *len, int l, int s, double scale, int n_init, int n_local, int k,
                          int k_tot, int *idx, int *count, double *scores, int n_blocks_cap)
{
    if (scale == 0.0)
        scale = 1.0 / sqrt((double)D);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int p = 0; p < n_pairs; ++p) {
        const int nb = blocks_of(len[p]);
        const int W = windows_of(len[p], l, s);
        int *out = idx + (size_t)p * k_tot;
        if (W > n_rows_cap || nb > n_blocks_cap) {
            bad |= 1;
            count[p] = 0;
            continue;
        }
        double *a = (double *)malloc(sizeof(double) * ((size_t)W + 1));
        double *pj = (double *)calloc((size_t)W + 1, sizeof(double));
        for (int h = 0; h < G; ++h) {
            double q[D];
            for (int d = 0; d < D; ++d)
                q[d] = bf16_value(Q[((size_t)p * G + h) * D + d]);
            double m = -INFINITY;
            for (int j = 0; j < W; ++j) {
                const double *kj = kcmp + ((size_t)p * n_rows_cap + j) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += q[d] * kj[d];
                a[j] = scale * acc;
                if (a[j] > m)
                    m = a[j];
            }
            double z = 0.0;
            for (int j = 0; j < W; ++j)
                z += exp(a[j] - m);
            for (int j = 0; j < W; ++j)
                pj[j] += exp(a[j] - m) / z;
        }
        double *sb = (double *)calloc((size_t)nb + 1, sizeof(double));
        for (int b = 0; b < nb; ++b) {
            double best = 0.0;
            for (int j = 0; j < W; ++j) {
                const long long w0 = (long long)s * j, w1 = w0 + l;
                const long long b0 = (long long)b * BLK, b1 = b0 + BLK;
                if (w0 < b1 && b0 < w1 && pj[j] > best)
                    best = pj[j];
            }
            sb[b] = best;
        }
        if (scores)
            for (int b = 0; b < n_blocks_cap; ++b)
                scores[(size_t)p * n_blocks_cap + b] = b < nb ? sb[b] : 0.0;
        bad |= select_from_scores(sb, nb, n_init, n_local, k, k_tot, out, count + p);
        free(sb);
        free(pj);
        free(a);
    }
    return bad ? -1 : 0;
}

/*
 * Prefill selection, [SparDA] §4.3 eq.(16) (the Forecast indexer's prefill cost
 * H_kv * T * N_b * d: every position scores the compressed keys) with the selection of
 * eq.(6) / Alg.1 step 2 per position.  Position t of pair p (its Forecast vector
 * F[p][t]) sees the blocks holding tokens 0..t, N_t = floor(t / 64) + 1, and takes
 * B_init ∪ B_local ∪ top-k among them exactly as oracle_select does for a sequence of
 * t + 1 tokens: s_j = F[p][t] . ktil[p][j].  Reading: ktil is the prefill's pooled keys
 * (the block holding t may include later tokens, but with n_local >= 1 it is a local
 * block and its score is never used).
 *   F     [n_pairs][T_cap][D] bf16 bits;  ktil [n_pairs][n_blocks_cap][D].
 *   rows  the positions to select for (n_rows of them, each < len[p]); NULL = all t < len[p].
 *   idx   [n_pairs][n_rows or T_cap][k_tot];  count [n_pairs][n_rows or T_cap].
 * Rows of positions at or past len[p] are left untouched.  Returns -1 when a position
 * needs more than k_tot entries or more than n_blocks_cap blocks.
 */
int oracle_prefill_select(const uint16_t *F, long long T_cap, const double *ktil, int n_blocks_cap, int n_pairs,
                          const long long *len, const int *rows, int n_rows, int n_init, int n_local, int k,
                          int k_tot, int *idx, int *count)
{
    int bad = 0;
    const long long per_pair = rows ? n_rows : T_cap;
#pragma omp parallel for collapse(2) schedule(dynamic, 64) reduction(| : bad)
    for (int p = 0; p < n_pairs; ++p) {
        for (long long r = 0; r < per_pair; ++r) {
            const long long t = rows ? rows[r] : r;
            if (t < 0 || t >= len[p])
                continue;
            const int nb = (int)(t / BLK) + 1;
            int *out = idx + ((size_t)p * per_pair + r) * k_tot;
            int *cnt = count + (size_t)p * per_pair + r;
            if (nb > n_blocks_cap) {
                bad |= 1;
                *cnt = 0;
                continue;
            }
            double Fp[D];
            for (int d = 0; d < D; ++d)
                Fp[d] = bf16_value(F[((size_t)p * T_cap + t) * D + d]);
            double *sc = (double *)malloc(sizeof(double) * (size_t)nb);
            for (int j = 0; j < nb; ++j) {
                const double *kj = ktil + ((size_t)p * n_blocks_cap + j) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += Fp[d] * kj[d];
                sc[j] = acc;
            }
            bad |= select_from_scores(sc, nb, n_init, n_local, k, k_tot, out, cnt);
            free(sc);
        }
    }
    return bad ? -1 : 0;
}

/*
 * One query row q over the token set { t : block(t) in set, t < len }:
 *   a_t = scale * <q, k_t>,  o = sum_t softmax(a)_t v_t,  lse = log sum_t exp(a_t).
 * member[j] != 0 marks block j as part of the set (a set: each block counts once).
 * An empty token set gives o = 0 and lse = -inf.
 */
static void attend_set(const uint16_t *q, const uint16_t *Kp, const uint16_t *Vp,
                       const char *member, int nb, long long len, double scale,
                       double *o, double *lse)
{
    double qd[D];
    for (int d = 0; d < D; ++d)
        qd[d] = bf16_value(q[d]);
    long long ntok = 0;
    for (int j = 0; j < nb; ++j)
        if (member[j])
            ntok += BLK;
    double *a = (double *)malloc(sizeof(double) * (size_t)(ntok > 0 ? ntok : 1));
    long long *tok = (long long *)malloc(sizeof(long long) * (size_t)(ntok > 0 ? ntok : 1));
    long long n = 0;
    double m = -INFINITY;
    for (int j = 0; j < nb; ++j) {
        if (!member[j])
            continue;
        for (long long t = (long long)j * BLK; t < (long long)(j + 1) * BLK && t < len; ++t) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += qd[d] * bf16_value(Kp[(size_t)t * D + d]);
            a[n] = scale * dot;
            tok[n] = t;
            if (a[n] > m)
                m = a[n];
            ++n;
        }
    }
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
    } else {
        double L = 0.0;
        for (long long i = 0; i < n; ++i) {
            double w = exp(a[i] - m);
            L += w;
            for (int d = 0; d < D; ++d)
                o[d] += w * bf16_value(Vp[(size_t)tok[i] * D + d]);
        }
        for (int d = 0; d < D; ++d)
            o[d] /= L;
        *lse = m + log(L);
    }
    free(tok);
    free(a);
}

/*
 * Sparse decode attention, [SparDA] eq.(7).
 *   Q       [n_pairs][G][D] bf16 bits: the G query heads of KV head g of batch b
 *           (query head h belongs to group floor(h / G), so [B][H_q][D] reshapes
 *           to [B*H_kv][G][D] unchanged).
 *   K, V    [n_pairs][pair_stride][D] bf16 bits, token t of a pair at row t.
 *   blocks  [n_pairs][k_tot] logical block ids, count[p] of them valid.  The set
 *           is what counts: a repeated id is one block; ids outside [0, N_b) hold
 *           no token t < len and add nothing.
 *   scale   multiplies q.k before the softmax; 1/sqrt(128) per the NSA formula.
 *   O       [n_pairs][G][D];  lse [n_pairs][G] (nullable), natural log.
 */
void oracle_attn(const uint16_t *Q, int G, const uint16_t *K, const uint16_t *V,
                 long long pair_stride, int n_pairs, const int *blocks, const int *count,
                 int k_tot, const long long *len, double scale, double *O, double *lse)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < n_pairs; ++p) {
        int nb = blocks_of(len[p]);
        char *member = (char *)calloc((size_t)nb + 1, 1);
        for (int i = 0; i < count[p] && i < k_tot; ++i) {
            int j = blocks[(size_t)p * k_tot + i];
            if (j >= 0 && j < nb)
                member[j] = 1;
        }
        const uint16_t *Kp = K + (size_t)p * (size_t)pair_stride * D;
        const uint16_t *Vp = V + (size_t)p * (size_t)pair_stride * D;
        for (int h = 0; h < G; ++h) {
            double l;
            attend_set(Q + ((size_t)p * G + h) * D, Kp, Vp, member, nb, len[p], scale,
                       O + ((size_t)p * G + h) * D, &l);
            if (lse)
                lse[(size_t)p * G + h] = l;
        }
        free(member);
    }
}

/*
 * Softmax attention of one query row over explicit rows: tokens [t0, t1) of K / V
 * (bf16 bits; attend_tokens), or n fp64 rows kr / vr (attend_rows).  o = 0 when empty.
 */
static void attend_tokens(const double *qd, const uint16_t *Kp, const uint16_t *Vp, long long t0, long long t1,
                          double scale, double *o)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (t1 <= t0)
        return;
    double *a = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
    double m = -INFINITY;
    for (long long t = t0; t < t1; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qd[d] * bf16_value(Kp[(size_t)t * D + d]);
        a[t - t0] = scale * dot;
        if (a[t - t0] > m)
            m = a[t - t0];
    }
    double L = 0.0;
    for (long long t = t0; t < t1; ++t) {
        double w = exp(a[t - t0] - m);
        L += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * bf16_value(Vp[(size_t)t * D + d]);
    }
    for (int d = 0; d < D; ++d)
        o[d] /= L;
    free(a);
}

static void attend_rows(const double *qd, const double *kr, const double *vr, int n, double scale, double *o)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (n <= 0)
        return;
    double *a = (double *)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qd[d] * kr[(size_t)j * D + d];
        a[j] = scale * dot;
        if (a[j] > m)
            m = a[j];
    }
    double L = 0.0;
    for (int j = 0; j < n; ++j) {
        double w = exp(a[j] - m);
        L += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * vr[(size_t)j * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= L;
    free(a);
}

/*
 * NSA's gated three-branch output, [SSV] "NSA three-branch math" steps 3-6, for the
 * decode query of each pair (len[p] tokens present):
 *   o^(s) = softmax(q . K_I / sqrt d) V_I over the tokens of the selected blocks I
 *           (blocks[p][0 .. count[p]), as oracle_attn);
 *   o^(c) = softmax(q . Khat / sqrt d) Vhat over the compressed rows, one per block
 *           holding a token (khat, vhat [n_pairs][n_blocks_cap][D], e.g. oracle_pool
 *           of K and of V);
 *   o^(w) = softmax over the last window_tokens tokens [len - w, len);
 *   o     = g_c o^(c) + g_s o^(s) + g_w o^(w),  gates [n_pairs][G][3] = (g_c, g_s, g_w).
 * Readings: the compressed values are mean-pooled like the keys ([SparDA] eq.(4)), the
 * compressed branch covers all N_b blocks (the last one the mean of the tokens
 * present), the window is token-granular, and a branch with no rows contributes zero.
 *   Q [n_pairs][G][D] bf16 bits; K, V [n_pairs][pair_stride][D] bf16 bits; O [n_pairs][G][D].
 */
static void nsa_impl(const uint16_t *Q, int G, const uint16_t *K, const uint16_t *V, long long pair_stride,
                     int n_pairs, const double *khat, const double *vhat, int n_rows_cap, const int *blocks,
                     const int *count, int k_tot, const long long *len, long long window_tokens,
                     const double *gates, double scale, int cmp_len, int cmp_stride, double *O)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < n_pairs; ++p) {
        int nb = blocks_of(len[p]);
        int nrows = cmp_len > 0 ? windows_of(len[p], cmp_len, cmp_stride) : nb;
        if (nrows > n_rows_cap)
            nrows = n_rows_cap;
        char *member = (char *)calloc((size_t)nb + 1, 1);
        for (int i = 0; i < count[p] && i < k_tot; ++i) {
            int j = blocks[(size_t)p * k_tot + i];
            if (j >= 0 && j < nb)
                member[j] = 1;
        }
        const uint16_t *Kp = K + (size_t)p * (size_t)pair_stride * D;
        const uint16_t *Vp = V + (size_t)p * (size_t)pair_stride * D;
        const double *kr = khat + (size_t)p * n_rows_cap * D;
        const double *vr = vhat + (size_t)p * n_rows_cap * D;
        long long w0 = len[p] - window_tokens;
        if (w0 < 0)
            w0 = 0;
        for (int h = 0; h < G; ++h) {
            const uint16_t *q = Q + ((size_t)p * G + h) * D;
            double qd[D], os[D], oc[D], ow[D], l;
            for (int d = 0; d < D; ++d)
                qd[d] = bf16_value(q[d]);
            attend_set(q, Kp, Vp, member, nb, len[p], scale, os, &l);
            attend_rows(qd, kr, vr, nrows, scale, oc);
            attend_tokens(qd, Kp, Vp, w0, len[p], scale, ow);
            const double *g = gates + ((size_t)p * G + h) * 3;
            double *o = O + ((size_t)p * G + h) * D;
            for (int d = 0; d < D; ++d)
                o[d] = g[0] * oc[d] + g[1] * os[d] + g[2] * ow[d];
        }
        free(member);
    }
}

void oracle_nsa(const uint16_t *Q, int G, const uint16_t *K, const uint16_t *V, long long pair_stride, int n_pairs,
                const double *khat, const double *vhat, int n_blocks_cap, const int *blocks, const int *count,
                int k_tot, const long long *len, long long window_tokens, const double *gates, double scale,
                double *O)
{
    nsa_impl(Q, G, K, V, pair_stride, n_pairs, khat, vhat, n_blocks_cap, blocks, count, k_tot, len, window_tokens,
             gates, scale, 0, 0, O);
}

/*
 * oracle_nsa with NSA's overlapping compression: the compressed branch attends over the
 * W(len) complete windows of kernel cmp_len and stride cmp_stride (khat, vhat
 * [n_pairs][n_rows_cap][D], e.g. oracle_pool_windows of K and of V).
 */
void oracle_nsa_windows(const uint16_t *Q, int G, const uint16_t *K, const uint16_t *V, long long pair_stride,
                        int n_pairs, const double *khat, const double *vhat, int n_rows_cap, const int *blocks,
                        const int *count, int k_tot, const long long *len, long long window_tokens,
                        const double *gates, double scale, int cmp_len, int cmp_stride, double *O)
{
    nsa_impl(Q, G, K, V, pair_stride, n_pairs, khat, vhat, n_rows_cap, blocks, count, k_tot, len, window_tokens,
             gates, scale, cmp_len, cmp_stride, O);
}

/*
 * Grouped speculative verification, [SSV] mechanism 1.
 *   Q   [B][N_q][H_q][D] bf16 bits: N_q verification queries per sequence, already in
 *       the flattened (BFS) order; groups are queries [gC, gC+C).
 *   K,V [B][H_kv][T_cap][D] bf16 bits (committed tokens only; draft tokens are not
 *       in the cache and are not attended).
 *   I   [B][H_kv][N_q][n_sel] per-query selected block ids.
 *   The sliding window is the last window_blocks blocks of the committed sequence
 *   (block-granular reading of "the last w tokens").
 * Mode A (exact merged schedule, oracle_verify): query q, head h attends over its own
 * set I_q ∪ W with the plain softmax of oracle_attn; the group loads the merged union.
 * Mode B (approximate shared layout, oracle_verify_shared): every query of a group
 * attends over the layout of the group's representative, its first query:
 * I_{q_rep} ∪ W; the group loads that one layout.
 *   O   [B][N_q][H_q][D].
 *   union_blocks     += the blocks a group loads, summed over (b, KV head, group)
 *   per_query_blocks += sum_q |I_q ∪ W| over the same: the loads without grouping.
 */
static void verify_impl(const uint16_t *Q, const uint16_t *K, const uint16_t *V, long long T_cap, int B, int H_q,
                        int H_kv, int N_q, const int *I, int n_sel, int C, int window_blocks, const long long *len,
                        double scale, double *O, long long *union_blocks, long long *per_query_blocks, int shared)
{
    int G = H_q / H_kv;
    long long tot_union = 0, tot_query = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(+ : tot_union, tot_query)
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < H_kv; ++g) {
            int nb = blocks_of(len[b]);
            const uint16_t *Kp = K + ((size_t)b * H_kv + g) * (size_t)T_cap * D;
            const uint16_t *Vp = V + ((size_t)b * H_kv + g) * (size_t)T_cap * D;
            char *merged = (char *)calloc((size_t)nb + 1, 1);
            char *member = (char *)calloc((size_t)nb + 1, 1);
            char *own = (char *)calloc((size_t)nb + 1, 1);
            for (int q0 = 0; q0 < N_q; q0 += C) {
                memset(merged, 0, (size_t)nb + 1);
                for (int q = q0; q < q0 + C && q < N_q; ++q) {
                    /* the query's own set I_q ∪ W, for the ungrouped count */
                    memset(own, 0, (size_t)nb + 1);
                    const int *Iq = I + (((size_t)b * H_kv + g) * N_q + q) * n_sel;
                    for (int i = 0; i < n_sel; ++i)
                        if (Iq[i] >= 0 && Iq[i] < nb)
                            own[Iq[i]] = 1;
                    for (int j = nb - window_blocks; j < nb; ++j)
                        if (j >= 0)
                            own[j] = 1;
                    for (int j = 0; j < nb; ++j)
                        tot_query += own[j];
                    /* the set it attends over: its own (mode A) or the representative's (mode B) */
                    memset(member, 0, (size_t)nb + 1);
                    const int *Ia = shared ? I + (((size_t)b * H_kv + g) * N_q + q0) * n_sel : Iq;
                    for (int i = 0; i < n_sel; ++i)
                        if (Ia[i] >= 0 && Ia[i] < nb)
                            member[Ia[i]] = 1;
                    for (int j = nb - window_blocks; j < nb; ++j)
                        if (j >= 0)
                            member[j] = 1;
                    for (int j = 0; j < nb; ++j)
                        merged[j] |= member[j];
                    for (int hh = 0; hh < G; ++hh) {
                        int h = g * G + hh;
                        double l;
                        attend_set(Q + (((size_t)b * N_q + q) * H_q + h) * D, Kp, Vp, member, nb,
                                   len[b], scale, O + (((size_t)b * N_q + q) * H_q + h) * D, &l);
                    }
                }
                for (int j = 0; j < nb; ++j)
                    tot_union += merged[j];
            }
            free(own);
            free(member);
            free(merged);
        }
    }
    if (union_blocks)
        *union_blocks = tot_union;
    if (per_query_blocks)
        *per_query_blocks = tot_query;
}

void oracle_verify(const uint16_t *Q, const uint16_t *K, const uint16_t *V, long long T_cap,
                   int B, int H_q, int H_kv, int N_q, const int *I, int n_sel, int C,
                   int window_blocks, const long long *len, double scale, double *O,
                   long long *union_blocks, long long *per_query_blocks)
{
    verify_impl(Q, K, V, T_cap, B, H_q, H_kv, N_q, I, n_sel, C, window_blocks, len, scale, O, union_blocks,
                per_query_blocks, 0);
}

void oracle_verify_shared(const uint16_t *Q, const uint16_t *K, const uint16_t *V, long long T_cap,
                          int B, int H_q, int H_kv, int N_q, const int *I, int n_sel, int C,
                          int window_blocks, const long long *len, double scale, double *O,
                          long long *union_blocks, long long *per_query_blocks)
{
    verify_impl(Q, K, V, T_cap, B, H_q, H_kv, N_q, I, n_sel, C, window_blocks, len, scale, O, union_blocks,
                per_query_blocks, 1);
}

/*
 * Offload staging, [SparDA] §4.5: copy the K (or V) rows of the selected blocks from
 * the host cache [n_pairs][T_host][D] into the staging layout [n_pairs][k_tot][64][D]:
 * slot i of pair p holds block idx[p][i].  Rows past T_host are zero; slots at or
 * beyond count[p] are left untouched.
 */
void oracle_gather(const uint16_t *src, long long T_host, int n_pairs, const int *idx,
                   const int *count, int k_tot, uint16_t *ring)
{
    for (int p = 0; p < n_pairs; ++p) {
        for (int i = 0; i < count[p] && i < k_tot; ++i) {
            int j = idx[(size_t)p * k_tot + i];
            uint16_t *dst = ring + (((size_t)p * k_tot + i) * BLK) * D;
            for (int r = 0; r < BLK; ++r) {
                long long t = (long long)j * BLK + r;
                for (int d = 0; d < D; ++d)
                    dst[(size_t)r * D + d] =
                        (j >= 0 && t < T_host) ? src[((size_t)p * T_host + t) * D + d] : 0;
            }
        }
    }
}
