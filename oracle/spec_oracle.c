/*
 * spec_oracle.c -- the ORACLE for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or run this file.  It shares no code,
 * header, helper or table with the CUDA library, and neither side includes the other.
 *
 * Everything here is plain, slow and written to be checked by eye against the pages:
 * every probability is a full fp64 softmax of the row, every sum is a left-to-right loop,
 * every search is a linear scan.  No blocking, no fusion, no reordering.
 *
 * Sources (page title -- section):
 *   [SD]  "7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead"
 *         -- "The rule", "The proof that this is exact", "Extending to a chain of gamma
 *         draft tokens", "A From-Scratch Implementation" (apply_temperature,
 *         speculative_step), "Tree Attention: Verifying Many Candidates at Once",
 *         "Exercises" 2 and 5 (verify_tree_greedy).
 *   [MS]  "Medusa, EAGLE and self-speculation" -- "Copying, verified against plain
 *         greedy" (speculative_greedy: longest matching prefix, then the correction
 *         argmax at the stop row).
 *   [HB]  "Speculative Decoding: Draft Models, EAGLE, and How to Actually Use It"
 *         -- "The Algorithm" (steps 1-4 and the worked p/q example).
 *         The "Medusa" paragraph and the closing note on typical acceptance (a
 *         threshold scaled by the step's entropy; oracle_verify_typical).
 *   [PH]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
 *         (SC'11): the Philox4x32-10 counter-based generator.
 *
 * Readings taken where the pages leave a step open:
 *   - uniforms: Philox4x32-10, key = seed, counter = (4*i + purpose, b, offset lo, offset hi),
 *     word 0, u = (w >> 8) * 2^-24 (exactly representable in fp32 and fp64).
 *   - accept test: u * q(x) < p(x)  (the page's strict "r < accept_prob" with the division
 *     cleared; q(x) = 0 < p(x) accepts, q(x) = p(x) = 0 rejects).
 *   - residual / bonus draw: inverse CDF in vocabulary-index order, the first j with
 *     C_j > u' * R; if rounding leaves none, the last j with r_j > 0.
 *   - residual mass R == 0 after a rejection: draw from p on that row instead.
 *   - a sequence with a NaN / +inf / all -inf row (sampling), a NaN row (greedy, tree) or a
 *     draft token outside [0, V) gets accepted_len = -1 and all its tokens = -1.
 *   - argmax ties go to the lowest index.
 *   - tree: the deepest accepted node wins; among equally deep ones the lowest node index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DTYPE_FP32 0
#define ORACLE_DTYPE_BF16 1

/* Flag bits reported per sequence by oracle_verify_sample. */
#define FLAG_ACCEPT_NEAR_THRESHOLD 1 /* some performed accept test had |u - p/q| < 1e-5     */
#define FLAG_CDF_NEAR_BOUNDARY 2     /* u'R within 1e-5 R of C_{j-1} or C_j of the drawn j  */
#define FLAG_RESIDUAL_NEAR_ZERO 4    /* R < 1e-6 after a rejection (fallback may trigger)   */
#define FLAG_RESIDUAL_FALLBACK 8     /* R == 0 exactly: the draw used p (reading above)     */

/* Flag bit reported per sequence by oracle_verify_tree_greedy. */
#define FLAG_TREE_FIRST_MATCH_DIFFERS 1 /* Exercise 5's first-matching-child walk picks another path */

static const double ACCEPT_WINDOW = 1e-5;
static const double CDF_WINDOW = 1e-5;
static const double RESIDUAL_SMALL = 1e-6;

/* ------------------------------------------------------------------------------------ */
/* Philox4x32-10 [PH]: ten rounds of the Philox S-box on a 4x32-bit counter, the 2x32-bit
 * key bumped by the Weyl constants between rounds.                                      */
/* ------------------------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u; /* round multipliers  */
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u; /* Weyl key increments */
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += W0;
            k1 += W1;
        }
        uint64_t prod0 = (uint64_t)M0 * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* The uniform the verifier draws at (sequence b, position i, purpose).
 * purpose 0: the accept test of draft position i; purpose 1: the final draw on row i. */
double oracle_uniform(uint64_t seed, uint64_t offset, uint32_t b, uint32_t i, uint32_t purpose)
{
    uint32_t ctr[4], key[2], w[4];
    ctr[0] = (i << 2) | (purpose & 3u);
    ctr[1] = b;
    ctr[2] = (uint32_t)(offset & 0xFFFFFFFFu);
    ctr[3] = (uint32_t)(offset >> 32);
    key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
    key[1] = (uint32_t)(seed >> 32);
    oracle_philox4x32_10(ctr, key, w);
    return (double)(w[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------------------ */
/* Reading logits                                                                        */
/* ------------------------------------------------------------------------------------ */
static double logit_at(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_DTYPE_FP32)
        return (double)((const float *)base)[idx];
    /* bf16 is the top half of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void load_row(const void *base, int dtype, int64_t row_start, int V, double *out)
{
    for (int j = 0; j < V; ++j)
        out[j] = logit_at(base, dtype, row_start + j);
}

/* ------------------------------------------------------------------------------------ */
/* apply_temperature [SD "A From-Scratch Implementation"]: p = softmax(logits / T).
 * Returns 0 and fills p, m = max_j l_j / T and S = sum_j exp(l_j / T - m) for a proper
 * distribution; returns -1 when the row has a NaN, a +inf or no finite entry.            */
/* ------------------------------------------------------------------------------------ */
static int softmax_row(const double *l, int V, double T, double *p, double *m_out, double *S_out)
{
    double m = -INFINITY;
    for (int j = 0; j < V; ++j) {
        if (isnan(l[j]) || l[j] == INFINITY)
            return -1;
        if (l[j] / T > m)
            m = l[j] / T;
    }
    if (m == -INFINITY)
        return -1;
    double S = 0.0;
    for (int j = 0; j < V; ++j)
        S += exp(l[j] / T - m);
    for (int j = 0; j < V; ++j)
        p[j] = exp(l[j] / T - m) / S;
    if (m_out)
        *m_out = m;
    if (S_out)
        *S_out = S;
    return 0;
}

/* Per-row statistics: m = max_j l_j / T and lse = m + ln sum_j exp(l_j / T - m), fp64.
 * Rows are [B][rows_per_seq][V] with the given batch and row strides (in elements).   */
int oracle_row_stats(const void *logits, int64_t batch_stride, int64_t row_stride, int dtype,
                     int B, int rows_per_seq, int V, double T, double *m_out, double *lse_out,
                     int *valid_out)
{
    double *l = (double *)malloc(sizeof(double) * (size_t)V);
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    if (!l || !p) {
        free(l);
        free(p);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        for (int r = 0; r < rows_per_seq; ++r) {
            int64_t k = (int64_t)b * rows_per_seq + r;
            load_row(logits, dtype, (int64_t)b * batch_stride + (int64_t)r * row_stride, V, l);
            double m = NAN, S = NAN;
            int ok = softmax_row(l, V, T, p, &m, &S) == 0;
            valid_out[k] = ok;
            m_out[k] = ok ? m : NAN;
            lse_out[k] = ok ? m + log(S) : NAN;
        }
    }
    free(l);
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* The accept probability min(1, p(x)/q(x)) [SD "The rule"], with the cleared-division
 * reading: it is the probability that u * q < p for u uniform on [0, 1).                */
/* ------------------------------------------------------------------------------------ */
static double accept_probability(double px, double qx)
{
    if (qx > 0.0)
        return px / qx < 1.0 ? px / qx : 1.0;
    return px > 0.0 ? 1.0 : 0.0;
}

/* The distribution the final token of a round is drawn from [SD "The rule", "Extending to
 * a chain"]: after a rejection the residual (p - q)+ (unnormalised), after a full accept
 * the target row p itself.  Returns the total mass R.  If a residual has R == 0 the
 * reading above draws from p instead and *fell_back is set.                            */
static double final_weights(const double *p, const double *q, int V, int residual, double *r,
                            int *fell_back)
{
    double R = 0.0;
    *fell_back = 0;
    if (residual) {
        for (int j = 0; j < V; ++j) {
            double d = p[j] - q[j];
            r[j] = d > 0.0 ? d : 0.0;
            R += r[j];
        }
        if (R > 0.0)
            return R;
        *fell_back = 1;
    }
    R = 0.0;
    for (int j = 0; j < V; ++j) {
        r[j] = p[j];
        R += r[j];
    }
    return R;
}

/* Inverse CDF in index order: the first j with C_j = r_0 + ... + r_j > u * R.
 * Also reports the distance from u * R to the nearer of C_{j-1} and C_j, divided by R.  */
static int inverse_cdf(const double *r, int V, double R, double u, double *margin)
{
    double target = u * R;
    double C = 0.0;
    int last_positive = -1;
    for (int j = 0; j < V; ++j) {
        double prev = C;
        C += r[j];
        if (r[j] > 0.0)
            last_positive = j;
        if (C > target) {
            *margin = fmin(fabs(target - prev), fabs(C - target)) / R;
            return j;
        }
    }
    *margin = 0.0;
    return last_positive;
}

/* ------------------------------------------------------------------------------------ */
/* Sampling verification [SD speculative_step, "Extending to a chain"; HB "The Algorithm"].
 *   target: [B][gamma+1][V] (row i predicts the token after the i-th draft; row gamma is
 *           the bonus row), draft: [B][gamma][V], draft_tokens: [B][gamma] contiguous.
 *   b0 is the global index of the first sequence passed (it keys the uniforms).
 * Outputs: accepted_len[B], out_tokens[B][gamma+1] (-1 padded), flags[B].              */
/* ------------------------------------------------------------------------------------ */
int oracle_verify_sample(const void *target, int64_t t_batch_stride, int64_t t_row_stride,
                         const void *draft, int64_t d_batch_stride, int64_t d_row_stride,
                         int dtype, int B, int b0, int gamma, int V, const int32_t *draft_tokens,
                         double T, uint64_t seed, uint64_t offset, int32_t *accepted_len,
                         int32_t *out_tokens, int32_t *flags, double *diag)
{
    size_t rowsz = sizeof(double) * (size_t)V;
    double *l = (double *)malloc(rowsz);
    double *p = (double *)malloc(rowsz * (size_t)(gamma + 1));
    double *q = (double *)malloc(rowsz * (size_t)(gamma > 0 ? gamma : 1));
    double *r = (double *)malloc(rowsz);
    if (!l || !p || !q || !r) {
        free(l);
        free(p);
        free(q);
        free(r);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        int32_t *out = out_tokens + (int64_t)b * (gamma + 1);
        for (int i = 0; i <= gamma; ++i)
            out[i] = -1;
        accepted_len[b] = -1;
        flags[b] = 0;
        if (diag) {
            diag[4 * b + 0] = -1.0; /* final draw: 0 bonus, 1 residual, 2 residual fell back to p */
            diag[4 * b + 1] = 0.0;  /* mass R of the final draw's weights */
            diag[4 * b + 2] = 0.0;  /* distance of u'R to the nearer CDF boundary, over R */
            diag[4 * b + 3] = INFINITY; /* smallest |u - p/q| over the accept tests performed */
        }

        /* every row is turned into a distribution first: p_i = softmax(t_i / T),
         * q_i = softmax(d_i / T) -- the temperature applies to BOTH models */
        int ok = 1;
        for (int i = 0; i <= gamma && ok; ++i) {
            load_row(target, dtype, (int64_t)b * t_batch_stride + (int64_t)i * t_row_stride, V, l);
            ok = softmax_row(l, V, T, p + (size_t)i * V, NULL, NULL) == 0;
        }
        for (int i = 0; i < gamma && ok; ++i) {
            load_row(draft, dtype, (int64_t)b * d_batch_stride + (int64_t)i * d_row_stride, V, l);
            ok = softmax_row(l, V, T, q + (size_t)i * V, NULL, NULL) == 0;
        }
        for (int i = 0; i < gamma && ok; ++i) {
            int32_t x = draft_tokens[(int64_t)b * gamma + i];
            ok = x >= 0 && x < V;
        }
        if (!ok)
            continue;

        /* walk the drafts left to right; the first rejection ends the round */
        int k = gamma, residual = 0;
        for (int i = 0; i < gamma; ++i) {
            int32_t x = draft_tokens[(int64_t)b * gamma + i];
            double px = p[(size_t)i * V + x], qx = q[(size_t)i * V + x];
            double u = oracle_uniform(seed, offset, (uint32_t)(b0 + b), (uint32_t)i, 0u);
            if (qx > 0.0 && fabs(u - px / qx) < ACCEPT_WINDOW)
                flags[b] |= FLAG_ACCEPT_NEAR_THRESHOLD;
            if (diag && qx > 0.0 && fabs(u - px / qx) < diag[4 * b + 3])
                diag[4 * b + 3] = fabs(u - px / qx);
            if (u * qx < px) {
                out[i] = x; /* accepted */
            } else {
                k = i; /* rejected: resample this position from the residual, then stop */
                residual = 1;
                break;
            }
        }

        /* the final token: residual after a rejection, the bonus from p after a full accept */
        int fell_back = 0;
        double margin = 0.0;
        double R = final_weights(p + (size_t)k * V, residual ? q + (size_t)k * V : NULL, V,
                                 residual, r, &fell_back);
        if (residual) {
            double Rres = 0.0;
            for (int j = 0; j < V; ++j) {
                double d = p[(size_t)k * V + j] - q[(size_t)k * V + j];
                Rres += d > 0.0 ? d : 0.0;
            }
            if (Rres < RESIDUAL_SMALL)
                flags[b] |= FLAG_RESIDUAL_NEAR_ZERO;
        }
        if (fell_back)
            flags[b] |= FLAG_RESIDUAL_FALLBACK;
        double u2 = oracle_uniform(seed, offset, (uint32_t)(b0 + b), (uint32_t)k, 1u);
        out[k] = inverse_cdf(r, V, R, u2, &margin);
        if (margin < CDF_WINDOW)
            flags[b] |= FLAG_CDF_NEAR_BOUNDARY;
        accepted_len[b] = k;
        if (diag) {
            diag[4 * b + 0] = fell_back ? 2.0 : (residual ? 1.0 : 0.0);
            diag[4 * b + 1] = R;
            diag[4 * b + 2] = margin;
        }
    }
    free(l);
    free(p);
    free(q);
    free(r);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Enumeration mode: the exact law of one round for fixed rows and fixed drafts.
 * Each uniform becomes branch weights: accept with min(1, p/q), the final token j with
 * r_j / R.  prob[k*V + j] = P(accepted_len = k and final token = j).  Logits are given
 * as fp64, target [(gamma+1)][V], draft [gamma][V].  Returns -1 on an invalid row.     */
/* ------------------------------------------------------------------------------------ */
int oracle_exact_probs(const double *t_logits, const double *d_logits, int gamma, int V,
                       const int32_t *x, double T, double *prob)
{
    size_t rowsz = sizeof(double) * (size_t)V;
    double *p = (double *)malloc(rowsz);
    double *q = (double *)malloc(rowsz);
    double *r = (double *)malloc(rowsz);
    int rc = 0;
    if (!p || !q || !r) {
        rc = -1;
        goto done;
    }
    for (int j = 0; j < (gamma + 1) * V; ++j)
        prob[j] = 0.0;
    double reach = 1.0; /* probability that drafts 0..i-1 were all accepted */
    for (int i = 0; i < gamma; ++i) {
        if (softmax_row(t_logits + (size_t)i * V, V, T, p, NULL, NULL) != 0 ||
            softmax_row(d_logits + (size_t)i * V, V, T, q, NULL, NULL) != 0 || x[i] < 0 ||
            x[i] >= V) {
            rc = -1;
            goto done;
        }
        double a = accept_probability(p[x[i]], q[x[i]]);
        int fell_back = 0;
        double R = final_weights(p, q, V, 1, r, &fell_back);
        for (int j = 0; j < V; ++j)
            prob[(size_t)i * V + j] += reach * (1.0 - a) * r[j] / R;
        reach *= a;
    }
    if (softmax_row(t_logits + (size_t)gamma * V, V, T, p, NULL, NULL) != 0) {
        rc = -1;
        goto done;
    }
    for (int j = 0; j < V; ++j)
        prob[(size_t)gamma * V + j] += reach * p[j];
done:
    free(p);
    free(q);
    free(r);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* Argmax with ties to the lowest index; -1 if the row holds a NaN.                      */
/* ------------------------------------------------------------------------------------ */
static int argmax_row(const double *l, int V)
{
    int best = 0;
    for (int j = 0; j < V; ++j)
        if (isnan(l[j]))
            return -1;
    for (int j = 1; j < V; ++j)
        if (l[j] > l[best])
            best = j;
    return best;
}

/* ------------------------------------------------------------------------------------ */
/* Greedy verification [SD "Extending to a chain" (temperature 0); MS speculative_greedy]:
 * a_i = argmax of target row i; accept the longest prefix with draft_i == a_i; the
 * token at the stop row is a_n (the correction, or the bonus when n == gamma).         */
/* ------------------------------------------------------------------------------------ */
int oracle_verify_greedy(const void *target, int64_t t_batch_stride, int64_t t_row_stride,
                         int dtype, int B, int gamma, int V, const int32_t *draft_tokens,
                         int32_t *accepted_len, int32_t *out_tokens)
{
    double *l = (double *)malloc(sizeof(double) * (size_t)V);
    int *a = (int *)malloc(sizeof(int) * (size_t)(gamma + 1));
    if (!l || !a) {
        free(l);
        free(a);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        int32_t *out = out_tokens + (int64_t)b * (gamma + 1);
        for (int i = 0; i <= gamma; ++i)
            out[i] = -1;
        accepted_len[b] = -1;
        int ok = 1;
        for (int i = 0; i <= gamma && ok; ++i) {
            load_row(target, dtype, (int64_t)b * t_batch_stride + (int64_t)i * t_row_stride, V, l);
            a[i] = argmax_row(l, V);
            ok = a[i] >= 0;
        }
        for (int i = 0; i < gamma && ok; ++i) {
            int32_t x = draft_tokens[(int64_t)b * gamma + i];
            ok = x >= 0 && x < V;
        }
        if (!ok)
            continue;
        int n = 0;
        while (n < gamma && draft_tokens[(int64_t)b * gamma + n] == a[n]) {
            out[n] = draft_tokens[(int64_t)b * gamma + n];
            ++n;
        }
        out[n] = a[n];
        accepted_len[b] = n;
    }
    free(l);
    free(a);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Greedy token-tree verification [SD "Tree Attention", Exercise 5 verify_tree_greedy].
 * parent[N]: parent[0] = -1, parent[v] < v.  node_tokens[B][N] ([b][0], the committed
 * root, is ignored).  target: [B][N][V], row v predicts the token after node v.
 * A node v != 0 is accepted when node_tokens[b][v] == argmax(row parent[v]) and its
 * parent is accepted (the root always is).  The deepest accepted node v* wins (lowest
 * index among equally deep ones).  Outputs, each row max_depth+1 wide, -1 padded:
 *   out_path[b]   = node ids root..v*,  out_tokens[b] = tokens of the path without the
 *   root, then argmax(row v*);  accepted_len[b] = depth(v*).
 * A tree that is malformed or deeper than max_depth makes every sequence -1.           */
/* ------------------------------------------------------------------------------------ */
int oracle_verify_tree_greedy(const void *target, int64_t t_batch_stride, int64_t t_row_stride,
                              int dtype, int B, int N, int V, const int32_t *parent,
                              const int32_t *node_tokens, int max_depth, int32_t *accepted_len,
                              int32_t *out_tokens, int32_t *out_path, int32_t *flags)
{
    int W = max_depth + 1;
    for (int b = 0; b < B; ++b) {
        accepted_len[b] = -1;
        flags[b] = 0;
        for (int i = 0; i < W; ++i) {
            out_tokens[(int64_t)b * W + i] = -1;
            if (out_path)
                out_path[(int64_t)b * W + i] = -1;
        }
    }
    int *depth = (int *)malloc(sizeof(int) * (size_t)N);
    int *a = (int *)malloc(sizeof(int) * (size_t)N);
    int *acc = (int *)malloc(sizeof(int) * (size_t)N);
    int *path = (int *)malloc(sizeof(int) * (size_t)N);
    double *l = (double *)malloc(sizeof(double) * (size_t)V);
    if (!depth || !a || !acc || !path || !l) {
        free(depth);
        free(a);
        free(acc);
        free(path);
        free(l);
        return -1;
    }
    /* the tree itself: parent before child, depth(root) = 0 */
    int tree_ok = N >= 1 && parent[0] == -1;
    for (int v = 1; v < N && tree_ok; ++v)
        tree_ok = parent[v] >= 0 && parent[v] < v;
    if (tree_ok) {
        depth[0] = 0;
        for (int v = 1; v < N; ++v) {
            depth[v] = depth[parent[v]] + 1;
            if (depth[v] > max_depth)
                tree_ok = 0;
        }
    }
    for (int b = 0; b < B && tree_ok; ++b) {
        int ok = 1;
        for (int v = 0; v < N && ok; ++v) {
            load_row(target, dtype, (int64_t)b * t_batch_stride + (int64_t)v * t_row_stride, V, l);
            a[v] = argmax_row(l, V);
            ok = a[v] >= 0;
        }
        for (int v = 1; v < N && ok; ++v) {
            int32_t tok = node_tokens[(int64_t)b * N + v];
            ok = tok >= 0 && tok < V;
        }
        if (!ok)
            continue;
        /* accepted: the root, and every node whose token is its parent's argmax and whose
         * parent is accepted (parents come first, so one forward sweep settles it) */
        acc[0] = 1;
        for (int v = 1; v < N; ++v)
            acc[v] = acc[parent[v]] && node_tokens[(int64_t)b * N + v] == a[parent[v]];
        int best = 0;
        for (int v = 1; v < N; ++v)
            if (acc[v] && depth[v] > depth[best])
                best = v;
        int d = depth[best];
        for (int v = best, s = d; s >= 0; --s) {
            path[s] = v;
            v = parent[v];
        }
        for (int s = 0; s <= d; ++s) {
            if (out_path)
                out_path[(int64_t)b * W + s] = path[s];
            if (s >= 1)
                out_tokens[(int64_t)b * W + s - 1] = node_tokens[(int64_t)b * N + path[s]];
        }
        out_tokens[(int64_t)b * W + d] = a[best];
        accepted_len[b] = d;

        /* Exercise 5's walk: from the root, step to the FIRST child whose token matches */
        int node = 0, walk_depth = 0, same = 1;
        for (;;) {
            int next = -1;
            for (int c = node + 1; c < N; ++c)
                if (parent[c] == node && node_tokens[(int64_t)b * N + c] == a[node]) {
                    next = c;
                    break;
                }
            if (next < 0)
                break;
            node = next;
            ++walk_depth;
            if (walk_depth > d || path[walk_depth] != node)
                same = 0;
        }
        if (!same || walk_depth != d)
            flags[b] |= FLAG_TREE_FIRST_MATCH_DIFFERS;
    }
    free(depth);
    free(a);
    free(acc);
    free(path);
    free(l);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Token-tree SAMPLING verification: multi-round (recursive) rejection sampling
 * [SD "Tree Attention: Verifying Many Candidates at Once", the paragraph after
 * build_tree_attn (SpecInfer's rule)].  At an accepted node v with children c_1 < c_2 <
 * ... (node-index order = the order the drafter drew them from q_v):
 *   test c_r's token x with the single-candidate rule against the CURRENT (p, q):
 *   accept iff u * q(x) < p(x), u = U(b, c_r - 1, 0); an accepted child becomes the new v;
 *   a rejection replaces p by the residual (p - q)+ / ||(p - q)+||_1 and, when the
 *   siblings were drawn without replacement, q by q with x removed, renormalised.
 * When every child of v is rejected the final token is drawn from the last residual;
 * at a leaf it is the bonus drawn from p_v; both with u' = U(b, v, 1) by inverse CDF.
 * With a chain-shaped tree (node i's only child is i + 1) this is exactly
 * oracle_verify_sample, uniforms included.
 * Readings: a residual of mass 0 leaves p unchanged (flagged); without
 * replacement a q with no mass left is 0 everywhere (a later sibling is then accepted iff
 * p(x) > 0, and the residual is p).  Validity: every node token in [0, V) and every row
 * the walk reads (the target row of each node it reaches, the draft row of each reached
 * node that has children) a distribution -- a row the rule never reads cannot change the
 * result; the tree well-formed and no deeper than max_depth.  Otherwise the sequence (or,
 * for the tree, every sequence) is -1.
 *   target, draft: [B][N][V] (row v: the target's / drafter's logits after the path to v)
 *   parent[N], node_tokens[B][N] as in oracle_verify_tree_greedy.
 * Outputs (max_depth + 1 wide, -1 padded): accepted_len[b] = depth of the final node,
 * out_tokens[b] = path tokens without the root then the final token, out_path[b] = node
 * ids root..final node, flags[b] as in oracle_verify_sample.                           */
/* ------------------------------------------------------------------------------------ */

/* After a rejected candidate x: r <- (p - q)+ (returns its mass R), p <- r / R (unchanged
 * if R == 0; *fell_back is set then), and without replacement q <- q without x,
 * renormalised.                                                                         */
static double reject_update(double *p, double *q, int V, int x, int without_replacement,
                            double *r, int *fell_back)
{
    double R = 0.0;
    for (int j = 0; j < V; ++j) {
        double d = p[j] - q[j];
        r[j] = d > 0.0 ? d : 0.0;
        R += r[j];
    }
    *fell_back = !(R > 0.0);
    if (R > 0.0)
        for (int j = 0; j < V; ++j)
            p[j] = r[j] / R;
    if (without_replacement) {
        q[x] = 0.0;
        double Q = 0.0;
        for (int j = 0; j < V; ++j)
            Q += q[j];
        for (int j = 0; j < V; ++j)
            q[j] = Q > 0.0 ? q[j] / Q : 0.0;
    }
    return R;
}

/* depth[] of a well-formed tree no deeper than max_depth; returns 0 otherwise. */
static int tree_depths(const int32_t *parent, int N, int max_depth, int *depth)
{
    if (N < 1 || parent[0] != -1)
        return 0;
    depth[0] = 0;
    for (int v = 1; v < N; ++v) {
        if (parent[v] < 0 || parent[v] >= v)
            return 0;
        depth[v] = depth[parent[v]] + 1;
        if (depth[v] > max_depth)
            return 0;
    }
    return 1;
}

int oracle_verify_tree_sample(const void *target, int64_t t_batch_stride, int64_t t_row_stride,
                              const void *draft, int64_t d_batch_stride, int64_t d_row_stride,
                              int dtype, int B, int b0, int N, int V, const int32_t *parent,
                              const int32_t *node_tokens, int max_depth, double T,
                              int without_replacement, uint64_t seed, uint64_t offset,
                              int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path,
                              int32_t *flags)
{
    int W = max_depth + 1;
    for (int b = 0; b < B; ++b) {
        accepted_len[b] = -1;
        flags[b] = 0;
        for (int i = 0; i < W; ++i) {
            out_tokens[(int64_t)b * W + i] = -1;
            if (out_path)
                out_path[(int64_t)b * W + i] = -1;
        }
    }
    size_t rowsz = sizeof(double) * (size_t)V;
    int *depth = (int *)malloc(sizeof(int) * (size_t)N);
    int *nchild = (int *)malloc(sizeof(int) * (size_t)N);
    double *l = (double *)malloc(rowsz);
    double *p = (double *)malloc(rowsz);
    double *q = (double *)malloc(rowsz);
    double *r = (double *)malloc(rowsz);
    if (!depth || !nchild || !l || !p || !q || !r) {
        free(depth);
        free(nchild);
        free(l);
        free(p);
        free(q);
        free(r);
        return -1;
    }
    int tree_ok = tree_depths(parent, N, max_depth, depth);
    for (int v = 0; v < N; ++v)
        nchild[v] = 0;
    for (int v = 1; v < N && tree_ok; ++v)
        nchild[parent[v]]++;
    for (int b = 0; b < B && tree_ok; ++b) {
        /* every node token must be in range; rows are checked as the walk reads them */
        int ok = 1;
        for (int v = 1; v < N && ok; ++v) {
            int32_t tok = node_tokens[(int64_t)b * N + v];
            ok = tok >= 0 && tok < V;
        }
        if (!ok)
            continue;

        /* the walk from the root; after a rejection r holds the unnormalised residual
         * (p - q)+ of mass Rr that the final draw uses, exactly as the chain rule does */
        int v = 0, rejected = 0;
        double Rr = 0.0;
        for (;;) {
            rejected = 0;
            load_row(target, dtype, (int64_t)b * t_batch_stride + (int64_t)v * t_row_stride, V, l);
            ok = softmax_row(l, V, T, p, NULL, NULL) == 0;
            if (ok && nchild[v] > 0) {
                load_row(draft, dtype, (int64_t)b * d_batch_stride + (int64_t)v * d_row_stride, V, l);
                ok = softmax_row(l, V, T, q, NULL, NULL) == 0;
            }
            if (!ok)
                break;
            int next = -1;
            for (int c = v + 1; c < N && next < 0; ++c) {
                if (parent[c] != v)
                    continue;
                int x = node_tokens[(int64_t)b * N + c];
                double u = oracle_uniform(seed, offset, (uint32_t)(b0 + b), (uint32_t)(c - 1), 0u);
                if (q[x] > 0.0 && fabs(u - p[x] / q[x]) < ACCEPT_WINDOW)
                    flags[b] |= FLAG_ACCEPT_NEAR_THRESHOLD;
                if (u * q[x] < p[x]) {
                    next = c; /* accepted */
                } else {
                    int fell_back = 0;
                    Rr = reject_update(p, q, V, x, without_replacement, r, &fell_back);
                    rejected = !fell_back;
                    if (Rr < RESIDUAL_SMALL)
                        flags[b] |= FLAG_RESIDUAL_NEAR_ZERO;
                    if (fell_back)
                        flags[b] |= FLAG_RESIDUAL_FALLBACK;
                }
            }
            if (next < 0)
                break;
            v = next;
        }

        if (!ok) {
            flags[b] = 0;
            continue;
        }
        /* the final token: from the last residual after the children were all rejected,
         * from p_v at a leaf (or where the last residual had no mass) */
        double R = 0.0, margin = 0.0;
        const double *w = p;
        if (rejected) {
            w = r;
            R = Rr;
        } else {
            for (int j = 0; j < V; ++j)
                R += p[j];
        }
        double u2 = oracle_uniform(seed, offset, (uint32_t)(b0 + b), (uint32_t)v, 1u);
        int tok = inverse_cdf(w, V, R, u2, &margin);
        if (margin < CDF_WINDOW)
            flags[b] |= FLAG_CDF_NEAR_BOUNDARY;
        int d = depth[v];
        for (int w = v, s = d; s >= 0; --s) {
            if (out_path)
                out_path[(int64_t)b * W + s] = w;
            if (s >= 1)
                out_tokens[(int64_t)b * W + s - 1] = node_tokens[(int64_t)b * N + w];
            w = parent[w];
        }
        out_tokens[(int64_t)b * W + d] = tok;
        accepted_len[b] = d;
    }
    free(depth);
    free(nchild);
    free(l);
    free(p);
    free(q);
    free(r);
    return 0;
}

/* Enumeration mode for the tree rule: for one sequence with fixed rows and fixed tokens,
 * prob[v * V + j] = P(the walk ends at node v and the final token is j), each uniform
 * replaced by its branch weights.  Logits fp64 [N][V].  Returns -1 on an invalid input. */
int oracle_exact_probs_tree(const double *t_logits, const double *d_logits, const int32_t *parent,
                            const int32_t *tokens, int N, int V, double T, int without_replacement,
                            double *prob)
{
    size_t rowsz = sizeof(double) * (size_t)V;
    int *depth = (int *)malloc(sizeof(int) * (size_t)N);
    double *reach = (double *)malloc(sizeof(double) * (size_t)N);
    double *p = (double *)malloc(rowsz);
    double *q = (double *)malloc(rowsz);
    double *r = (double *)malloc(rowsz);
    int rc = 0;
    if (!depth || !reach || !p || !q || !r || !tree_depths(parent, N, N, depth)) {
        rc = -1;
        goto done;
    }
    for (int j = 0; j < N * V; ++j)
        prob[j] = 0.0;
    for (int v = 0; v < N; ++v)
        reach[v] = v == 0 ? 1.0 : 0.0;
    for (int v = 0; v < N; ++v) { /* parents come before children */
        int has_child = 0;
        for (int c = v + 1; c < N; ++c)
            has_child |= parent[c] == v;
        if (softmax_row(t_logits + (size_t)v * V, V, T, p, NULL, NULL) != 0 ||
            (has_child && softmax_row(d_logits + (size_t)v * V, V, T, q, NULL, NULL) != 0)) {
            rc = -1;
            goto done;
        }
        double rest = 1.0; /* probability that the children tested so far were all rejected */
        for (int c = v + 1; c < N; ++c) {
            if (parent[c] != v)
                continue;
            int x = tokens[c];
            if (x < 0 || x >= V) {
                rc = -1;
                goto done;
            }
            double a = accept_probability(p[x], q[x]);
            reach[c] += reach[v] * rest * a;
            rest *= 1.0 - a;
            int fell_back = 0;
            reject_update(p, q, V, x, without_replacement, r, &fell_back);
        }
        for (int j = 0; j < V; ++j)
            prob[(size_t)v * V + j] += reach[v] * rest * p[j];
    }
done:
    free(depth);
    free(reach);
    free(p);
    free(q);
    free(r);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* Typical acceptance [SD "Medusa" paragraph ("accepts any token whose target probability
 * exceeds a threshold") and the closing note on typical acceptance ("a threshold that
 * scales with the step's entropy"; not distribution-preserving)].  The pages fix neither
 * the form nor the constants; the reading taken:
 *   p_i   = softmax(t_i / T)                                   (rows i = 0 .. gamma)
 *   H_i   = -sum_j p_i(j) ln p_i(j)                            (0 ln 0 = 0)
 *   tau_i = min(epsilon, delta * exp(-H_i))                    (exp(-H): 1 / perplexity)
 *   draft x_i is accepted iff p_i(x_i) > tau_i, left to right; the first failure k ends the
 *   prefix (k = gamma if none fails) and the token at k is drawn from p_k itself (no
 *   residual: the rule does not preserve the target law anyway), by the inverse CDF with
 *   u' = U(b, k, purpose 1).
 * Rows are read as the rule needs them (0 .. k): a bad row past the stop does not count.
 * A token outside [0, V) or a row read that is not a distribution gives -1.
 * Outputs as oracle_verify_sample; entropy [B][gamma+1] (or NULL): H_i of the rows read,
 * NAN elsewhere.  Flags: FLAG_ACCEPT_NEAR_THRESHOLD when |p - tau| < 1e-5 max(p, tau) in a
 * test performed, FLAG_CDF_NEAR_BOUNDARY as for sampling.                              */
/* ------------------------------------------------------------------------------------ */
int oracle_verify_typical(const void *target, int64_t t_batch_stride, int64_t t_row_stride,
                          int dtype, int B, int b0, int gamma, int V, const int32_t *draft_tokens,
                          double T, double epsilon, double delta, uint64_t seed, uint64_t offset,
                          int32_t *accepted_len, int32_t *out_tokens, int32_t *flags,
                          double *entropy)
{
    double *l = (double *)malloc(sizeof(double) * (size_t)V);
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    if (!l || !p) {
        free(l);
        free(p);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        int32_t *out = out_tokens + (int64_t)b * (gamma + 1);
        const int32_t *x = draft_tokens + (int64_t)b * gamma;
        for (int i = 0; i <= gamma; ++i) {
            out[i] = -1;
            if (entropy)
                entropy[(int64_t)b * (gamma + 1) + i] = NAN;
        }
        accepted_len[b] = -1;
        flags[b] = 0;
        int ok = 1;
        for (int i = 0; i < gamma && ok; ++i)
            ok = x[i] >= 0 && x[i] < V;
        if (!ok)
            continue;
        int k = -1;
        for (int i = 0; i <= gamma; ++i) {
            load_row(target, dtype, (int64_t)b * t_batch_stride + (int64_t)i * t_row_stride, V, l);
            if (softmax_row(l, V, T, p, NULL, NULL) != 0) {
                ok = 0;
                break;
            }
            double H = 0.0;
            for (int j = 0; j < V; ++j)
                if (p[j] > 0.0)
                    H -= p[j] * log(p[j]);
            if (entropy)
                entropy[(int64_t)b * (gamma + 1) + i] = H;
            if (i == gamma) {
                k = gamma;
                break;
            }
            double tau = delta * exp(-H);
            if (epsilon < tau)
                tau = epsilon;
            double px = p[x[i]];
            double big = px > tau ? px : tau;
            if (fabs(px - tau) < ACCEPT_WINDOW * big)
                flags[b] |= FLAG_ACCEPT_NEAR_THRESHOLD;
            if (!(px > tau)) {
                k = i;
                break;
            }
        }
        if (!ok) {
            flags[b] = 0;
            continue;
        }
        /* p holds p_k: the final token from it */
        double R = 0.0, margin = 0.0;
        for (int j = 0; j < V; ++j)
            R += p[j];
        double u2 = oracle_uniform(seed, offset, (uint32_t)(b0 + b), (uint32_t)k, 1u);
        int tok = inverse_cdf(p, V, R, u2, &margin);
        if (margin < CDF_WINDOW)
            flags[b] |= FLAG_CDF_NEAR_BOUNDARY;
        for (int i = 0; i < k; ++i)
            out[i] = x[i];
        out[k] = tok;
        accepted_len[b] = k;
    }
    free(l);
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Prompt-lookup (n-gram) drafting [MS lookup_draft; SD Exercise 4 ngram_draft].
 * history: [B][stride] tokens, len[b] of them valid.  For each sequence:
 *   tail  = its last n tokens;
 *   match = the largest i in [0, len - n - 1] with history[i + t] == tail[t] for every t
 *           (the most recent EARLIER occurrence; the continuation starts at i + n <= len - 1);
 *   drafts[m] = history[match + n + m] for m = 0, 1, ... while match + n + m < len, at most k;
 *   pad != 0 (Exercise 4's fallback): the remaining slots, or all k when there is no match,
 *           repeat the last token, so k tokens are always proposed (for len >= 1).
 * count[b] = the number of drafts; unused slots are -1.  Exercise 4 is n = 1, pad = 1;
 * lookup_draft is pad = 0 (n = 3, k = 4 in the page's example).                        */
/* ------------------------------------------------------------------------------------ */
int oracle_ngram_draft(const int32_t *history, int64_t stride, const int32_t *len, int B, int n, int k, int pad,
                       int32_t *drafts, int32_t *count)
{
    if (n < 1 || k < 0)
        return -1;
    for (int b = 0; b < B; ++b) {
        const int32_t *h = history + (int64_t)b * stride;
        int L = len[b];
        int32_t *out = drafts + (int64_t)b * k;
        for (int m = 0; m < k; ++m)
            out[m] = -1;
        count[b] = 0;
        int match = -1;
        for (int i = L - n - 1; i >= 0 && match < 0; --i) { /* right to left: the first hit is the latest */
            int same = 1;
            for (int t = 0; t < n && same; ++t)
                same = h[i + t] == h[L - n + t];
            if (same)
                match = i;
        }
        int c = 0;
        if (match >= 0)
            for (; c < k && match + n + c < L; ++c)
                out[c] = h[match + n + c];
        if (pad && L >= 1)
            for (; c < k; ++c)
                out[c] = h[L - 1];
        count[b] = c;
    }
    return 0;
}
