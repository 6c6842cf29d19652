/*
 * oracle.c -- plain, slow fp64 CPU oracle for tile-sparse masked softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
 * bench's CPU-baseline leg call it to produce expected values; the product
 * path (the CUDA library) never links, loads or calls it, and this file shares
 * no header, table or helper with it.
 *
 * What it computes is the plain definition that the pages' method reaches
 * exactly (up to rounding order):
 *
 *  - the mask M[i][j] of a mask program, evaluated element by element
 *    (mask_mod hook: speedrun notes "FlexAttention", code block after the
 *    Context paragraph; tutorial "The two hooks: score_mod and mask_mod",
 *    Pattern 1 document masking, Pattern 2 sliding window with sinks, and the
 *    and_masks / or_masks composition in Pattern 3);
 *  - for caller-chosen tiles (tutorial, opening section: sparse patterns that
 *    attend only to a selected subset of blocks; "Decoding and paged KV
 *    caches": BlockMask.from_kv_blocks), the mask those tiles leave: a pair is
 *    visible when its tile is listed as full, or listed as partial and the
 *    program holds there, and never when its tile is not listed;
 *  - the tile classes of a BLOCK x BLOCK grid by brute force: a tile is EMPTY
 *    when no in-range entry is visible, FULL when every one is, PARTIAL
 *    otherwise (tutorial, "The two hooks": empty / partially masked / full
 *    blocks; speedrun notes, tile-summary paragraph);
 *  - exact softmax attention over the visible set V_i = { j : M[i][j] }:
 *      x_ij   = scale * (q_i . k_j)
 *      s_ij   = score_mod(x_ij, h, i, j)           (tutorial Pattern 3)
 *      out_i  = sum_{j in V_i} exp(s_ij - LSE_i) v_j
 *      LSE_i  = log sum_{j in V_i} exp(s_ij)       (natural log)
 *    A row with V_i empty has out_i = 0 and LSE_i = -inf.
 *  - the gradients of L = sum(out * dO) with respect to q, k and v through
 *    the softmax and the score_mod (tutorial Pattern 3: both score mods are
 *    differentiable and the backward is fused):
 *      P_ij   = exp(s_ij - LSE_i)
 *      dP_ij  = dO_i . v_j
 *      dS_ij  = P_ij (dP_ij - sum_{k in V_i} P_ik dP_ik) * ds_ij/dx_ij
 *      dq_i   = scale * sum_j dS_ij k_j
 *      dk_j   = scale * sum_i dS_ij q_i
 *      dv_j   = sum_i P_ij dO_i
 *
 * Score mods: none (s = x); soft-cap s = c tanh(x / c), ds/dx = 1 - tanh^2(x / c);
 * ALiBi s = x - slope_h (i - j), ds/dx = 1; a learned relative-position bias
 * s = x + bias_h[clamp(i - j - d0, 0, L - 1)], ds/dx = 1: one table entry per
 * query-minus-key distance from d0 to d0 + L - 1, distances outside that range
 * taking the nearest end entry.
 *
 *  - the gradient of L with respect to the score mod's parameter (tutorial
 *    Pattern 3: a learned relative-position bias trains through the fused
 *    backward):  dL/dparam = sum_{i, j in V_i} P_ij (dP_ij - Delta_i) ds_ij/dparam
 *    with ds/dslope_h = -(i - j) for ALiBi and ds/dc = tanh(x/c) - (x/c)(1 - tanh^2(x/c))
 *    for the soft-cap; for the bias table, dL/dbias_h[t] is that sum over the
 *    pairs whose distance maps to entry t (ds/dbias_h[t] = 1 there, 0 elsewhere).
 *
 * All arithmetic is double precision on the bf16-rounded inputs that the
 * caller widens to double.  Loops are parallel over independent rows or
 * columns only (OpenMP); there is no tiling, fusion or reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Mask program node kinds (this file's own numbering). */
enum {
    OR_TRUE = 0,    /* every pair visible                              */
    OR_CAUSAL = 1,  /* q_idx >= kv_idx                                 */
    OR_SAME_DOC = 2,/* doc[q_idx] == doc[kv_idx]                       */
    OR_WINDOW = 3,  /* q_idx - kv_idx < arg                            */
    OR_SINK = 4,    /* kv_idx < arg                                    */
    OR_PREFIX = 5,  /* kv_idx < arg (prefix length of this batch row)  */
    OR_AND = 6,
    OR_OR = 7
};

enum { OR_SCORE_NONE = 0, OR_SCORE_SOFTCAP = 1, OR_SCORE_ALIBI = 2, OR_SCORE_RELBIAS = 3 };

/* A score mod for one head: the soft-cap c or ALiBi slope in `param`; the
 * bias table of this head (len entries, entry 0 at distance d0) for RELBIAS. */
typedef struct {
    int32_t op;
    double param;
    const double *bias;
    int64_t d0, len;
} or_score;

/* The bias table entry of the pair at query position i and key j. */
static int64_t bias_entry(const or_score *sc, int64_t i, int64_t j)
{
    int64_t t = i - j - sc->d0;
    if (t < 0) t = 0;
    if (t > sc->len - 1) t = sc->len - 1;
    return t;
}

typedef struct {
    int32_t n;             /* number of nodes (postfix order)            */
    int32_t op[16];
    int64_t arg[16];       /* window W, sink count or prefix length      */
    const int32_t *doc;    /* document id of each position of this batch row */
    /* Optional selection of tiles, row-major [nq][sel_nkv] of sel_block x
     * sel_block tiles: 0 not listed, 1 listed partial, 2 listed full. */
    const int8_t *sel;
    int64_t sel_block, sel_nkv;
    /* Position of query row 0 in the sequence the program describes: row i is
     * position i + q_off for CAUSAL, WINDOW, SAME_DOC and ALiBi (decoding new
     * tokens at the end of a cache). */
    int64_t q_off;
} or_program;

/* The program's value at (i, j), evaluated with an explicit stack. */
static int program_at(const or_program *p, int64_t row, int64_t j)
{
    const int64_t i = row + p->q_off;  /* the query's position */
    int st[16];
    int sp = 0;
    for (int n = 0; n < p->n; ++n) {
        switch (p->op[n]) {
        case OR_TRUE:     st[sp++] = 1; break;
        case OR_CAUSAL:   st[sp++] = (i >= j); break;
        case OR_SAME_DOC: st[sp++] = (p->doc[i] == p->doc[j]); break;
        case OR_WINDOW:   st[sp++] = (i - j < p->arg[n]); break;
        case OR_SINK:     st[sp++] = (j < p->arg[n]); break;
        case OR_PREFIX:   st[sp++] = (j < p->arg[n]); break;
        case OR_AND:      sp -= 1; st[sp - 1] = st[sp - 1] && st[sp]; break;
        case OR_OR:       sp -= 1; st[sp - 1] = st[sp - 1] || st[sp]; break;
        default:          return 0;
        }
    }
    return st[0];
}

/* M[i][j]: the program's value, restricted by the tile selection if any. */
static int mask_at(const or_program *p, int64_t i, int64_t j)
{
    if (p->sel != NULL) {
        const int8_t c = p->sel[(i / p->sel_block) * p->sel_nkv + j / p->sel_block];
        if (c == 2)
            return 1;
        if (c != 1)
            return 0;
    }
    return program_at(p, i, j);
}

/* Explicit [q_len][kv_len] byte mask. */
void oracle_mask_dense(const or_program *p, int64_t q_len, int64_t kv_len, uint8_t *M)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < q_len; ++i)
        for (int64_t j = 0; j < kv_len; ++j)
            M[i * kv_len + j] = (uint8_t)mask_at(p, i, j);
}

/* Brute-force tile classes: 0 EMPTY, 1 PARTIAL, 2 FULL, row-major [nq][nkv].
 * The last tile row / column may be cut short by q_len / kv_len; only
 * in-range entries count. */
void oracle_classify_tiles(const or_program *p, int64_t q_len, int64_t kv_len, int32_t block,
                           int8_t *cls)
{
    const int64_t nq = (q_len + block - 1) / block;
    const int64_t nkv = (kv_len + block - 1) / block;
    #pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t I = 0; I < nq; ++I) {
        for (int64_t J = 0; J < nkv; ++J) {
            const int64_t i0 = I * block, i1 = (i0 + block < q_len) ? i0 + block : q_len;
            const int64_t j0 = J * block, j1 = (j0 + block < kv_len) ? j0 + block : kv_len;
            int64_t visible = 0;
            for (int64_t i = i0; i < i1; ++i)
                for (int64_t j = j0; j < j1; ++j)
                    visible += mask_at(p, i, j);
            const int64_t area = (i1 - i0) * (j1 - j0);
            cls[I * nkv + J] = (int8_t)(visible == 0 ? 0 : (visible == area ? 2 : 1));
        }
    }
}

static double dot(const double *a, const double *b, int D)
{
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += a[d] * b[d];
    return s;
}

/* s = score_mod(x) and ds/dx for one pair (i the query's position). */
static double score_mod(const or_score *sc, double x, int64_t i, int64_t j, double *dsdx)
{
    if (sc->op == OR_SCORE_SOFTCAP) {
        const double t = tanh(x / sc->param);
        if (dsdx) *dsdx = 1.0 - t * t;
        return sc->param * t;
    }
    if (dsdx) *dsdx = 1.0;
    if (sc->op == OR_SCORE_ALIBI)
        return x - sc->param * (double)(i - j);
    if (sc->op == OR_SCORE_RELBIAS)
        return x + sc->bias[bias_entry(sc, i, j)];
    return x;
}

/* ds/dparam for one pair: the soft-cap c or the ALiBi slope (0 without a
 * scalar parameter; the bias table has its own gradient below). */
static double score_mod_dparam(const or_score *sc, double x, int64_t i, int64_t j)
{
    if (sc->op == OR_SCORE_SOFTCAP) {
        const double t = tanh(x / sc->param);
        return t - (x / sc->param) * (1.0 - t * t);
    }
    if (sc->op == OR_SCORE_ALIBI)
        return -(double)(i - j);
    return 0.0;
}

static or_score make_score(int32_t op, double param, const double *bias, int64_t d0, int64_t len)
{
    or_score sc;
    sc.op = op;
    sc.param = param;
    sc.bias = bias;
    sc.d0 = d0;
    sc.len = len;
    return sc;
}

/*
 * Forward for one (b, h): q [q_len][D], k, v [kv_len][D] (row-major doubles).
 * rows: the query rows to compute (NULL = all q_len rows, in order); out is
 * [n_rows][D] and lse [n_rows].  score_param is the soft-cap c or the ALiBi
 * slope of this head; bias / bias_d0 / bias_len this head's bias table (RELBIAS).
 */
void oracle_forward_head(const double *q, const double *k, const double *v,
                         int64_t q_len, int64_t kv_len, int32_t D,
                         const or_program *p, int32_t score_op, double score_param, double scale,
                         const int64_t *rows, int64_t n_rows, double *out, double *lse,
                         const double *bias, int64_t bias_d0, int64_t bias_len)
{
    const or_score sc_ = make_score(score_op, score_param, bias, bias_d0, bias_len);
    const or_score *sc = &sc_;
    if (rows == NULL) n_rows = q_len;
    #pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        uint8_t *vis = (uint8_t *)malloc((size_t)(kv_len > 0 ? kv_len : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < n_rows; ++r) {
            const int64_t i = rows ? rows[r] : r;
            const double *qi = q + i * D;
            double m = -INFINITY;
            int64_t nvis = 0;
            for (int64_t j = 0; j < kv_len; ++j) {
                vis[j] = (uint8_t)mask_at(p, i, j);
                if (!vis[j]) continue;
                const double x = scale * dot(qi, k + j * D, D);
                s[j] = score_mod(sc, x, i + p->q_off, j, NULL);
                if (s[j] > m) m = s[j];
                ++nvis;
            }
            double *o = out + r * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (nvis == 0) {
                lse[r] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int64_t j = 0; j < kv_len; ++j) {
                if (!vis[j]) continue;
                const double e = exp(s[j] - m);
                l += e;
                for (int d = 0; d < D; ++d) o[d] += e * v[j * D + d];
            }
            for (int d = 0; d < D; ++d) o[d] /= l;
            lse[r] = m + log(l);
        }
        free(s);
        free(vis);
    }
}

/*
 * Backward for one (b, h).  dout [q_len][D].  Computes dq for `rows`
 * (NULL = all, dq [n_rows][D]) and dk, dv for `cols` (NULL = all,
 * [n_cols][D]).  LSE_i and sum_k P_ik dP_ik are computed for every row
 * first, since any column may need them.  lse_all / delta_all, when not
 * NULL, receive those per-row values ([q_len]).
 */
void oracle_backward_head(const double *q, const double *k, const double *v, const double *dout,
                          int64_t q_len, int64_t kv_len, int32_t D,
                          const or_program *p, int32_t score_op, double score_param, double scale,
                          const int64_t *rows, int64_t n_rows, const int64_t *cols, int64_t n_cols,
                          double *dq, double *dk, double *dv, double *lse_all, double *delta_all,
                          const double *bias, int64_t bias_d0, int64_t bias_len)
{
    const or_score sc_ = make_score(score_op, score_param, bias, bias_d0, bias_len);
    const or_score *sc = &sc_;
    double *lse = (double *)malloc(sizeof(double) * (size_t)(q_len > 0 ? q_len : 1));
    double *delta = (double *)malloc(sizeof(double) * (size_t)(q_len > 0 ? q_len : 1));
    if (rows == NULL) n_rows = q_len;
    if (cols == NULL) n_cols = kv_len;

    /* Row statistics for every row: LSE_i and sum_j P_ij dP_ij. */
    #pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        uint8_t *vis = (uint8_t *)malloc((size_t)(kv_len > 0 ? kv_len : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < q_len; ++i) {
            double m = -INFINITY;
            int64_t nvis = 0;
            for (int64_t j = 0; j < kv_len; ++j) {
                vis[j] = (uint8_t)mask_at(p, i, j);
                if (!vis[j]) continue;
                const double x = scale * dot(q + i * D, k + j * D, D);
                s[j] = score_mod(sc, x, i + p->q_off, j, NULL);
                if (s[j] > m) m = s[j];
                ++nvis;
            }
            if (nvis == 0) {
                lse[i] = -INFINITY;
                delta[i] = 0.0;
                continue;
            }
            double l = 0.0;
            for (int64_t j = 0; j < kv_len; ++j)
                if (vis[j]) l += exp(s[j] - m);
            lse[i] = m + log(l);
            double acc = 0.0;
            for (int64_t j = 0; j < kv_len; ++j) {
                if (!vis[j]) continue;
                const double P = exp(s[j] - lse[i]);
                acc += P * dot(dout + i * D, v + j * D, D);
            }
            delta[i] = acc;
        }
        free(s);
        free(vis);
    }

    /* dq_i = scale * sum_j dS_ij k_j */
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *g = dq + r * D;
        for (int d = 0; d < D; ++d) g[d] = 0.0;
        if (lse[i] == -INFINITY) continue;
        for (int64_t j = 0; j < kv_len; ++j) {
            if (!mask_at(p, i, j)) continue;
            double dsdx;
            const double x = scale * dot(q + i * D, k + j * D, D);
            const double sij = score_mod(sc, x, i + p->q_off, j, &dsdx);
            const double P = exp(sij - lse[i]);
            const double dP = dot(dout + i * D, v + j * D, D);
            const double dS = P * (dP - delta[i]) * dsdx;
            for (int d = 0; d < D; ++d) g[d] += scale * dS * k[j * D + d];
        }
    }

    /* dk_j = scale * sum_i dS_ij q_i ; dv_j = sum_i P_ij dO_i */
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t c = 0; c < n_cols; ++c) {
        const int64_t j = cols ? cols[c] : c;
        double *gk = dk + c * D;
        double *gv = dv + c * D;
        for (int d = 0; d < D; ++d) { gk[d] = 0.0; gv[d] = 0.0; }
        for (int64_t i = 0; i < q_len; ++i) {
            if (!mask_at(p, i, j)) continue;
            double dsdx;
            const double x = scale * dot(q + i * D, k + j * D, D);
            const double sij = score_mod(sc, x, i + p->q_off, j, &dsdx);
            const double P = exp(sij - lse[i]);
            const double dP = dot(dout + i * D, v + j * D, D);
            const double dS = P * (dP - delta[i]) * dsdx;
            for (int d = 0; d < D; ++d) {
                gk[d] += scale * dS * q[i * D + d];
                gv[d] += P * dout[i * D + d];
            }
        }
    }

    if (lse_all) memcpy(lse_all, lse, sizeof(double) * (size_t)q_len);
    if (delta_all) memcpy(delta_all, delta, sizeof(double) * (size_t)q_len);
    free(lse);
    free(delta);
}

/*
 * dL/d(score parameter) for one (b, h): the sum over every visible pair of
 * P_ij (dP_ij - Delta_i) ds_ij/dparam, with LSE_i and Delta_i = sum_j P_ij dP_ij
 * of each row computed first (row by row, as in the backward above).
 */
double oracle_score_param_grad_head(const double *q, const double *k, const double *v, const double *dout,
                                    int64_t q_len, int64_t kv_len, int32_t D,
                                    const or_program *p, int32_t score_op, double score_param, double scale,
                                    const double *bias, int64_t bias_d0, int64_t bias_len)
{
    const or_score sc_ = make_score(score_op, score_param, bias, bias_d0, bias_len);
    const or_score *sc = &sc_;
    double total = 0.0;
    #pragma omp parallel reduction(+ : total)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        double *x = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        uint8_t *vis = (uint8_t *)malloc((size_t)(kv_len > 0 ? kv_len : 1));
        #pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < q_len; ++i) {
            double m = -INFINITY;
            int64_t nvis = 0;
            for (int64_t j = 0; j < kv_len; ++j) {
                vis[j] = (uint8_t)mask_at(p, i, j);
                if (!vis[j]) continue;
                x[j] = scale * dot(q + i * D, k + j * D, D);
                s[j] = score_mod(sc, x[j], i + p->q_off, j, NULL);
                dp[j] = dot(dout + i * D, v + j * D, D);
                if (s[j] > m) m = s[j];
                ++nvis;
            }
            if (nvis == 0) continue;
            double l = 0.0;
            for (int64_t j = 0; j < kv_len; ++j)
                if (vis[j]) l += exp(s[j] - m);
            const double lse = m + log(l);
            double delta = 0.0;
            for (int64_t j = 0; j < kv_len; ++j)
                if (vis[j]) delta += exp(s[j] - lse) * dp[j];
            for (int64_t j = 0; j < kv_len; ++j) {
                if (!vis[j]) continue;
                const double P = exp(s[j] - lse);
                total += P * (dp[j] - delta) * score_mod_dparam(sc, x[j], i + p->q_off, j);
            }
        }
        free(s);
        free(x);
        free(dp);
        free(vis);
    }
    return total;
}

/*
 * dL/dbias_h[t] for one (b, h) under the RELBIAS score mod, ADDED into
 * grad[bias_len]: for every visible pair, P_ij (dP_ij - Delta_i) goes to the
 * entry its distance maps to.  Rows are taken one at a time (no threads, so
 * that the sums need no reduction across threads).
 */
void oracle_bias_grad_head(const double *q, const double *k, const double *v, const double *dout,
                           int64_t q_len, int64_t kv_len, int32_t D, const or_program *p,
                           const double *bias, int64_t bias_d0, int64_t bias_len, double scale, double *grad)
{
    const or_score sc_ = make_score(OR_SCORE_RELBIAS, 0.0, bias, bias_d0, bias_len);
    const or_score *sc = &sc_;
    double *s = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
    uint8_t *vis = (uint8_t *)malloc((size_t)(kv_len > 0 ? kv_len : 1));
    for (int64_t i = 0; i < q_len; ++i) {
        double m = -INFINITY;
        int64_t nvis = 0;
        for (int64_t j = 0; j < kv_len; ++j) {
            vis[j] = (uint8_t)mask_at(p, i, j);
            if (!vis[j]) continue;
            const double x = scale * dot(q + i * D, k + j * D, D);
            s[j] = score_mod(sc, x, i + p->q_off, j, NULL);
            dp[j] = dot(dout + i * D, v + j * D, D);
            if (s[j] > m) m = s[j];
            ++nvis;
        }
        if (nvis == 0) continue;
        double l = 0.0;
        for (int64_t j = 0; j < kv_len; ++j)
            if (vis[j]) l += exp(s[j] - m);
        const double lse = m + log(l);
        double delta = 0.0;
        for (int64_t j = 0; j < kv_len; ++j)
            if (vis[j]) delta += exp(s[j] - lse) * dp[j];
        for (int64_t j = 0; j < kv_len; ++j) {
            if (!vis[j]) continue;
            grad[bias_entry(sc, i + p->q_off, j)] += exp(s[j] - lse) * (dp[j] - delta);
        }
    }
    free(s);
    free(dp);
    free(vis);
}
