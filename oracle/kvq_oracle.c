/*
 * kvq_oracle.c -- plain CPU oracle for the rate-adaptive KV-cache block
 * quantizer (ECASQ applied per cache block).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * CUDA path is compared against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it; the product path never does.
 * It shares no code, header, table or constant generator with the CUDA
 * library.
 *
 * Everything here is written for clarity, not speed: full sort of every block,
 * fp64 arithmetic, distortion and masses summed element by element from the
 * sorted block, an O(m^3 s) dynamic program over exact level counts, and a
 * sequential bisection.  Build flags: -O2 -ffp-contract=off (no FMA
 * contraction; the stochastic-rounding step must round every fp32 operation
 * on its own).
 *
 * Source: "Rate-adaptive KV-cache quantizer" (synthcore idea 2502),
 *   - "Mathematical statement": per-block problem, dual separability, the
 *     interpolation probabilities, conditional MSE and mean, entropy of the
 *     expected codepoint frequencies, subgradient update of lambda;
 *   - "Key formulas": the constrained objective, the Lagrangian, the
 *     probability / distortion formulas, the lambda update;
 *   - "Implementation notes": blocks of one head x 32 tokens (or a feature
 *     group), candidate alphabet from min / max / quantiles, D_r from interval
 *     statistics, H_r from expected (not sampled) frequencies, one global
 *     lambda, a small DP over ordered codepoints, store codebook + symbols.
 * Readings where the page leaves a step open are listed at each function.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KVQO_M 17          /* candidate levels per block (order statistics) */
#define KVQO_SMAX 16       /* codes are stored in 4 bits */

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 decode / encode (exact).                               */
/* ------------------------------------------------------------------------ */

/* binary16 bit pattern -> double, exactly.  -0 is returned as +0 (the method
 * compares values, and -0 == +0). */
double kvqo_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);
    if (v == 0.0)
        return 0.0;
    return sign ? -v : v;
}

/* double that is exactly a binary16 value -> its bit pattern.  Returns 0 and
 * sets *ok = 0 if v is not exactly representable. */
uint16_t kvqo_double_to_f16(double v, int *ok)
{
    *ok = 1;
    if (v == 0.0)
        return 0;
    if (isnan(v)) { *ok = 0; return 0x7e00; }
    uint16_t sign = v < 0 ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7c00;
    int e;
    double fr = frexp(a, &e);          /* a = fr * 2^e, fr in [0.5, 1) */
    int eb = e - 1 + 15;               /* biased exponent of 1.xxx form */
    if (eb >= 31) { *ok = 0; return sign | 0x7c00; }
    if (eb <= 0) {                     /* subnormal: a = m * 2^-24 */
        double m = ldexp(a, 24);
        if (m != floor(m) || m >= 1024) { *ok = 0; }
        return sign | (uint16_t)m;
    }
    double m = ldexp(fr * 2.0 - 1.0, 10);   /* 10-bit fraction */
    if (m != floor(m)) *ok = 0;
    return sign | (uint16_t)(eb << 10) | (uint16_t)m;
}

/* ------------------------------------------------------------------------ */
/* Block partition ("Implementation notes": one block per attention head per */
/* 32 tokens, or per head and feature group).                               */
/* Input is [S, T, D] row-major fp16.  Block b = (h, tb, g) in row-major     */
/* order over (h, tb, g); inside a block, element e = (t - 32 tb) * G +      */
/* (f - g G).                                                                */
/* ------------------------------------------------------------------------ */

int64_t kvqo_num_blocks(int64_t S, int64_t T, int D, int G)
{
    return S * (T / 32) * (int64_t)(D / G);
}

/* flat [S,T,D] index of element e of block b */
int64_t kvqo_flat_index(int64_t T, int D, int G, int64_t b, int e)
{
    int64_t nG = D / G, nTB = T / 32;
    int64_t g = b % nG;
    int64_t tb = (b / nG) % nTB;
    int64_t h = b / (nG * nTB);
    int64_t t = 32 * tb + e / G;
    int64_t f = g * G + e % G;
    return (h * T + t) * D + f;
}

/* ------------------------------------------------------------------------ */
/* Candidate alphabet ("Implementation notes": build a candidate alphabet    */
/* from the block's minimum, maximum and quantiles).                         */
/* Reading: 17 order statistics at 0-based sorted ranks                      */
/* r_j = floor((j (d-1) + 8) / 16), j = 0..16 (rank j(d-1)/16 rounded half   */
/* up); r_0 = 0 is the minimum and r_16 = d-1 the maximum.  Equal values are */
/* merged, giving m' <= 17 strictly increasing levels.                       */
/* ------------------------------------------------------------------------ */

/* ------------------------------------------------------------------------ */
/* Weights ("Implementation notes": D_r may be weighted by the attention     */
/* sensitivity measured on a calibration batch).                             */
/* Reading: the caller gives one weight w_e >= 0 per entry (fp32, the same   */
/* [S,T,D] layout as x; NULL = every weight 1) and the block's distortion    */
/* becomes D_r = sum_e w_e E[(hat x_e - x_e)^2]; the rate H_r stays the      */
/* entropy of the unweighted expected codepoint frequencies, because it      */
/* counts the stored symbols.  A weight that is negative, NaN or infinite is */
/* reported (flag bit 1) and counted as 0.                                   */
/* ------------------------------------------------------------------------ */

typedef struct { double v, w; } kvqo_entry_t;

static int cmp_entry(const void *a, const void *b)
{
    double x = ((const kvqo_entry_t *)a)->v, y = ((const kvqo_entry_t *)b)->v;
    return (x > y) - (x < y);
}

/* values (sorted) of block b with their weights carried along; returns bit 0
 * if any value is NaN or infinite, bit 1 if any weight is invalid */
static int block_sorted(const uint16_t *x, const float *wt, int64_t T, int D,
                        int G, int64_t b, double *v, double *wv)
{
    int d = 32 * G, bad = 0;
    kvqo_entry_t *ent = (kvqo_entry_t *)malloc(sizeof(kvqo_entry_t) * d);
    for (int e = 0; e < d; e++) {
        int64_t f = kvqo_flat_index(T, D, G, b, e);
        double xv = kvqo_f16_to_double(x[f]);
        double w = wt ? (double)wt[f] : 1.0;
        if (!isfinite(xv)) { bad |= 1; xv = 0.0; }
        if (!(w >= 0.0) || !isfinite(w)) { bad |= 2; w = 0.0; }
        ent[e].v = xv;
        ent[e].w = w;
    }
    qsort(ent, (size_t)d, sizeof(kvqo_entry_t), cmp_entry);
    for (int e = 0; e < d; e++) {
        v[e] = ent[e].v;
        if (wv) wv[e] = ent[e].w;
    }
    free(ent);
    return bad;
}

static int candidates_from_sorted(const double *v, int d, double *c)
{
    int mp = 0;
    for (int j = 0; j < KVQO_M; j++) {
        int64_t r = ((int64_t)j * (d - 1) + 8) / 16;
        double val = v[r];
        if (mp == 0 || val != c[mp - 1])
            c[mp++] = val;
    }
    return mp;
}

/* Atom statistics (the GPU summarises a block by these): atom p, p = 0..m'-2,
 * holds the elements with c_p <= x < c_{p+1}; the last atom also holds the
 * elements equal to the maximum.  Per atom: n, s1 = sum(x - c_p),
 * t1 = sum(c_{p+1} - x), e = sum((x - c_p)(c_{p+1} - x)); with weights wt
 * (non-NULL) every sum is weighted: n = sum w, s1 = sum w (x - c_p), ...
 * Outputs for blocks [b0, b0+nb): cand[nb][17] (padded with the maximum),
 * mprime[nb], atoms[nb][16][4], flags[nb] (bit 0 non-finite value, bit 1
 * invalid weight). */
void kvqo_stats(const uint16_t *x, const float *wt, int64_t S, int64_t T,
                int D, int G, int64_t b0, int64_t nb, double *cand,
                int32_t *mprime, double *atoms, int32_t *nonfinite)
{
    (void)S;
    int d = 32 * G;
#pragma omp parallel
    {
        double *v = (double *)malloc(sizeof(double) * d);
        double *wv = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < nb; i++) {
            int64_t b = b0 + i;
            double c[KVQO_M];
            nonfinite[i] = block_sorted(x, wt, T, D, G, b, v, wv);
            int mp = candidates_from_sorted(v, d, c);
            mprime[i] = mp;
            for (int j = 0; j < KVQO_M; j++)
                cand[i * KVQO_M + j] = j < mp ? c[j] : c[mp - 1];
            double *a = atoms + i * 16 * 4;
            for (int j = 0; j < 16 * 4; j++) a[j] = 0.0;
            if (mp < 2) continue;
            for (int e = 0; e < d; e++) {
                int p = 0;
                while (p + 1 <= mp - 2 && v[e] >= c[p + 1]) p++;
                double y = v[e] - c[p], t = c[p + 1] - v[e], w = wv[e];
                a[p * 4 + 0] += w;
                a[p * 4 + 1] += w * y;
                a[p * 4 + 2] += w * t;
                a[p * 4 + 3] += w * y * t;
            }
        }
        free(v);
        free(wv);
    }
}

/* ------------------------------------------------------------------------ */
/* Interval quantities, straight from the definition ("Key formulas":        */
/* P(q_i | x) = (q_{i+1} - x)/(q_{i+1} - q_i), P(q_{i+1} | x) =              */
/* (x - q_i)/(q_{i+1} - q_i), conditional MSE (q_{i+1} - x)(x - q_i)).       */
/* For levels a = c_P < b = c_Q and the elements x of the block in [a, b)    */
/* (plus x == b when b is the maximum):                                      */
/*   Dpq[P][Q] = sum w (b - x)(x - a)        conditional MSE, weighted       */
/*   Mup[P][Q] = sum (x - a)/(b - a)         expected count sent to b        */
/*   Mdn[P][Q] = sum (b - x)/(b - a)         expected count sent to a        */
/* ------------------------------------------------------------------------ */

typedef struct {
    int d, mp;
    double wmax;                 /* largest weight of the block */
    double c[KVQO_M];
    double Dpq[KVQO_M][KVQO_M];
    double Mup[KVQO_M][KVQO_M];
    double Mdn[KVQO_M][KVQO_M];
} kvqo_block_t;

static void block_tables(const double *v, const double *wv, int d,
                         kvqo_block_t *B)
{
    B->d = d;
    B->mp = candidates_from_sorted(v, d, B->c);
    B->wmax = 0.0;
    for (int e = 0; e < d; e++)
        if (wv[e] > B->wmax) B->wmax = wv[e];
    memset(B->Dpq, 0, sizeof B->Dpq);
    memset(B->Mup, 0, sizeof B->Mup);
    memset(B->Mdn, 0, sizeof B->Mdn);
    int mp = B->mp;
    for (int P = 0; P < mp; P++)
        for (int Q = P + 1; Q < mp; Q++) {
            double a = B->c[P], b = B->c[Q], W = b - a;
            double Ds = 0, Us = 0, Ls = 0;
            for (int e = 0; e < d; e++) {
                double xv = v[e];
                int in = (xv >= a && xv < b) || (Q == mp - 1 && xv == b);
                if (!in) continue;
                Ds += wv[e] * ((b - xv) * (xv - a));
                Us += (xv - a) / W;
                Ls += (b - xv) / W;
            }
            B->Dpq[P][Q] = Ds;
            B->Mup[P][Q] = Us;
            B->Mdn[P][Q] = Ls;
        }
}

/* Entropy contribution of a codepoint with expected count M out of d
 * ("Mathematical statement": H_r = -sum_j pi_j log2 pi_j, pi_j the expected
 * frequency of codepoint j): h(M) = -M log2(M/d), so sum_j h(M_j) = d_r H_r. */
static double hterm(double M, int d)
{
    return M > 0.0 ? -M * log2(M / (double)d) : 0.0;
}

/* ------------------------------------------------------------------------ */
/* Per-block codebook choice ("Implementation notes": for each block choose  */
/* argmin_Q [D_r + lambda d_r H_r] by a small dynamic program over ordered   */
/* codepoints, k <= s; "Mathematical statement": |Q_r| <= s_r and            */
/* E[hat X] = X).                                                            */
/* Readings: Q is a subset of the m' candidates that contains the minimum    */
/* and the maximum (unbiased interpolation needs every x inside [q_0,        */
/* q_{k-1}]), 2 <= k <= s (k = 1 only when m' = 1).  Exact minimum over all  */
/* such subsets.  Ties: smaller objective, then fewer levels, then the       */
/* lexicographically smaller list of candidate indices.                      */
/* The DP state is (k, i, j): chains with exactly k levels whose last two    */
/* are candidates i < j; the entropy term of level j waits for the next      */
/* level, because its expected count gets Mup(i, j) from below and Mdn(j, l) */
/* from above.  The two best distinct chains are kept, for the tie gap.      */
/* ------------------------------------------------------------------------ */

typedef struct { double o1; uint32_t m1; double o2; uint32_t m2; } top2_t;

static int chain_better(double oa, uint32_t ma, double ob, uint32_t mb)
{
    if (oa != ob) return oa < ob;
    int ka = __builtin_popcount(ma), kb = __builtin_popcount(mb);
    if (ka != kb) return ka < kb;
    if (ma == mb) return 0;
    uint32_t dif = ma ^ mb, low = dif & (~dif + 1u);
    return (ma & low) != 0;
}

static void top2_insert(top2_t *t, double o, uint32_t m)
{
    if (chain_better(o, m, t->o1, t->m1)) {
        t->o2 = t->o1; t->m2 = t->m1;
        t->o1 = o; t->m1 = m;
    } else if (chain_better(o, m, t->o2, t->m2)) {
        t->o2 = o; t->m2 = m;
    }
}

/* D_r and d_r H_r of a given chain (mask over candidate indices), recomputed
 * from the interval tables. */
static void chain_cost(const kvqo_block_t *B, uint32_t mask, double *Dr,
                       double *Rr)
{
    int lev[KVQO_M], k = 0;
    for (int j = 0; j < B->mp; j++)
        if (mask >> j & 1u) lev[k++] = j;
    double D = 0, R = 0;
    if (k >= 2) {
        for (int i = 0; i + 1 < k; i++) D += B->Dpq[lev[i]][lev[i + 1]];
        for (int i = 0; i < k; i++) {
            double M = 0;
            if (i > 0) M += B->Mup[lev[i - 1]][lev[i]];
            if (i + 1 < k) M += B->Mdn[lev[i]][lev[i + 1]];
            R += hterm(M, B->d);
        }
    }
    *Dr = D;
    *Rr = R;
}

static void block_dp(const kvqo_block_t *B, int s, double lambda, int want2,
                     uint32_t *best_mask, double *best_obj, double *second_obj)
{
    int mp = B->mp, d = B->d;
    const double INF = INFINITY;
    if (mp == 1) {
        *best_mask = 1u; *best_obj = 0.0; *second_obj = INF;
        return;
    }
    int kmax = s < mp ? s : mp;
    static __thread top2_t F[KVQO_SMAX + 2][KVQO_M][KVQO_M];
    for (int k = 0; k <= kmax; k++)
        for (int i = 0; i < mp; i++)
            for (int j = 0; j < mp; j++) {
                F[k][i][j].o1 = INF; F[k][i][j].m1 = 0;
                F[k][i][j].o2 = INF; F[k][i][j].m2 = 0;
            }
    for (int j = 1; j < mp; j++) {
        double o = B->Dpq[0][j] + lambda * hterm(B->Mdn[0][j], d);
        top2_insert(&F[2][0][j], o, 1u | (1u << j));
    }
    for (int k = 2; k < kmax; k++)
        for (int i = 0; i < mp; i++)
            for (int j = i + 1; j < mp - 1; j++) {
                top2_t *src = &F[k][i][j];
                if (!(src->o1 < INF)) continue;
                for (int l = j + 1; l < mp; l++) {
                    double add = B->Dpq[j][l] +
                        lambda * hterm(B->Mup[i][j] + B->Mdn[j][l], d);
                    top2_insert(&F[k + 1][j][l], src->o1 + add,
                                src->m1 | (1u << l));
                    if (want2 && src->o2 < INF)
                        top2_insert(&F[k + 1][j][l], src->o2 + add,
                                    src->m2 | (1u << l));
                }
            }
    top2_t fin = {INF, 0, INF, 0};
    for (int k = 2; k <= kmax; k++)
        for (int i = 0; i < mp - 1; i++) {
            top2_t *t = &F[k][i][mp - 1];
            double e = lambda * hterm(B->Mup[i][mp - 1], d);
            if (t->o1 < INF) top2_insert(&fin, t->o1 + e, t->m1);
            if (want2 && t->o2 < INF) top2_insert(&fin, t->o2 + e, t->m2);
        }
    *best_mask = fin.m1;
    *best_obj = fin.o1;
    *second_obj = fin.o2;
}

/* Results for one block at one lambda. */
typedef struct {
    uint32_t mask;
    int k;
    double obj, obj2, Dr, Rr;
} kvqo_choice_t;

static void block_choose(const kvqo_block_t *B, int s, double lambda,
                         int want2, kvqo_choice_t *out)
{
    block_dp(B, s, lambda, want2, &out->mask, &out->obj, &out->obj2);
    out->k = __builtin_popcount(out->mask);
    chain_cost(B, out->mask, &out->Dr, &out->Rr);
}

/* ------------------------------------------------------------------------ */
/* Whole-tensor allocation with one global lambda ("Mathematical statement": */
/* minimise sum_r D_r s.t. sum_r d_r H_r <= B; the Lagrangian separates the  */
/* blocks, coupled only through lambda).                                     */
/* Reading of the lambda search (the page names none; taken here as a fixed  */
/* 40-step bisection): R(lambda) = sum_r d_r H_r summed in block order       */
/* in fp64, feasible iff R <= B.                                             */
/*   1. if R(0) <= B: lambda = 0.                                            */
/*   2. lo = 0, hi = max_r (c_max - c_min)^2 (times the block's largest      */
/*      weight when D_r is weighted); while R(hi) > B, hi *= 2, at           */
/*      most 30 times; still infeasible -> status 4 (infeasible), lambda =   */
/*      hi, and the allocation at hi is returned.                            */
/*   3. 40 steps: mid = 0.5 (lo + hi); R(mid) <= B ? hi = mid : lo = mid.    */
/*   4. lambda = hi (the feasible end).                                      */
/* Subgradient mode ("Key formulas": lambda <- max{0, lambda + eta (sum_r    */
/* d_r H_r - B)}): choose at the given lambda, return R and the updated      */
/* lambda in out_lambda_next.                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t nb;
    int d;
    kvqo_block_t *blk;
    int32_t *bad;
} kvqo_set_t;

static void set_build(const uint16_t *x, const float *wt, int64_t T, int D,
                      int G, const int64_t *ids, int64_t nb, kvqo_set_t *st)
{
    int d = 32 * G;
    st->nb = nb;
    st->d = d;
    st->blk = (kvqo_block_t *)malloc(sizeof(kvqo_block_t) * (size_t)nb);
    st->bad = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb);
#pragma omp parallel
    {
        double *v = (double *)malloc(sizeof(double) * d);
        double *wv = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 8)
        for (int64_t i = 0; i < nb; i++) {
            st->bad[i] = block_sorted(x, wt, T, D, G, ids ? ids[i] : i, v, wv);
            block_tables(v, wv, d, &st->blk[i]);
        }
        free(v);
        free(wv);
    }
}

static void set_free(kvqo_set_t *st)
{
    free(st->blk);
    free(st->bad);
}

static double set_rate(const kvqo_set_t *st, int s, double lambda,
                       double *rates)
{
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t i = 0; i < st->nb; i++) {
        kvqo_choice_t ch;
        block_choose(&st->blk[i], s, lambda, 0, &ch);
        rates[i] = ch.Rr;
    }
    double R = 0.0;
    for (int64_t i = 0; i < st->nb; i++) R += rates[i];   /* block order */
    return R;
}

/* per-block outputs at one lambda */
static void set_emit(const kvqo_set_t *st, int s, double lambda,
                     float *codebook, uint8_t *kout, double *Dr, double *Hr,
                     double *gap, uint32_t *masks, double *totals)
{
    int64_t nb = st->nb;
    double *rr = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1));
    double *dd = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1));
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t i = 0; i < nb; i++) {
        const kvqo_block_t *B = &st->blk[i];
        kvqo_choice_t ch;
        block_choose(B, s, lambda, 1, &ch);
        int k = 0;
        float q[KVQO_SMAX];
        for (int j = 0; j < B->mp; j++)
            if (ch.mask >> j & 1u) q[k++] = (float)B->c[j];
        for (int j = k; j < KVQO_SMAX; j++) q[j] = q[k - 1];
        if (codebook) memcpy(codebook + i * KVQO_SMAX, q, sizeof q);
        if (kout) kout[i] = (uint8_t)k;
        if (Dr) Dr[i] = ch.Dr;
        if (Hr) Hr[i] = ch.Rr / (double)B->d;
        if (masks) masks[i] = ch.mask;
        if (gap) {
            if (!(ch.obj2 < INFINITY)) gap[i] = INFINITY;
            else if (ch.obj == 0.0) gap[i] = ch.obj2 > 0.0 ? INFINITY : 0.0;
            else gap[i] = (ch.obj2 - ch.obj) / fabs(ch.obj);
        }
        rr[i] = ch.Rr;
        dd[i] = ch.Dr;
    }
    if (totals) {
        double R = 0, Dsum = 0;
        for (int64_t i = 0; i < nb; i++) {   /* block order */
            R += rr[i];
            Dsum += dd[i];
        }
        totals[0] = R;
        totals[1] = Dsum;
        totals[2] = lambda;
    }
    free(rr);
    free(dd);
}

/* Status codes shared by meaning (not by code) with the library header. */
#define KVQO_OK 0
#define KVQO_INFEASIBLE 4
#define KVQO_NONFINITE 3
#define KVQO_BAD_WEIGHT 8

/* status of a block set: an invalid weight outranks a non-finite value */
static int set_status(const kvqo_set_t *st)
{
    int status = KVQO_OK;
    for (int64_t i = 0; i < st->nb; i++) {
        if (st->bad[i] & 2) return KVQO_BAD_WEIGHT;
        if (st->bad[i] & 1) status = KVQO_NONFINITE;
    }
    return status;
}

/* Bisection over blocks ids[0..nb) (ids == NULL: blocks 0..nb-1).
 * bracket[0..1] receives the final (lo, hi).  Returns the status. */
int kvqo_allocate_bisect(const uint16_t *x, const float *wt, int64_t S,
                         int64_t T, int D, int G, const int64_t *ids, int64_t nb, int s,
                         double budget_bits, double *lambda_out,
                         double *bracket, float *codebook, uint8_t *kout,
                         double *Dr, double *Hr, double *gap, uint32_t *masks,
                         double *totals)
{
    (void)S;
    kvqo_set_t st;
    set_build(x, wt, T, D, G, ids, nb, &st);
    int status = set_status(&st);
    double *rates = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1));
    double lo = 0.0, hi = 0.0, lambda;
    if (set_rate(&st, s, 0.0, rates) <= budget_bits) {
        lambda = 0.0;
    } else {
        for (int64_t i = 0; i < nb; i++) {
            const kvqo_block_t *B = &st.blk[i];
            double w = B->c[B->mp - 1] - B->c[0];
            double h = (w * w) * B->wmax;   /* wmax = 1 without weights */
            if (h > hi) hi = h;
        }
        int n = 0;
        int feas = set_rate(&st, s, hi, rates) <= budget_bits;
        while (!feas && n < 30) {
            hi *= 2.0;
            n++;
            feas = set_rate(&st, s, hi, rates) <= budget_bits;
        }
        if (!feas) {
            if (status == KVQO_OK) status = KVQO_INFEASIBLE;
        } else {
            for (int step = 0; step < 40; step++) {
                double mid = 0.5 * (lo + hi);
                if (set_rate(&st, s, mid, rates) <= budget_bits) hi = mid;
                else lo = mid;
            }
        }
        lambda = hi;
    }
    if (bracket) { bracket[0] = lo; bracket[1] = hi; }
    *lambda_out = lambda;
    set_emit(&st, s, lambda, codebook, kout, Dr, Hr, gap, masks, totals);
    free(rates);
    set_free(&st);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Fixed-rate comparator ("Implementation notes": compare against fixed-rate  */
/* entropy coding at equal total cache bytes).                               */
/* Reading: the same per-block quantizer, but every block r holds the same   */
/* rate, d_r H_r <= b d_r with b = the budget per entry, through its own      */
/* lambda_r found by the bisection above applied to that block alone (R_r(0) */
/* <= b d_r -> lambda_r = 0; hi = (c_max - c_min)^2 (times the block's       */
/* largest weight) doubled at most 30 times; 40 steps; lambda_r = hi).  The  */
/* total rate then meets the same total budget b * entries, so the stored    */
/* bytes are equal and only the allocation across blocks differs.  A block   */
/* still infeasible at hi * 2^30 keeps its choice there (status 4).          */
/* ------------------------------------------------------------------------ */

static int block_bisect(const kvqo_block_t *B, int s, double budget,
                        double *lambda_out)
{
    kvqo_choice_t ch;
    block_choose(B, s, 0.0, 0, &ch);
    if (ch.Rr <= budget) { *lambda_out = 0.0; return KVQO_OK; }
    double w = B->c[B->mp - 1] - B->c[0];
    double lo = 0.0, hi = (w * w) * B->wmax;
    int n = 0;
    block_choose(B, s, hi, 0, &ch);
    int feas = ch.Rr <= budget;
    while (!feas && n < 30) {
        hi *= 2.0;
        n++;
        block_choose(B, s, hi, 0, &ch);
        feas = ch.Rr <= budget;
    }
    if (!feas) { *lambda_out = hi; return KVQO_INFEASIBLE; }
    for (int step = 0; step < 40; step++) {
        double mid = 0.5 * (lo + hi);
        block_choose(B, s, mid, 0, &ch);
        if (ch.Rr <= budget) hi = mid;
        else lo = mid;
    }
    *lambda_out = hi;
    return KVQO_OK;
}

int kvqo_allocate_fixed_rate(const uint16_t *x, const float *wt, int64_t S,
                             int64_t T, int D, int G, const int64_t *ids, int64_t nb,
                             int s, double bits_per_entry, double *lambdas,
                             float *codebook, uint8_t *kout, double *Dr,
                             double *Hr, double *gap, uint32_t *masks,
                             double *totals)
{
    (void)S;
    kvqo_set_t st;
    set_build(x, wt, T, D, G, ids, nb, &st);
    int status = set_status(&st);
    int infeasible = 0;
    double *rr = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1));
    double *dd = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1));
#pragma omp parallel for schedule(dynamic, 4) reduction(|:infeasible)
    for (int64_t i = 0; i < nb; i++) {
        const kvqo_block_t *B = &st.blk[i];
        double lam = 0.0;
        if (block_bisect(B, s, bits_per_entry * (double)B->d, &lam) != KVQO_OK) infeasible = 1;
        lambdas[i] = lam;
        kvqo_choice_t ch;
        block_choose(B, s, lam, 1, &ch);
        int k = 0;
        float q[KVQO_SMAX];
        for (int j = 0; j < B->mp; j++)
            if (ch.mask >> j & 1u) q[k++] = (float)B->c[j];
        for (int j = k; j < KVQO_SMAX; j++) q[j] = q[k - 1];
        if (codebook) memcpy(codebook + i * KVQO_SMAX, q, sizeof q);
        if (kout) kout[i] = (uint8_t)k;
        if (Dr) Dr[i] = ch.Dr;
        if (Hr) Hr[i] = ch.Rr / (double)B->d;
        if (masks) masks[i] = ch.mask;
        if (gap) {
            if (!(ch.obj2 < INFINITY)) gap[i] = INFINITY;
            else if (ch.obj == 0.0) gap[i] = ch.obj2 > 0.0 ? INFINITY : 0.0;
            else gap[i] = (ch.obj2 - ch.obj) / fabs(ch.obj);
        }
        rr[i] = ch.Rr;
        dd[i] = ch.Dr;
    }
    if (totals) {
        double R = 0, Dsum = 0;
        for (int64_t i = 0; i < nb; i++) {   /* block order */
            R += rr[i];
            Dsum += dd[i];
        }
        totals[0] = R;
        totals[1] = Dsum;
        totals[2] = 0.0;
    }
    free(rr);
    free(dd);
    set_free(&st);
    if (status == KVQO_OK && infeasible) status = KVQO_INFEASIBLE;
    return status;
}

/* Choice at a fixed lambda (used for the one-step subgradient map, and to
 * check the codebooks at a given lambda).  *lambda_next receives
 * max(0, lambda + eta (R - budget_bits)). */
int kvqo_allocate_at(const uint16_t *x, const float *wt, int64_t S, int64_t T,
                     int D, int G, const int64_t *ids, int64_t nb, int s, double lambda,
                     double eta, double budget_bits, double *lambda_next,
                     float *codebook, uint8_t *kout, double *Dr, double *Hr,
                     double *gap, uint32_t *masks, double *totals)
{
    (void)S;
    kvqo_set_t st;
    set_build(x, wt, T, D, G, ids, nb, &st);
    int status = set_status(&st);
    double tot[3];
    set_emit(&st, s, lambda, codebook, kout, Dr, Hr, gap, masks, tot);
    if (totals) memcpy(totals, tot, sizeof tot);
    if (lambda_next) {
        double nl = lambda + eta * (tot[0] - budget_bits);
        *lambda_next = nl > 0.0 ? nl : 0.0;
    }
    set_free(&st);
    return status;
}

/* Rate R(lambda) = sum_r d_r H_r over the given blocks (fp64, block order). */
double kvqo_rate_at(const uint16_t *x, const float *wt, int64_t S, int64_t T,
                    int D, int G, const int64_t *ids, int64_t nb, int s,
                    double lambda)
{
    (void)S;
    kvqo_set_t st;
    set_build(x, wt, T, D, G, ids, nb, &st);
    double *rates = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1));
    double R = set_rate(&st, s, lambda, rates);
    free(rates);
    set_free(&st);
    return R;
}

/* Interval tables of one block (for the tests' independent checks). */
int kvqo_block_tables(const uint16_t *x, const float *wt, int64_t T, int D,
                      int G, int64_t b, double *cand, double *Dpq, double *Mup,
                      double *Mdn)
{
    int d = 32 * G;
    double *v = (double *)malloc(sizeof(double) * d);
    double *wv = (double *)malloc(sizeof(double) * d);
    kvqo_block_t B;
    block_sorted(x, wt, T, D, G, b, v, wv);
    block_tables(v, wv, d, &B);
    free(v);
    free(wv);
    for (int j = 0; j < KVQO_M; j++) cand[j] = j < B.mp ? B.c[j] : B.c[B.mp - 1];
    memcpy(Dpq, B.Dpq, sizeof B.Dpq);
    memcpy(Mup, B.Mup, sizeof B.Mup);
    memcpy(Mdn, B.Mdn, sizeof B.Mdn);
    return B.mp;
}

/* Objective pieces of an arbitrary chain (mask over candidate indices) of
 * block b: Dr, d_r H_r. */
void kvqo_chain_cost(const uint16_t *x, const float *wt, int64_t T, int D,
                     int G, int64_t b, uint32_t mask, double *Dr, double *Rr)
{
    int d = 32 * G;
    double *v = (double *)malloc(sizeof(double) * d);
    double *wv = (double *)malloc(sizeof(double) * d);
    kvqo_block_t B;
    block_sorted(x, wt, T, D, G, b, v, wv);
    block_tables(v, wv, d, &B);
    free(v);
    free(wv);
    chain_cost(&B, mask, Dr, Rr);
}

/* ------------------------------------------------------------------------ */
/* Counter-based uniform for the stochastic interpolation.                   */
/* Reading (the page only asks for an unbiased random choice; taken here as  */
/* a counter-based hash with u = hash(seed, index) >> 8): the Philox4x32     */
/* block function (Salmon, Moraes, Dror and Shaw, "Parallel random numbers:  */
/* as easy as 1, 2, 3", SC 2011) with 7 rounds, the fewest rounds that paper  */
/* found to pass TestU01's BigCrush.  Index i uses counter block c = i >> 2  */
/* as the counter (c mod 2^32, c >> 32, 0, 0) and the key (seed mod 2^32,    */
/* seed >> 32); hash(seed, i) is output word i mod 4.                        */
/* One round: the products M0 * x0 and M1 * x2 (32 x 32 -> 64 bits) give     */
/* hi/lo words, the new block is (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0),   */
/* and the key is bumped by the Weyl constants (W0, W1) after each round.    */
/* ------------------------------------------------------------------------ */

#define KVQO_PHILOX_ROUNDS 7

void kvqo_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds,
                     uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < rounds; r++) {
        uint64_t p0 = (uint64_t)M0 * x0;
        uint64_t p1 = (uint64_t)M1 * x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        x0 = hi1 ^ x1 ^ k0;
        x1 = lo1;
        x2 = hi0 ^ x3 ^ k1;
        x3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

uint32_t kvqo_hash32(uint64_t seed, uint64_t i)
{
    uint64_t c = i >> 2;
    uint32_t ctr[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    kvqo_philox4x32(ctr, key, KVQO_PHILOX_ROUNDS, out);
    return out[i & 3u];
}

/* many hashes at once: out[n] = hash(seed, i0 + n) */
void kvqo_hash_many(uint64_t seed, uint64_t i0, int64_t n, uint32_t *out)
{
    for (int64_t j = 0; j < n; j++) out[j] = kvqo_hash32(seed, i0 + (uint64_t)j);
}

/* number of OpenMP threads used by the oracle (<= 0: leave the default) */
int kvqo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Unbiased stochastic interpolation + 4-bit packing ("Key formulas":        */
/* P(hat x = q_{i+1} | x) = (x - q_i)/(q_{i+1} - q_i)).                      */
/* Readings: i = the largest level index with q_i <= x, capped at k-2; with  */
/* u = hash(seed, index_base + flat index) >> 8 and t = u * 2^-24,           */
/* choose i+1 iff fl(t * w) < fl(x - q_i), w = fl(q_{i+1} - q_i), every      */
/* operation fp32 round-to-nearest and none fused.  Code byte e/2 of the     */
/* block holds element e in its low nibble when e is even, high nibble when  */
/* odd.                                                                       */
/* ------------------------------------------------------------------------ */

static uint8_t code_of(float xv, const float *q, int k, uint32_t h)
{
    if (k <= 1) return 0;
    int i = 0;
    while (i + 1 <= k - 2 && q[i + 1] <= xv) i++;
    volatile float w = q[i + 1] - q[i];
    volatile float r = xv - q[i];
    float t = (float)(h >> 8) * 0x1p-24f;
    volatile float tw = t * w;
    return (uint8_t)(i + (tw < r ? 1 : 0));
}

void kvqo_quantize(const uint16_t *x, int64_t S, int64_t T, int D, int G,
                   const float *codebook, const uint8_t *kk, uint64_t seed,
                   uint64_t index_base, int64_t b0, int64_t nb, uint8_t *codes)
{
    (void)S;
    int d = 32 * G;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < nb; i++) {
        int64_t b = b0 + i;
        const float *q = codebook + i * KVQO_SMAX;
        int k = kk[i];
        uint8_t *out = codes + i * (d / 2);
        for (int e = 0; e < d; e += 2) {
            uint8_t c2[2];
            for (int u = 0; u < 2; u++) {
                int64_t f = kvqo_flat_index(T, D, G, b, e + u);
                float xv = (float)kvqo_f16_to_double(x[f]);
                c2[u] = code_of(xv, q, k,
                                kvqo_hash32(seed, index_base + (uint64_t)f));
            }
            out[e / 2] = (uint8_t)(c2[0] | (c2[1] << 4));
        }
    }
}

/* Decode ("Implementation notes": decode before attention): y = q[code]
 * written back as binary16 (exact: every level is a binary16 value). */
int kvqo_dequantize(const uint8_t *codes, const float *codebook, int64_t S,
                    int64_t T, int D, int G, int64_t b0, int64_t nb,
                    uint16_t *y)
{
    (void)S;
    int d = 32 * G, bad = 0;
    for (int64_t i = 0; i < nb; i++) {
        int64_t b = b0 + i;
        const float *q = codebook + i * KVQO_SMAX;
        const uint8_t *in = codes + i * (d / 2);
        for (int e = 0; e < d; e++) {
            int c = (in[e / 2] >> ((e & 1) * 4)) & 15;
            int ok;
            y[kvqo_flat_index(T, D, G, b, e)] =
                kvqo_double_to_f16((double)q[c], &ok);
            if (!ok) bad = 1;
        }
    }
    return bad;
}
