/*
 * santa_oracle.c -- plain, slow CPU oracle for stochastic sparse decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant with the CUDA library: it restates, in double precision,
 * one query head at a time and single threaded, what the method computes.
 *
 * Sources (page title, section):
 *   [SSA] "Stochastic Sparse Attention for Memory-Bound Inference" (paper notes)
 *     Overall framework   score stage q K^T -> softmax -> A; value stage A V.
 *     Key design 1        estimator (1/S) sum_s V_{i_s}, i_s ~ A; stratified
 *                         T_m ~ Unif(I_m); systematic U ~ Unif[0, 1/S),
 *                         T_m = U + m/S, J_m = F_q^{-1}(T_m).
 *     Key design 2        S2ANTA-prop: tile partition sums Z_tile, Z = sum Z_tile,
 *                         budget S_tile in proportion to S * Z_tile / Z.
 *     Key design 3        S2ANTA-flash: every tile assumes it holds all the
 *                         mass and draws S/T samples; the merge rescales the
 *                         tile estimates by Z_tile / Z.
 *     Key design 4        Bernoulli q K^T: the query scaled into [-1, 1] gives
 *                         Bernoulli probabilities of a ternary {-1, 0, +1} query
 *                         whose product with K estimates q K^T without bias, so
 *                         only the features it selects are read from K.
 *     Ablation table      mean group query: the GQA group's queries averaged
 *                         before the draw, so the group shares one feature set.
 *   [DP]  "Double-P: Hierarchical Top-P Sparse Attention for Long-Context LLMs"
 *         (paper review), Stage 1, Eq. 3: logit x = q k^T / sqrt(d).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - the logit scale is 1/sqrt(d) ([DP] Eq. 3; [SSA] prints none);
 *   - F(i) is the inclusive CDF, set to exactly 1 from the last key of positive
 *     mass on, and F^{-1}(t) is the smallest i with F(i) > t, i.e. key i owns
 *     the half-open [F(i-1), F(i)), so zero-mass keys are never drawn;
 *   - thresholds use m = 0 .. S-1, so every T_m lies in [0, 1);
 *   - samples are counted with multiplicity (the estimator of Key design 1);
 *   - flash: S_loc = ceil(S / T) samples per tile, all tiles share the offset
 *     U_t = U * S / S_loc in [0, 1/S_loc).
 *   - Bernoulli q K^T: the scale into [-1, 1] is division by max_i |q_i|; a
 *     ternary entry is drawn as sign(q_i) when a caller uniform u < |q_i| / max|q|
 *     and 0 otherwise; `draws` independent draws are averaged; the estimate
 *     replaces q in the logit (x = estimate of q k / sqrt(d)).  The mean group
 *     query draws one selection per KV group from the mean of the group's
 *     queries, p_i = |mean_i| / max|mean|, and head g weights a selected feature
 *     by q_gi / p_i (the Horvitz-Thompson weight), so that every head's estimate
 *     stays unbiased.  The draw decision (u < p) is taken in single precision,
 *     the precision of the queries and uniforms, as the GPU takes it.
 *
 * Matrices are row-major; row i of K starts at K + i * ldk (likewise V).
 * Every function returns 0, or -1 if it could not allocate scratch memory.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* [DP] Stage 1, Eq. 3: x_i = (sum_j q_j k_ij) / sqrt(d). */
void oracle_logits(long n, int d, const double *q, const double *K, long ldk, double *x)
{
    for (long i = 0; i < n; ++i) {
        double s = 0.0;
        for (int j = 0; j < d; ++j)
            s += q[j] * K[i * ldk + j];
        x[i] = s / sqrt((double)d);
    }
}

/* [SSA] Overall framework: A = softmax(x), computed as exp(x_i - max x) / sum. */
void oracle_softmax(long n, const double *x, double *A)
{
    if (n <= 0)
        return;
    double M = x[0];
    for (long i = 1; i < n; ++i)
        if (x[i] > M)
            M = x[i];
    double sum = 0.0;
    for (long i = 0; i < n; ++i) {
        A[i] = exp(x[i] - M);
        sum += A[i];
    }
    for (long i = 0; i < n; ++i)
        A[i] /= sum;
}

/* Inclusive CDF of a probability vector.  Rounding can leave the running sum a
 * hair below 1, so F is set to exactly 1 from the last key of positive mass on:
 * every threshold in [0, 1) then lands on a key of positive mass. */
void oracle_cdf(long n, const double *A, double *F)
{
    double run = 0.0;
    long last = n - 1;
    for (long i = 0; i < n; ++i) {
        run += A[i];
        F[i] = run;
        if (A[i] > 0.0)
            last = i;
    }
    for (long i = last; i >= 0 && i < n; ++i)
        F[i] = 1.0;
}

/* [SSA] Key design 1, J = F_q^{-1}(t): the smallest i with F(i) > t.
 * Thresholds lie in [0, 1) mathematically, but a sum such as U + m/S can round
 * up to exactly 1; such a t is taken as the largest double below 1, so it lands
 * on the last key of positive mass, where F first reaches 1.
 * Binary search; invariant: the answer lies in [lo, hi] and F(hi) > t
 * (true at the start because F(n-1) = 1 > t). */
long oracle_inverse_cdf(long n, const double *F, double t)
{
    if (t >= 1.0)
        t = nextafter(1.0, 0.0);
    long lo = 0, hi = n - 1;
    while (lo < hi) {
        long mid = lo + (hi - lo) / 2;
        if (F[mid] > t)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

/* [SSA] Key design 1, S2ANTA-sys: thresholds T_m = U + m/S, m = 0..S-1. */
void oracle_sys_indices(long n, const double *F, int S, double U, long *J)
{
    for (int m = 0; m < S; ++m)
        J[m] = oracle_inverse_cdf(n, F, U + (double)m / (double)S);
}

/* [SSA] Key design 1, S2ANTA-strat: one draw per stratum I_m = [m/S, (m+1)/S),
 * T_m = (m + u_m) / S with u_m in [0, 1) supplied by the caller. */
void oracle_strat_indices(long n, const double *F, int S, const double *u, long *J)
{
    for (int m = 0; m < S; ++m)
        J[m] = oracle_inverse_cdf(n, F, ((double)m + u[m]) / (double)S);
}

/* [SSA] Key design 1, SANTA: i.i.d. draws i_s = F^{-1}(u_s), u_s in [0, 1). */
void oracle_iid_indices(long n, const double *F, int S, const double *u, long *J)
{
    for (int s = 0; s < S; ++s)
        J[s] = oracle_inverse_cdf(n, F, u[s]);
}

/* [SSA] Key design 1: the estimate (1/S) sum_s V_{J_s}, duplicates counted. */
void oracle_gather_mean(int S, const long *J, int d, const double *V, long ldv, double *out)
{
    for (int j = 0; j < d; ++j)
        out[j] = 0.0;
    for (int s = 0; s < S; ++s)
        for (int j = 0; j < d; ++j)
            out[j] += V[J[s] * ldv + j];
    for (int j = 0; j < d; ++j)
        out[j] /= (double)S;
}

/* Exact value stage: o = sum_i A_i V_i. */
void oracle_exact_av(long n, int d, const double *A, const double *V, long ldv, double *out)
{
    for (int j = 0; j < d; ++j)
        out[j] = 0.0;
    for (long i = 0; i < n; ++i)
        for (int j = 0; j < d; ++j)
            out[j] += A[i] * V[i * ldv + j];
}

/* Exact decode for one query head: logits, softmax, A V.  n = 0 gives zeros. */
int oracle_exact_head(long n, int d, const double *q, const double *K, long ldk,
                      const double *V, long ldv, double *out)
{
    if (n <= 0) {
        for (int j = 0; j < d; ++j)
            out[j] = 0.0;
        return 0;
    }
    double *x = malloc(sizeof(double) * (size_t)n);
    double *A = malloc(sizeof(double) * (size_t)n);
    if (!x || !A) {
        free(x);
        free(A);
        return -1;
    }
    oracle_logits(n, d, q, K, ldk, x);
    oracle_softmax(n, x, A);
    oracle_exact_av(n, d, A, V, ldv, out);
    free(x);
    free(A);
    return 0;
}

/*
 * S2ANTA-prop for one query head ([SSA] Key designs 1 and 2).
 *
 * The pass structure (tile partition sums, a reducer placing the S systematic
 * thresholds, an in-tile search) reproduces exactly the global systematic
 * sample set; so the oracle draws that set directly from the global CDF and
 * reports, per tile of `tile` keys, the tile's probability mass Z_tile / Z and
 * its budget S_tile = the number of samples that fell in it.
 *
 * Outputs (any of J, counts, tile_mass, F may be NULL):
 *   out[d]          (1/S) sum_m V_{J_m}
 *   J[S]            sample index within the sequence, in threshold order
 *   counts[T]       S_tile, T = ceil(n / tile)
 *   tile_mass[T]    sum of A over the tile's keys
 *   F[n]            the global CDF the samples were drawn from
 */
int oracle_prop_head(long n, int d, int tile, int S, double U,
                     const double *q, const double *K, long ldk,
                     const double *V, long ldv,
                     double *out, long *J, int *counts, double *tile_mass, double *F)
{
    long T = n > 0 ? (n + tile - 1) / tile : 0;
    for (long t = 0; t < T; ++t) {
        if (counts)
            counts[t] = 0;
        if (tile_mass)
            tile_mass[t] = 0.0;
    }
    if (n <= 0) {
        for (int j = 0; j < d; ++j)
            out[j] = 0.0;
        return 0;
    }
    double *x = malloc(sizeof(double) * (size_t)n);
    double *A = malloc(sizeof(double) * (size_t)n);
    double *Fl = F ? F : malloc(sizeof(double) * (size_t)n);
    long *Jl = J ? J : malloc(sizeof(long) * (size_t)S);
    if (!x || !A || !Fl || !Jl) {
        free(x);
        free(A);
        if (!F)
            free(Fl);
        if (!J)
            free(Jl);
        return -1;
    }
    oracle_logits(n, d, q, K, ldk, x);
    oracle_softmax(n, x, A);
    oracle_cdf(n, A, Fl);
    oracle_sys_indices(n, Fl, S, U, Jl);
    oracle_gather_mean(S, Jl, d, V, ldv, out);
    if (counts)
        for (int m = 0; m < S; ++m)
            counts[Jl[m] / tile] += 1;
    if (tile_mass)
        for (long i = 0; i < n; ++i)
            tile_mass[i / tile] += A[i];
    free(x);
    free(A);
    if (!F)
        free(Fl);
    if (!J)
        free(Jl);
    return 0;
}

/*
 * SANTA (i.i.d.) or S2ANTA-strat for one query head, fed S caller uniforms
 * u[s] in [0, 1) ([SSA] Key design 1).  mode 0 = i.i.d., 1 = stratified.
 */
int oracle_sampled_head(int mode, long n, int d, int S, const double *u,
                        const double *q, const double *K, long ldk,
                        const double *V, long ldv, double *out, long *J)
{
    if (n <= 0) {
        for (int j = 0; j < d; ++j)
            out[j] = 0.0;
        return 0;
    }
    double *x = malloc(sizeof(double) * (size_t)n);
    double *A = malloc(sizeof(double) * (size_t)n);
    double *F = malloc(sizeof(double) * (size_t)n);
    long *Jl = J ? J : malloc(sizeof(long) * (size_t)S);
    if (!x || !A || !F || !Jl) {
        free(x);
        free(A);
        free(F);
        if (!J)
            free(Jl);
        return -1;
    }
    oracle_logits(n, d, q, K, ldk, x);
    oracle_softmax(n, x, A);
    oracle_cdf(n, A, F);
    if (mode == 0)
        oracle_iid_indices(n, F, S, u, Jl);
    else
        oracle_strat_indices(n, F, S, u, Jl);
    oracle_gather_mean(S, Jl, d, V, ldv, out);
    free(x);
    free(A);
    free(F);
    if (!J)
        free(Jl);
    return 0;
}

/*
 * S2ANTA-flash for one query head ([SSA] Key design 3).
 *
 * For every tile t of `tile` keys (T = ceil(n / tile) tiles):
 *   m_t = max logit in the tile, e_i = exp(x_i - m_t), z_t = sum e_i;
 *   the tile's own distribution A_i = e_i / z_t and its CDF F_t;
 *   S_loc = ceil(S / T) systematic thresholds U_t + m / S_loc with the shared
 *   offset U_t = U * S / S_loc in [0, 1/S_loc);
 *   the tile estimate o_t = (1/S_loc) sum V_{J}.
 * Merge: M = max m_t, w_t = z_t exp(m_t - M) (the tile's partition sum on a
 * common scale), Z = sum w_t, out = sum_t (w_t / Z) o_t.
 *
 * Outputs (J, tile_m, tile_z, weight may be NULL):
 *   J[T * S_loc]   per tile, the sampled key index within the sequence
 *   tile_m[T], tile_z[T], weight[T] = w_t / Z.
 * Returns S_loc (>= 0), or -1 on allocation failure.
 */
int oracle_flash_head(long n, int d, int tile, int S, double U,
                      const double *q, const double *K, long ldk,
                      const double *V, long ldv,
                      double *out, long *J, double *tile_m, double *tile_z, double *weight)
{
    for (int j = 0; j < d; ++j)
        out[j] = 0.0;
    if (n <= 0)
        return 0;
    long T = (n + tile - 1) / tile;
    int S_loc = (int)((S + T - 1) / T);
    double U_t = U * (double)S / (double)S_loc;

    double *x = malloc(sizeof(double) * (size_t)n);
    double *At = malloc(sizeof(double) * (size_t)tile);
    double *Ft = malloc(sizeof(double) * (size_t)tile);
    double *mt = malloc(sizeof(double) * (size_t)T);
    double *zt = malloc(sizeof(double) * (size_t)T);
    double *ot = malloc(sizeof(double) * (size_t)T * (size_t)d);
    long *Jt = malloc(sizeof(long) * (size_t)S_loc);
    if (!x || !At || !Ft || !mt || !zt || !ot || !Jt) {
        free(x);
        free(At);
        free(Ft);
        free(mt);
        free(zt);
        free(ot);
        free(Jt);
        return -1;
    }
    oracle_logits(n, d, q, K, ldk, x);

    for (long t = 0; t < T; ++t) {
        long k0 = t * tile;
        long len = (k0 + tile <= n) ? tile : n - k0;
        double m = x[k0];
        for (long i = 1; i < len; ++i)
            if (x[k0 + i] > m)
                m = x[k0 + i];
        double z = 0.0;
        for (long i = 0; i < len; ++i)
            z += exp(x[k0 + i] - m);
        /* the tile's own distribution e_i / z_t and its CDF */
        for (long i = 0; i < len; ++i)
            At[i] = exp(x[k0 + i] - m) / z;
        oracle_cdf(len, At, Ft);
        for (int s = 0; s < S_loc; ++s)
            Jt[s] = k0 + oracle_inverse_cdf(len, Ft, U_t + (double)s / (double)S_loc);
        oracle_gather_mean(S_loc, Jt, d, V, ldv, ot + t * d);
        if (J)
            memcpy(J + t * S_loc, Jt, sizeof(long) * (size_t)S_loc);
        mt[t] = m;
        zt[t] = z;
    }

    double M = mt[0];
    for (long t = 1; t < T; ++t)
        if (mt[t] > M)
            M = mt[t];
    double Z = 0.0;
    for (long t = 0; t < T; ++t)
        Z += zt[t] * exp(mt[t] - M);
    for (long t = 0; t < T; ++t) {
        double w = zt[t] * exp(mt[t] - M) / Z;
        for (int j = 0; j < d; ++j)
            out[j] += w * ot[t * d + j];
        if (tile_m)
            tile_m[t] = mt[t];
        if (tile_z)
            tile_z[t] = zt[t];
        if (weight)
            weight[t] = w;
    }
    free(x);
    free(At);
    free(Ft);
    free(mt);
    free(zt);
    free(ot);
    free(Jt);
    return S_loc;
}

/*
 * Bernoulli q K^T ([SSA] Key design 4; mean group query: [SSA] ablation table)
 * for one KV group of G query heads: the effective queries c_g such that
 * c_g . k is the estimate of q_g . k for every key k.
 *   q[G][d]              the group's queries (values of single precision)
 *   u[ns][draws][d]      uniforms in [0, 1) (single precision values); ns = G
 *                        (one draw set per head) or 1 (group_mean)
 *   c[G][d]              out: the effective queries
 *   read[d]              out: 1 if some draw of the group selected feature i
 * Per head: p_gi = |q_gi| / max_j |q_gj|; draw b selects i when u[g][b][i] < p_gi,
 * giving the ternary entry t = sign(q_gi), else 0; c_gi = max|q_g| * mean_b t.
 * Group mean: qbar = (q_0 + ... + q_{G-1}) / G, p_i = |qbar_i| / max_j |qbar_j|;
 * draw b selects i when u[0][b][i] < p_i; c_gi = (selections of i / draws) * q_gi / p_i.
 * A query (or mean) of all zeros selects nothing: c = 0, and so does p_i = 0.
 * Returns the number of features read.
 */
int oracle_bernoulli_query(int G, int d, int draws, int group_mean, const double *q, const double *u, double *c,
                           int *read)
{
    int nread = 0;
    for (int i = 0; i < d; ++i)
        read[i] = 0;
    if (!group_mean) {
        for (int g = 0; g < G; ++g) {
            const double *qg = q + (size_t)g * d;
            float mx = 0.0f;
            for (int i = 0; i < d; ++i) {
                float a = fabsf((float)qg[i]);
                if (a > mx)
                    mx = a;
            }
            for (int i = 0; i < d; ++i) {
                int hits = 0;
                if (mx > 0.0f) {
                    float p = fabsf((float)qg[i]) / mx;
                    for (int b = 0; b < draws; ++b)
                        hits += (float)u[((size_t)g * draws + b) * d + i] < p;
                }
                double sign = qg[i] > 0.0 ? 1.0 : (qg[i] < 0.0 ? -1.0 : 0.0);
                c[(size_t)g * d + i] = (double)mx * sign * (double)hits / (double)draws;
                if (hits > 0)
                    read[i] = 1;
            }
        }
    } else {
        float *mean = malloc(sizeof(float) * (size_t)d);
        if (!mean)
            return -1;
        float mx = 0.0f;
        for (int i = 0; i < d; ++i) {
            float s = 0.0f;
            for (int g = 0; g < G; ++g)
                s += (float)q[(size_t)g * d + i];
            mean[i] = s / (float)G;
            if (fabsf(mean[i]) > mx)
                mx = fabsf(mean[i]);
        }
        for (int i = 0; i < d; ++i) {
            int hits = 0;
            float p = mx > 0.0f ? fabsf(mean[i]) / mx : 0.0f;
            if (p > 0.0f)
                for (int b = 0; b < draws; ++b)
                    hits += (float)u[(size_t)b * d + i] < p;
            for (int g = 0; g < G; ++g)
                c[(size_t)g * d + i] = hits > 0 ? q[(size_t)g * d + i] / (double)p * (double)hits / (double)draws : 0.0;
            if (hits > 0)
                read[i] = 1;
        }
        free(mean);
    }
    for (int i = 0; i < d; ++i)
        nread += read[i];
    return nread;
}
