/*
 * CPU oracle of the routed int4 MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads this library:
 * only the tests, the package's smoke check and the bench's CPU-baseline and
 * reference legs do.  It shares no code, header or constant with the CUDA
 * library; it is written from the definitions alone.
 *
 * Every value is an IEEE double; loops run in the plain order of each
 * definition, with no blocking, fusion or reordering.
 *
 * What it follows (Swiftlet project pages):
 *   - each layer routes each token to 10 of 512 (80B) or 8 of 256 (35B)
 *     experts (Swiftlet README "How it works");
 *   - the router and a shared expert are resident (Swiftlet README "How it works");
 *   - weights use MLX affine int4 or int8 group quantisation,
 *     W ~= scale*q + bias per group (Swiftlet README "Relation to TurboFieldfare");
 *   - the layer is checked against an exact CPU reference, and streaming an
 *     expert from cache or from storage never changes the result (Swiftlet README
 *     "Correctness").
 * The softmax over the selected experts, the SwiGLU expert MLP and the
 * sigmoid gate of the shared expert follow the Qwen3-Next / Qwen3.5-3.6
 * layer that the pages name but do not write out; readings are listed in the
 * repository's design notes.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Built twice: plain (the tests' oracle), and with OpenMP, where the loops
 * over output rows below are shared among threads.  Each output row is still
 * computed by one thread in the same order, so both builds give the same
 * doubles; the OpenMP build only exists to time the oracle on all cores. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

/* Router: logits[t,e] = sum_h w_router[e,h] * x[t,h] + bias[e]  (bias may be
 * NULL, meaning zero), and the shared-gate logit s[t] = sum_h w_sg[h] x[t,h]
 * (w_sg may be NULL when there is no shared expert). */
void oracle_router(int T, int H, int E, const double *x, const double *w_router,
                   const double *bias, const double *w_sg, double *logits, double *s)
{
    for (int t = 0; t < T; ++t) {
        const double *xt = x + (size_t)t * H;
#pragma omp parallel for schedule(static)
        for (int e = 0; e < E; ++e) {
            const double *we = w_router + (size_t)e * H;
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += we[h] * xt[h];
            logits[(size_t)t * E + e] = acc + (bias ? bias[e] : 0.0);
        }
        if (w_sg) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += w_sg[h] * xt[h];
            s[t] = acc;
        }
    }
}

/* Top-k with renormalised softmax weights for one token.
 * Selection: the k largest logits; among equal logits the lower expert id
 * ranks first; output in that (descending) order.
 * Weights: w_r = exp(l_r - l_max) / sum_{j in top-k} exp(l_j - l_max), which
 * equals a softmax over all E followed by renormalisation over the k. */
void oracle_topk(int E, int k, const double *logits, int32_t *idx, double *w)
{
    for (int r = 0; r < k; ++r) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            int taken = 0;
            for (int j = 0; j < r; ++j)
                if (idx[j] == e)
                    taken = 1;
            if (taken)
                continue;
            if (best < 0 || logits[e] > logits[best])
                best = e;
        }
        idx[r] = best;
    }
    double lmax = logits[idx[0]];
    double den = 0.0;
    for (int r = 0; r < k; ++r)
        den += exp(logits[idx[r]] - lmax);
    for (int r = 0; r < k; ++r)
        w[r] = exp(logits[idx[r]] - lmax) / den;
}

/* One dequantised weight of an affine matrix [n_out, n_in] with b-bit codes
 * (b = bits, 4 or 8; p = 32/b codes a word) and groups of G input columns:
 * the code of column c of row o sits in word q[o, c/p] at bits
 * b*(c%p) .. b*(c%p)+b-1; W[o,c] = scale[o,c/G]*code + bias[o,c/G]. */
static double dequant(const uint32_t *q, const double *scale, const double *bias,
                      int n_in, int G, int bits, int o, int c)
{
    const int p = 32 / bits;
    uint32_t word = q[(size_t)o * (n_in / p) + c / p];
    unsigned code = (word >> (bits * (c % p))) & ((1u << bits) - 1u);
    size_t g = (size_t)o * (n_in / G) + c / G;
    return scale[g] * (double)code + bias[g];
}

/* The whole dense matrix W [n_out, n_in]. */
void oracle_dequant(int n_out, int n_in, int G, int bits, const uint32_t *q, const double *scale,
                    const double *bias, double *W)
{
    for (int o = 0; o < n_out; ++o)
        for (int c = 0; c < n_in; ++c)
            W[(size_t)o * n_in + c] = dequant(q, scale, bias, n_in, G, bits, o, c);
}

/* y = W v for an affine matrix with b-bit codes. */
void oracle_qmatvec(int n_out, int n_in, int G, int bits, const uint32_t *q, const double *scale,
                    const double *bias, const double *v, double *y)
{
#pragma omp parallel for schedule(static)
    for (int o = 0; o < n_out; ++o) {
        double acc = 0.0;
        for (int c = 0; c < n_in; ++c)
            acc += dequant(q, scale, bias, n_in, G, bits, o, c) * v[c];
        y[o] = acc;
    }
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* One SwiGLU expert on one token: g = Wg x, u = Wu x, a = silu(g) * u,
 * y = Wd a.  Wg, Wu: [I, H]; Wd: [H, I].  work: 3*I doubles. */
void oracle_expert(int H, int I, int G, int bits,
                   const uint32_t *qg, const double *sg, const double *bg,
                   const uint32_t *qu, const double *su, const double *bu,
                   const uint32_t *qd, const double *sd, const double *bd,
                   const double *x, double *y, double *work)
{
    double *g = work, *u = work + I, *a = work + 2 * (size_t)I;
    oracle_qmatvec(I, H, G, bits, qg, sg, bg, x, g);
    oracle_qmatvec(I, H, G, bits, qu, su, bu, x, u);
    for (int i = 0; i < I; ++i)
        a[i] = silu(g[i]) * u[i];
    oracle_qmatvec(H, I, G, bits, qd, sd, bd, a, y);
}

/* Token -> expert bucketing: a stable counting sort of the T*k (token, rank)
 * pairs by expert id.  counts[e] = pairs routed to e; offsets = exclusive
 * prefix sum (E+1 entries); perm_tok / perm_rank list the pairs ordered by
 * (expert, token, rank). */
void oracle_bucket(int T, int k, int E, const int32_t *idx, int32_t *counts,
                   int32_t *offsets, int32_t *perm_tok, int32_t *perm_rank)
{
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int p = 0; p < T * k; ++p)
        counts[idx[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    for (int e = 0; e < E; ++e) {
        int n = offsets[e];
        for (int t = 0; t < T; ++t)
            for (int r = 0; r < k; ++r)
                if (idx[(size_t)t * k + r] == e) {
                    perm_tok[n] = t;
                    perm_rank[n] = r;
                    ++n;
                }
    }
}
