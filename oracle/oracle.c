/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the LM-head contraction and its
 * consumer-surface projection.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The CUDA path never calls it and shares no
 * code, header, table or helper with it.
 *
 * What it follows -- "SemBridge: Compiling Consumer Observations into Cross-Stack
 * Communication Plans" (Chen, Zhu, Lin):
 *   - Section 5.2 (Data, Result, and Control Paths): the tail output head
 *     materialises the full logits; a complete-logits request slices them by TP
 *     lane and rebuilds the full value; a token-only request applies the
 *     deterministic sampler (argmax) to the same tensor.
 *   - Section 3.1 (Boundary Contract): the registered projection operator Q names
 *     its input/output types and a deterministic tie-breaking rule.  The rule is
 *     not named on the page; this oracle takes "lowest global vocabulary index".
 *   - Section 2.2 (Consumer Surfaces and Delivery Obligations): the surfaces are
 *     complete logits, log-probabilities and token IDs.
 *   - Figure 1: full-logit transfer (R0) and source projection (P0) expose the
 *     same token; they differ only in where argmax runs.  The per-shard outputs
 *     below let a test check that argmax over the whole row equals the merge of
 *     the k lane-shard argmaxes.
 *   - Section 2.2 also states that stochastic sampling is outside the page's
 *     contract because it carries no RNG state.  The counter-based Gumbel-max
 *     surface below carries that state explicitly: the stream index of each
 *     (row, column) draw.  SplitMix64 follows Steele, Lea and Flood, "Fast
 *     splittable pseudorandom number generators", OOPSLA 2014; the Gumbel-max
 *     identity is the textbook one (argmax of y + Gumbel noise is a draw from
 *     softmax(y)).
 *
 * Every floating-point step is fp64.  Inputs are raw bf16 bit patterns, widened
 * exactly.  z[r][j] = sum_i h[r][i] * w[j][i], summed with i ascending; no bias,
 * scale or soft-cap (the page names none).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening to double is exact. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Logits of the output head (Section 5.2: "the native tail output head
 * materializes full logits").  Z[r][j] = sum_{i=0}^{d-1} H[r][i] * W[j][i] with
 * H [M][d] and W [V][d] row-major bf16 bits; Z [M][V] row-major.
 * Each sum runs over i in ascending order.  Four rows are carried at once only
 * so the four independent sums overlap in the pipeline; each sum's order is
 * unchanged.
 */
void oracle_logits(const uint16_t *H, const uint16_t *W, int64_t M, int64_t d,
                   int64_t V, double *Z) {
    double *Hd = (double *)malloc(sizeof(double) * (size_t)(M * d));
    for (int64_t t = 0; t < M * d; ++t) Hd[t] = oracle_bf16_to_double(H[t]);
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
        for (int64_t j = 0; j < V; ++j) {
            for (int64_t i = 0; i < d; ++i) w[i] = oracle_bf16_to_double(W[j * d + i]);
            int64_t r = 0;
            for (; r + 4 <= M; r += 4) {
                const double *h0 = Hd + (r + 0) * d, *h1 = Hd + (r + 1) * d;
                const double *h2 = Hd + (r + 2) * d, *h3 = Hd + (r + 3) * d;
                double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
                for (int64_t i = 0; i < d; ++i) {
                    a0 += h0[i] * w[i];
                    a1 += h1[i] * w[i];
                    a2 += h2[i] * w[i];
                    a3 += h3[i] * w[i];
                }
                Z[(r + 0) * V + j] = a0;
                Z[(r + 1) * V + j] = a1;
                Z[(r + 2) * V + j] = a2;
                Z[(r + 3) * V + j] = a3;
            }
            for (; r < M; ++r) {
                const double *h = Hd + r * d;
                double a = 0.0;
                for (int64_t i = 0; i < d; ++i) a += h[i] * w[i];
                Z[r * V + j] = a;
            }
        }
        free(w);
    }
    free(Hd);
}

/*
 * SplitMix64 (Steele, Lea and Flood 2014): the generator's state advances by the
 * golden-ratio increment 0x9E3779B97F4A7C15 before each output, and the output
 * is the state passed through the variant-13 finaliser.  The n-th output
 * (n = 0, 1, ...) of the stream seeded with `seed` therefore depends only on
 * seed + (n + 1) * increment (mod 2^64): that is the counter form used here.
 */
uint64_t oracle_splitmix64(uint64_t seed, uint64_t n) {
    uint64_t x = seed + (n + 1u) * 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

/* Uniform draw: the top 24 bits of the SplitMix64 output, scaled by 2^-24, so
 * u lies on the grid {0, 2^-24, ..., 1 - 2^-24}. */
double oracle_uniform24(uint64_t seed, uint64_t n) {
    return (double)(oracle_splitmix64(seed, n) >> 40) * (1.0 / 16777216.0);
}

/* Standard Gumbel noise g = -log(-log u).  u = 0 gives -infinity, a key that
 * can never win the argmax. */
double oracle_gumbel(uint64_t seed, uint64_t n) {
    double u = oracle_uniform24(seed, n);
    if (u == 0.0) return -INFINITY;
    return -log(-log(u));
}

/*
 * Selection key of column j of a row.  Deterministic surfaces select on the
 * logit itself.  The Gumbel-max surface selects on y + g with y = z / T and g
 * drawn at stream index row * V + j (the row's global index, not its position
 * in a subset).
 */
double oracle_selection_key(double z, int64_t row, int64_t col, int64_t V,
                            int32_t gumbel, double temperature, uint64_t seed) {
    if (!gumbel) return z;
    return z / temperature + oracle_gumbel(seed, (uint64_t)row * (uint64_t)V + (uint64_t)col);
}

/* Natural-log logsumexp of y[lo..hi), shifted by the range maximum. */
static double lse_range(const double *y, int64_t lo, int64_t hi) {
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j)
        if (y[j] > m) m = y[j];
    double s = 0.0;
    for (int64_t j = lo; j < hi; ++j) s += exp(y[j] - m);
    return m + log(s);
}

/* Lowest index attaining the maximum key over [lo, hi) (the tie rule). */
static int64_t argmax_lowest(const double *key, int64_t lo, int64_t hi) {
    int64_t best = lo;
    for (int64_t j = lo + 1; j < hi; ++j)
        if (key[j] > key[best]) best = j;
    return best;
}

/*
 * The consumer-surface projection of each row (Sections 2.2, 3.1 and 5.2; the
 * Gumbel-max surface as described at the top of this file).
 *
 * Inputs: H [M][d], W [V][d] bf16 bits; row_ids [M] = the global row index of
 * each H row (NULL = 0..M-1; it only matters for Gumbel draws); the vocabulary
 * splits into k contiguous lane shards of S = V / k columns; targets [M] (NULL =
 * none).
 *
 * Per row, with y = z (or z / T for the Gumbel surface) and key = y (or y + g):
 *   token          = lowest j attaining max key
 *   lse            = log sum_j exp(y_j)
 *   logprob        = y[token] - lse
 *   target_logprob = y[target] - lse (NaN if no targets)
 *   key_top1/top2  = largest and second-largest key (a duplicate maximum counts
 *                    twice, so top1 - top2 is the decision margin)
 * Per (row, shard s) over columns [s*S, (s+1)*S): shard_max = max key,
 * shard_token = its lowest argmax, shard_lse = logsumexp of y.
 *
 * Z [M][V] receives z when not NULL.  Returns 0, or -1 on invalid arguments.
 */
int oracle_project(const uint16_t *H, const uint16_t *W, const int64_t *row_ids,
                   int64_t M, int64_t d, int64_t V, int32_t k, int32_t gumbel,
                   double temperature, uint64_t seed, const int32_t *targets,
                   int32_t *token, double *lse, double *logprob, double *target_logprob,
                   double *key_top1, double *key_top2, double *shard_max,
                   int32_t *shard_token, double *shard_lse, double *Z) {
    if (M < 1 || d < 1 || V < 1 || k < 1 || V % k != 0) return -1;
    if (gumbel && !(temperature > 0.0)) return -1;
    const int64_t S = V / k;
    double *z = Z ? Z : (double *)malloc(sizeof(double) * (size_t)(M * V));
    if (!z) return -1;
    oracle_logits(H, W, M, d, V, z);
    int bad_target = 0;
#pragma omp parallel
    {
        double *y = (double *)malloc(sizeof(double) * (size_t)V);
        double *key = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < M; ++r) {
            const int64_t row = row_ids ? row_ids[r] : r;
            const double *zr = z + r * V;
            for (int64_t j = 0; j < V; ++j) {
                y[j] = gumbel ? zr[j] / temperature : zr[j];
                key[j] = oracle_selection_key(zr[j], row, j, V, gumbel, temperature, seed);
            }
            const int64_t tok = argmax_lowest(key, 0, V);
            double top2 = -INFINITY;
            for (int64_t j = 0; j < V; ++j)
                if (j != tok && key[j] > top2) top2 = key[j];
            const double l = lse_range(y, 0, V);
            token[r] = (int32_t)tok;
            lse[r] = l;
            logprob[r] = y[tok] - l;
            if (key_top1) key_top1[r] = key[tok];
            if (key_top2) key_top2[r] = top2;
            if (target_logprob) {
                if (targets) {
                    const int64_t t = targets[r];
                    if (t < 0 || t >= V) {
#pragma omp atomic write
                        bad_target = 1;
                        target_logprob[r] = NAN;
                    } else {
                        target_logprob[r] = y[t] - l;
                    }
                } else {
                    target_logprob[r] = NAN;
                }
            }
            for (int32_t s = 0; s < k; ++s) {
                const int64_t lo = (int64_t)s * S, hi = lo + S;
                const int64_t st = argmax_lowest(key, lo, hi);
                if (shard_max) shard_max[r * k + s] = key[st];
                if (shard_token) shard_token[r * k + s] = (int32_t)st;
                if (shard_lse) shard_lse[r * k + s] = lse_range(y, lo, hi);
            }
        }
        free(y);
        free(key);
    }
    if (!Z) free(z);
    return bad_target ? -1 : 0;
}

/*
 * Top-K log-probability surface (a "registered projection" in the sense of Section 2.2:
 * the log-probabilities of the K most likely tokens instead of all V): per row, the K
 * columns with the largest logits, ordered by logit descending and, among equal logits, by
 * column ascending (the deterministic tie rule of Section 3.1), each with its natural-log
 * log-probability z_j - lse.  Selection is K passes of "lowest index attaining the maximum
 * among the columns not yet taken".  ids [M][K], logprob [M][K], lse [M] (NULL allowed).
 * Returns 0, or -1 on invalid arguments (K < 1 or K > V).
 */
int oracle_topk(const uint16_t *H, const uint16_t *W, int64_t M, int64_t d, int64_t V,
                int32_t K, int32_t *ids, double *logprob, double *lse_out) {
    if (M < 1 || d < 1 || V < 1 || K < 1 || K > V) return -1;
    double *z = (double *)malloc(sizeof(double) * (size_t)(M * V));
    if (!z) return -1;
    oracle_logits(H, W, M, d, V, z);
#pragma omp parallel
    {
        unsigned char *taken = (unsigned char *)malloc((size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < M; ++r) {
            const double *zr = z + r * V;
            const double l = lse_range(zr, 0, V);
            if (lse_out) lse_out[r] = l;
            memset(taken, 0, (size_t)V);
            for (int32_t q = 0; q < K; ++q) {
                int64_t best = -1;
                for (int64_t j = 0; j < V; ++j)
                    if (!taken[j] && (best < 0 || zr[j] > zr[best])) best = j;
                taken[best] = 1;
                ids[r * K + q] = (int32_t)best;
                logprob[r * K + q] = zr[best] - l;
            }
        }
        free(taken);
    }
    free(z);
    return 0;
}

/*
 * Partial completion of a row-parallel projection ("SemBridge", Section 6.4 and Table 3: the
 * MLP down projection is the canonical completion boundary; each tensor-parallel lane owns
 * a slice of the reduction dimension and produces an incomplete full-width output, and the
 * partials must be summed before any consumer observes the value; Section 3.5 lists sum
 * among the registered completion operators).
 *   X [M][K] activations and W [N][K] weights (bf16 bits); lane l owns reduction columns
 *   [l*K/lanes, (l+1)*K/lanes).
 *   P[l][m][n] = sum over lane l's columns i (ascending) of X[m][i] * W[n][i]   (fp64)
 *   Y[m][n]    = sum over lanes l = 0, 1, ... of P[l][m][n]                    (fp64)
 * P may be NULL.  Returns 0, or -1 when K is not a multiple of lanes.
 */
int oracle_partial_completion(const uint16_t *X, const uint16_t *W, int64_t M, int64_t N,
                              int64_t K, int32_t lanes, double *Y, double *P) {
    if (M < 1 || N < 1 || K < 1 || lanes < 1 || K % lanes != 0) return -1;
    const int64_t Kl = K / lanes;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double y = 0.0;
            for (int32_t l = 0; l < lanes; ++l) {
                double part = 0.0;
                for (int64_t i = l * Kl; i < (l + 1) * Kl; ++i)
                    part += oracle_bf16_to_double(X[m * K + i]) * oracle_bf16_to_double(W[n * K + i]);
                if (P) P[(l * M + m) * N + n] = part;
                y += part;
            }
            Y[m * N + n] = y;
        }
    return 0;
}

/*
 * Fabric-aware selection between checker-accepted plans, Equation (7) of Section 8.2: the
 * specialised plan s (source projection) is preferred over the reference plan r
 * (complete-logit transfer) when the transfer it saves exceeds the local cost it adds,
 *   (B_r - B_s) / beta + alpha * (F_r - F_s) > L_s - L_r,
 * with B the remote bytes, F the remote frames (startups), beta the link bandwidth in
 * bytes per second, alpha the cost of one frame startup in seconds, and L the local cost
 * (projection and native collectives) in seconds.  *margin (if not NULL) receives the left
 * side minus the right side.  Returns 1 (project at the source), 0 (transfer the complete
 * logits) or -1 for a non-positive or non-finite bandwidth or a negative or non-finite
 * byte, frame or startup input.
 */
int oracle_select_source_projection(double B_r, double B_s, double F_r, double F_s, double beta,
                                    double alpha, double L_s, double L_r, double *margin) {
    if (!(beta > 0.0) || !isfinite(beta) || !(B_r >= 0.0) || !(B_s >= 0.0) || !(F_r >= 0.0) ||
        !(F_s >= 0.0) || !(alpha >= 0.0) || !isfinite(B_r) || !isfinite(B_s) || !isfinite(F_r) ||
        !isfinite(F_s) || !isfinite(alpha) || !isfinite(L_s) || !isfinite(L_r))
        return -1;
    const double lhs = (B_r - B_s) / beta + alpha * (F_r - F_s);
    const double rhs = L_s - L_r;
    if (margin) *margin = lhs - rhs;
    return lhs > rhs ? 1 : 0;
}

/*
 * Result bytes a consumer receives per row: the token surface carries one int32
 * ID, the complete-logit surface carries V bf16 logits (the payload contrast of
 * Figure 1 and Figure 3a: k int32 IDs instead of V logit elements).
 * surface: 0 = token ID, 1 = token ID + chosen log-prob (fp32), 2 = complete
 * bf16 logits.
 */
double oracle_payload_bytes_per_row(int32_t surface, int64_t V) {
    switch (surface) {
    case 0: return 4.0;
    case 1: return 8.0;
    case 2: return 2.0 * (double)V;
    default: return NAN;
    }
}
