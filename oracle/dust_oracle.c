/*
 * Plain fp64 CPU oracle for Dust's per-token zeroth-order estimator of one
 * linear layer y_t = W x_t.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg load this library. The CUDA
 * library shares no source, header, table or helper with this file, and the
 * product path never calls into it.
 *
 * Source of truth: "Dust: every token is a member of the population"
 * (ai.satyajit.si), section "Perturb the activations, not the weights":
 *
 *     r_t = sum_{s >= t} gamma^(s-t) c_s
 *     g_t = -(1 / (K sigma)) sum_i r_t^(i) a_t^(i)
 *     GW  = sum_t g_t x_t^T
 *
 * with c_s the centred loss reduction at token s (same page, "What the
 * released code actually does", step 2: reward = clean loss - perturbed loss,
 * centred across the draws that share a forward) and the contraction of step 7
 * of that list (einsum over batch and token, optionally divided by the token
 * count, here the `scale` argument).
 *
 * The noise generator follows the family named in "RandOpt Speedrun", section
 * "What was slow, and the fix": a counter-based murmur3 fmix32 hash over a
 * folded position. The exact folding, the sign rule and the Box-Muller
 * mapping are this project's own definition (see noise_word / noise_value).
 *
 * Every function here is the plain definition: one loop per sum, fp64
 * throughout, no blocking and no reordering of any sum. OpenMP parallelises
 * only loops whose iterations are independent outputs.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_EXPORT __attribute__((visibility("default")))

enum { OR_RADEMACHER = 0, OR_GAUSSIAN = 1, OR_RADEMACHER_PACKED = 3 };
enum { OR_CENTER = 1, OR_ANTITHETIC = 2 };

static const double OR_PI = 3.14159265358979323846264338327950288;

/* ------------------------------------------------------------------ hash -- */

/* MurmurHash3's 32-bit finaliser (Appleby, public domain): three xor-shifts
 * and two multiplications by the published odd constants, all mod 2^32. */
static uint32_t or_fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

/* floor(2^32 / golden ratio), the usual Weyl increment. */
static const uint32_t OR_WEYL = 0x9E3779B9u;

/* The 64-bit seed folded to one 32-bit key. */
static uint32_t or_seed_key(uint64_t seed) {
    uint32_t lo = (uint32_t)(seed & 0xffffffffu);
    uint32_t hi = (uint32_t)(seed >> 32);
    return or_fmix32(lo ^ or_fmix32(hi + OR_WEYL));
}

/* Key of draw i, word stream s in {0, 1}. */
static uint32_t or_draw_key(uint64_t seed, int64_t i, int s) {
    uint32_t m = (uint32_t)((uint64_t)(2 * i + s) & 0xffffffffu);
    return or_fmix32(or_seed_key(seed) ^ (uint32_t)(m * OR_WEYL));
}

/* The hash word of (seed, draw i, token t, channel c, stream s). Token and
 * channel form the low 32-bit counter t*d_out + c (callers guarantee
 * T*d_out <= 2^32, so the counter is distinct for every (t, c)). */
static uint32_t or_word(uint64_t seed, int64_t i, int64_t t, int64_t c,
                        int64_t d_out, int s) {
    uint32_t n = (uint32_t)((uint64_t)(t * d_out + c) & 0xffffffffu);
    return or_fmix32(or_draw_key(seed, i, s) ^ n);
}

/* a_t^(i)[c] for one element-draw.
 *  Rademacher: +1 when the top bit of the stream-0 word is clear, else -1.
 *  Gaussian:   Box-Muller on the channel pair p = c & ~1, from the stream-0
 *              word w0 and the stream-1 word w1 of channel p:
 *                 u1 = 1 - (w0 >> 9) 2^-23  in [2^-23, 1]
 *                 u2 =     (w1 >> 9) 2^-23  in [0, 1)
 *                 rho = sqrt(-2 ln u1)
 *              even c -> rho cos(2 pi u2), odd c -> rho sin(2 pi u2).
 *  Antithetic: draw i uses base draw i >> 1 and sign (-1)^(i & 1), so draws
 *              2j and 2j+1 are an opposite-sign pair (same page as above,
 *              "What a zeroth-order gradient is"). */
static double or_noise_value(int kind, uint64_t seed, int64_t i, int64_t t,
                             int64_t c, int64_t d_out, uint32_t flags) {
    double sign = 1.0;
    if (flags & OR_ANTITHETIC) {
        sign = (i & 1) ? -1.0 : 1.0;
        i = i >> 1;
    }
    if (kind == OR_RADEMACHER) {
        uint32_t w = or_word(seed, i, t, c, d_out, 0);
        return sign * ((w >> 31) ? -1.0 : 1.0);
    }
    if (kind == OR_RADEMACHER_PACKED) {
        /* 32 signs per word: channel c takes bit c mod 32 of the word of its
         * group's first channel 32 floor(c / 32); bit 0 gives +1. */
        uint32_t w = or_word(seed, i, t, c & ~(int64_t)31, d_out, 0);
        return sign * (((w >> (c & 31)) & 1u) ? -1.0 : 1.0);
    }
    int64_t p = c & ~(int64_t)1;
    uint32_t w0 = or_word(seed, i, t, p, d_out, 0);
    uint32_t w1 = or_word(seed, i, t, p, d_out, 1);
    double u1 = 1.0 - (double)(w0 >> 9) * ldexp(1.0, -23);
    double u2 = (double)(w1 >> 9) * ldexp(1.0, -23);
    double rho = sqrt(-2.0 * log(u1));
    double v = (c & 1) ? rho * sin(2.0 * OR_PI * u2) : rho * cos(2.0 * OR_PI * u2);
    return sign * v;
}

OR_EXPORT uint32_t dust_oracle_fmix32(uint32_t h) { return or_fmix32(h); }
OR_EXPORT uint32_t dust_oracle_seed_key(uint64_t seed) { return or_seed_key(seed); }
OR_EXPORT uint32_t dust_oracle_draw_key(uint64_t seed, int64_t i, int32_t s) {
    return or_draw_key(seed, i, s);
}

OR_EXPORT int32_t dust_oracle_num_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

OR_EXPORT void dust_oracle_set_threads(int32_t n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Raw words word(draw_begin + k, t, c, stream), out[n_draws][T][d_out]. */
OR_EXPORT void dust_oracle_words(uint32_t* out, uint64_t seed, int64_t draw_begin,
                                 int64_t n_draws, int64_t T, int64_t d_out,
                                 int32_t stream) {
    for (int64_t k = 0; k < n_draws; ++k) {
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t c = 0; c < d_out; ++c)
                out[(k * T + t) * d_out + c] =
                    or_word(seed, draw_begin + k, t, c, d_out, stream);
    }
}

/* Noise values a_t^(draw_begin + k)[c], out[n_draws][T][d_out]. */
OR_EXPORT void dust_oracle_noise(double* out, uint64_t seed, int32_t kind,
                                 int64_t draw_begin, int64_t n_draws, int64_t T,
                                 int64_t d_out, uint32_t flags) {
    for (int64_t k = 0; k < n_draws; ++k) {
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t c = 0; c < d_out; ++c)
                out[(k * T + t) * d_out + c] =
                    or_noise_value(kind, seed, draw_begin + k, t, c, d_out, flags);
    }
}

/* Noise values at a list of (draw, token, channel) triples. */
OR_EXPORT void dust_oracle_noise_at(double* out, const int64_t* draw, const int64_t* tok,
                                    const int64_t* chan, int64_t n, uint64_t seed,
                                    int32_t kind, int64_t d_out, uint32_t flags) {
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k)
        out[k] = or_noise_value(kind, seed, draw[k], tok[k], chan[k], d_out, flags);
}

/* ------------------------------------------------------- estimator steps -- */

/* Centred loss reductions. The API's delta[i][t] is the loss change
 * L(perturbed) - L(clean); the reduction is its negative (reward = clean -
 * perturbed). With OR_CENTER and K > 1 the per-token mean over the K draws is
 * subtracted. c_out[K][T]. */
OR_EXPORT void dust_oracle_center(const double* delta, int64_t K, int64_t T,
                                  uint32_t flags, double* c_out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double mean = 0.0;
        if ((flags & OR_CENTER) && K > 1) {
            for (int64_t i = 0; i < K; ++i) mean += -delta[i * T + t];
            mean /= (double)K;
        }
        for (int64_t i = 0; i < K; ++i) c_out[i * T + t] = -delta[i * T + t] - mean;
    }
}

/* Reverse credit scan, restarted at every sequence:
 *   r[i][t] = c[i][t] + gamma * r[i][t+1]   inside [o_k, o_{k+1}),
 * with r = 0 past a sequence's last token. r_out[K][T]. */
OR_EXPORT void dust_oracle_scan(const double* c, int64_t K, int64_t T,
                                const int32_t* seq_offsets, int64_t n_seq,
                                double gamma, double* r_out) {
    (void)T;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < K; ++i) {
        for (int64_t q = 0; q < n_seq; ++q) {
            int64_t lo = seq_offsets[q], hi = seq_offsets[q + 1];
            double next = 0.0;
            for (int64_t t = hi - 1; t >= lo; --t) {
                next = c[i * T + t] + gamma * next;
                r_out[i * T + t] = next;
            }
        }
    }
}

/* Per-token output-error estimate
 *   g[t][c] = -(1 / (K sigma)) sum_i r[i][t] a_t^(draw_begin + i)[c].
 * r is [K][T]; g_out is [T][d_out]. */
OR_EXPORT void dust_oracle_error_estimate(const double* r, int64_t K, int64_t T,
                                          int64_t d_out, uint64_t seed, int32_t kind,
                                          int64_t draw_begin, double sigma,
                                          uint32_t flags, double* g_out) {
    double coef = -1.0 / ((double)K * sigma);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < d_out; ++c) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i)
                acc += r[i * T + t] *
                       or_noise_value(kind, seed, draw_begin + i, t, c, d_out, flags);
            g_out[t * d_out + c] = coef * acc;
        }
    }
}

/* Weight-gradient contraction GW[c][j] = scale * sum_t g[t][c] x[t][j]. */
OR_EXPORT void dust_oracle_contract(const double* g, const double* X, int64_t T,
                                    int64_t d_in, int64_t d_out, double scale,
                                    double* gW) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < d_out; ++c) {
        double* row = gW + c * d_in;
        for (int64_t j = 0; j < d_in; ++j) row[j] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            double gtc = g[t * d_out + c];
            const double* xt = X + t * d_in;
            for (int64_t j = 0; j < d_in; ++j) row[j] += gtc * xt[j];
        }
        for (int64_t j = 0; j < d_in; ++j) row[j] *= scale;
    }
}

/* The whole path: delta -> centre -> scan -> g -> GW. Scratch is allocated
 * here (this is CPU test code). */
OR_EXPORT int32_t dust_oracle_estimate_gW(const double* X, int64_t T, int64_t d_in,
                                          const double* delta, int64_t K, int64_t d_out,
                                          const int32_t* seq_offsets, int64_t n_seq,
                                          uint64_t seed, int32_t kind, int64_t draw_begin,
                                          double sigma, double gamma, double scale,
                                          uint32_t flags, double* gW) {
    double* c = (double*)malloc(sizeof(double) * (size_t)(K * T));
    double* r = (double*)malloc(sizeof(double) * (size_t)(K * T));
    double* g = (double*)malloc(sizeof(double) * (size_t)(T * d_out));
    if (!c || !r || !g) {
        free(c); free(r); free(g);
        return -1;
    }
    dust_oracle_center(delta, K, T, flags, c);
    dust_oracle_scan(c, K, T, seq_offsets, n_seq, gamma, r);
    dust_oracle_error_estimate(r, K, T, d_out, seed, kind, draw_begin, sigma, flags, g);
    dust_oracle_contract(g, X, T, d_in, d_out, scale, gW);
    free(c); free(r); free(g);
    return 0;
}

/* Rows of g at selected tokens, from full-length r ([K][T]). out[n_tok][d_out]. */
OR_EXPORT void dust_oracle_error_rows(const double* r, int64_t K, int64_t T, int64_t d_out,
                                      const int64_t* toks, int64_t n_tok, uint64_t seed,
                                      int32_t kind, int64_t draw_begin, double sigma,
                                      uint32_t flags, double* out) {
    double coef = -1.0 / ((double)K * sigma);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < n_tok; ++q) {
        int64_t t = toks[q];
        for (int64_t c = 0; c < d_out; ++c) {
            double acc = 0.0;
            for (int64_t i = 0; i < K; ++i)
                acc += r[i * T + t] *
                       or_noise_value(kind, seed, draw_begin + i, t, c, d_out, flags);
            out[q * d_out + c] = coef * acc;
        }
    }
}

/* Selected entries GW[chan[q]][col[q]], computed one by one from the full
 * column g[:, chan[q]] (full-length r, [K][T]) and X. */
OR_EXPORT void dust_oracle_gW_entries(const double* X, int64_t T, int64_t d_in,
                                      const double* r, int64_t K, int64_t d_out,
                                      const int64_t* chan, const int64_t* col, int64_t n,
                                      uint64_t seed, int32_t kind, int64_t draw_begin,
                                      double sigma, double scale, uint32_t flags,
                                      double* out) {
    double coef = -1.0 / ((double)K * sigma);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < n; ++q) {
        int64_t c = chan[q], j = col[q];
        double acc = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            double gsum = 0.0;
            for (int64_t i = 0; i < K; ++i)
                gsum += r[i * T + t] *
                        or_noise_value(kind, seed, draw_begin + i, t, c, d_out, flags);
            acc += coef * gsum * X[t * d_in + j];
        }
        out[q] = scale * acc;
    }
}

/* Brute force for tiny inputs: the same GW with no scan and no intermediate
 * g, straight from the three equations:
 *   GW[c][j] = -scale/(K sigma) sum_t sum_i sum_{s>=t, same sequence}
 *              gamma^(s-t) cen[i][s] a_t^(i)[c] x[t][j]. */
OR_EXPORT void dust_oracle_bruteforce_gW(const double* X, int64_t T, int64_t d_in,
                                         const double* delta, int64_t K, int64_t d_out,
                                         const int32_t* seq_offsets, int64_t n_seq,
                                         uint64_t seed, int32_t kind, int64_t draw_begin,
                                         double sigma, double gamma, double scale,
                                         uint32_t flags, double* gW) {
    for (int64_t c = 0; c < d_out; ++c)
        for (int64_t j = 0; j < d_in; ++j) {
            double acc = 0.0;
            for (int64_t q = 0; q < n_seq; ++q)
                for (int64_t t = seq_offsets[q]; t < seq_offsets[q + 1]; ++t)
                    for (int64_t i = 0; i < K; ++i)
                        for (int64_t s = t; s < seq_offsets[q + 1]; ++s) {
                            double mean = 0.0;
                            if ((flags & OR_CENTER) && K > 1) {
                                for (int64_t m = 0; m < K; ++m) mean += -delta[m * T + s];
                                mean /= (double)K;
                            }
                            double cen = -delta[i * T + s] - mean;
                            acc += pow(gamma, (double)(s - t)) * cen *
                                   or_noise_value(kind, seed, draw_begin + i, t, c, d_out,
                                                  flags) *
                                   X[t * d_in + j];
                        }
            gW[c * d_in + j] = -scale / ((double)K * sigma) * acc;
        }
}

/* Jitter of the forward: y[t][c] += sigma * a_t^(draw)[c], y row stride ld_y. */
OR_EXPORT void dust_oracle_jitter(double* y, int64_t ld_y, int64_t T, int64_t d_out,
                                  uint64_t seed, int32_t kind, int64_t draw, double sigma,
                                  uint32_t flags) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < d_out; ++c)
            y[t * ld_y + c] += sigma * or_noise_value(kind, seed, draw, t, c, d_out, flags);
}

/* The jittered forward of a linear layer for several draws from one product
 * ("Dust: every token is a member of the population", "Perturb the
 * activations, not the weights": y_t -> y_t + sigma a_t, the jitter added
 * after the layer's product): y = X W^T, then
 *   out[clean + k][t][c] = y[t][c] + sigma a_t^(draw_begin + k)[c],
 * with out[0] = y itself when clean = 1. X [T][d_in], W [d_out][d_in]. */
OR_EXPORT void dust_oracle_forward_jitter(const double* X, const double* W, int64_t T,
                                          int64_t d_in, int64_t d_out, uint64_t seed,
                                          int32_t kind, int64_t draw_begin, int64_t n_draws,
                                          double sigma, uint32_t flags, int32_t clean,
                                          double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < d_out; ++c) {
            double y = 0.0;
            for (int64_t j = 0; j < d_in; ++j) y += X[t * d_in + j] * W[c * d_in + j];
            if (clean) out[t * d_out + c] = y;
            for (int64_t k = 0; k < n_draws; ++k)
                out[((clean + k) * T + t) * d_out + c] =
                    y + sigma * or_noise_value(kind, seed, draw_begin + k, t, c, d_out, flags);
        }
}

/* Embedding reassembly ("Dust: every token is a member of the population",
 * "What the released code actually does", step 7: "a scatter-add for an
 * embedding"): the error estimate of token t adds into the row of its token
 * id, gE[v][c] = scale * sum_{t : ids[t] = v} g[t][c], summed in token order.
 * Returns the number of ids outside [0, V) (skipped). */
OR_EXPORT int64_t dust_oracle_scatter_gE(const double* g, const int32_t* ids, int64_t T,
                                         int64_t d, int64_t V, double scale, double* gE) {
    int64_t bad = 0;
    for (int64_t q = 0; q < V * d; ++q) gE[q] = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t v = ids[t];
        if (v < 0 || v >= V) {
            ++bad;
            continue;
        }
        for (int64_t c = 0; c < d; ++c) gE[v * d + c] += g[t * d + c];
    }
    for (int64_t q = 0; q < V * d; ++q) gE[q] *= scale;
    return bad;
}

/* Local scores of blocks whose output does not reach the loss directly
 * ("Dust: every token is a member of the population", section "What the
 * released code actually does", step 4): the score of a jittered draw at
 * token s is c_s = -<g_s, delta_o_s>, the estimated output error g_s against
 * the change delta_o_s of the block's output under that draw. Returned as the
 * first-order loss change delta[k][s] = <g_s, delta_o[k][s]>, the quantity
 * the scan consumes (its reduction -delta is the page's c_s).
 *   g [T][d], delta_o [K][T][d], delta [K][T]. */
OR_EXPORT void dust_oracle_local_score(const double* g, const double* delta_o, int64_t K,
                                       int64_t T, int64_t d, double* delta) {
#pragma omp parallel for schedule(static)
    for (int64_t q = 0; q < K * T; ++q) {
        const int64_t t = q % T;
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j) acc += g[t * d + j] * delta_o[q * d + j];
        delta[q] = acc;
    }
}

/* Loss changes of a planted per-token quadratic loss, the workload of the
 * configurations this project measures:
 *   delta[k][t] = sigma <dplant_t, a_t^(draw_begin+k)>
 *                 + curv * 0.5 sigma^2 |a_t^(draw_begin+k)|^2 + eps[k][t].
 * For a loss L_t(y) = <dplant_t, y> + 0.5 curv |y|^2 this is exactly
 * L_t(y + sigma a) - L_t(y). dplant is [T][d_out]; eps (may be NULL) and
 * delta are [n_draws][T]. */
OR_EXPORT void dust_oracle_planted_delta(double* delta, const double* dplant,
                                         const double* eps, int64_t n_draws, int64_t T,
                                         int64_t d_out, uint64_t seed, int32_t kind,
                                         int64_t draw_begin, double sigma, double curv,
                                         uint32_t flags) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t k = 0; k < n_draws; ++k) {
            double dot = 0.0, sq = 0.0;
            for (int64_t c = 0; c < d_out; ++c) {
                double a = or_noise_value(kind, seed, draw_begin + k, t, c, d_out, flags);
                dot += dplant[t * d_out + c] * a;
                sq += a * a;
            }
            double e = eps ? eps[k * T + t] : 0.0;
            delta[k * T + t] = sigma * dot + curv * 0.5 * sigma * sigma * sq + e;
        }
    }
}
