/*
 * dust.h — C ABI of the GB300 (sm_103a) library for Dust's per-token
 * zeroth-order weight-gradient estimator of one linear layer y_t = W x_t.
 *
 * What the library computes ("Dust: every token is a member of the
 * population", ai.satyajit.si, section "Perturb the activations, not the
 * weights", the three equations for r_t, g_t and G_W):
 *
 *   c[i][t]  = -(delta[i][t] - mean_j delta[j][t])       centred loss reduction
 *   r[i][t]  = sum_{s >= t, same sequence} gamma^(s-t) c[i][s]   credit scan
 *   g[t][c]  = -(1 / (K sigma)) sum_i r[i][t] a_t^(i)[c]         output error
 *   GW[c][j] = scale * sum_t g[t][c] x[t][j]                     weight gradient
 *
 * delta[i][t] is the loss change L(perturbed) - L(clean) of draw i at token t,
 * so the reward (loss reduction) is its negative, as in the page's section
 * "What the released code actually does" (step 2: reward = clean loss minus
 * perturbed loss, centred across draws that share a forward). The
 * contraction is that section's step 7 (an einsum over tokens; `scale`
 * carries the optional division by the token count).
 *
 * The jitter a_t^(i) ~ N(0, I) (or Rademacher +-1) is never stored: it is
 * regenerated from a counter-based hash, the murmur3 fmix32 family of "RandOpt
 * Speedrun", section "What was slow, and the fix". This library's definition:
 *
 *   fmix32      MurmurHash3's 32-bit finaliser
 *   seed_key    fmix32(lo32(seed) ^ fmix32(hi32(seed) + 0x9E3779B9))
 *   draw_key    fmix32(seed_key ^ (2*i + s) * 0x9E3779B9)    (mod 2^32)
 *   word        fmix32(draw_key(i, s) ^ (t * d_out + c))      (mod 2^32)
 *   Rademacher  a = +1 if word(i,t,c,0) < 2^31, else -1
 *   Packed      (DUST_NOISE_RADEMACHER_PACKED) 32 signs per word: channel c
 *               takes bit c mod 32 of word(i, t, 32 floor(c/32), 0); bit 0
 *               gives +1, bit 1 gives -1
 *   Gaussian    pair p = c & ~1, w0 = word(i,t,p,0), w1 = word(i,t,p,1),
 *               u1 = 1 - (w0 >> 9) 2^-23, u2 = (w1 >> 9) 2^-23,
 *               rho = sqrt(-2 ln u1); even c: rho cos(2 pi u2),
 *               odd c: rho sin(2 pi u2) (the last channel of an odd d_out
 *               takes the cosine).
 *   Antithetic  (DUST_ANTITHETIC) draw i uses base draw i >> 1 times
 *               (-1)^(i & 1): draws 2j and 2j+1 are an opposite-sign pair.
 * i is the absolute draw index (draw_begin + local index); t is the row of the
 * flattened token matrix. T * d_out must not exceed 2^32.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are device memory of the current device; the
 *    caller owns every buffer (this library allocates no device memory).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Work is
 *    enqueued asynchronously on it; no entry point synchronises the device
 *    except dust_last_error.
 *  - Argument errors are detected on the host before anything is enqueued;
 *    the call then returns a non-zero dust_status and launches nothing.
 *  - A failed launch returns DUST_ERR_CUDA. Device-side errors (a bounded wait
 *    that ran out) are recorded in a device status word read by
 *    dust_last_error.
 *  - Row-major, contiguous layouts unless a leading dimension is given.
 *  - bf16 is IEEE bfloat16 (1-8-7), stored as uint16.
 */
#ifndef DUST_H
#define DUST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DUST_OK = 0,
    DUST_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum/flag */
    DUST_ERR_RANGE = 2,        /* a size beyond a documented limit */
    DUST_ERR_UNSUPPORTED = 3,  /* valid request this build cannot serve */
    DUST_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    DUST_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out */
    DUST_ERR_WORKSPACE = 6     /* workspace missing, too small or misaligned */
} dust_status;

typedef enum {
    DUST_NOISE_RADEMACHER = 0,
    DUST_NOISE_GAUSSIAN = 1,
    DUST_NOISE_RAW_WORDS = 2,  /* dust_noise only: the uint32 hash words */
    DUST_NOISE_RADEMACHER_PACKED = 3  /* +-1 signs, 32 per hash word */
} dust_noise_kind;

typedef enum {
    DUST_F32 = 0,
    DUST_BF16 = 1,
    DUST_U32 = 2               /* dust_noise with DUST_NOISE_RAW_WORDS only */
} dust_dtype;

/* Flags (bitwise OR). */
enum {
    DUST_CENTER = 1u,          /* centre each token's loss changes over the K draws (K > 1) */
    DUST_ANTITHETIC = 2u,      /* draws 2j, 2j+1 are an opposite-sign pair (needs even K,
                                  even draw_begin for the estimator) */
    DUST_ACCUMULATE = 4u,      /* GW += result instead of GW = result */
    DUST_FORCE_UNFUSED = 8u,   /* estimator: write g to the workspace, then contract */
    DUST_FORCE_FUSED = 16u,    /* estimator: produce g tiles inside the contraction
                                  (needs bf16 X, d_in <= 512, d_in % 8 == 0,
                                  d_out % 8 == 0, K <= 64, not the packed noise;
                                  else DUST_ERR_UNSUPPORTED) */
    DUST_WORD_STREAM1 = 32u,   /* dust_noise RAW_WORDS: words of stream s = 1 */
    DUST_FORCE_SIMT = 64u      /* estimator: contraction on CUDA cores (fp32 FFMA) */
};

/* Contraction paths reported by dust_estimate_gW_path. */
typedef enum {
    DUST_PATH_FUSED_TC = 1,    /* fused g-producer + tcgen05 MMA, bf16 in, fp32 accumulate
                                  (g never written to HBM); opt-in via DUST_FORCE_FUSED */
    DUST_PATH_UNFUSED_TC = 2,  /* weighting kernel -> g (bf16) -> tcgen05 GEMM; default for bf16 */
    DUST_PATH_SIMT = 3         /* weighting kernel -> g (fp32 or bf16) -> FFMA GEMM */
} dust_path;

/* Limits. */
#define DUST_MAX_DRAWS 8192          /* K and n_draws */
#define DUST_MAX_COUNTER 4294967296LL /* T * d_out */

/* Human-readable name of a status. Never NULL; static storage. */
const char* dust_status_string(dust_status s);

/* Library version as major*10000 + minor*100 + patch. */
int32_t dust_version(void);

/*
 * dust_noise — materialise the jitter of draws [draw_begin, draw_begin +
 * n_draws): out[k][t][c] = a_t^(draw_begin+k)[c] ("Perturb the activations,
 * not the weights": y_t -> y_t + sigma a_t with a_t ~ N(0, I)). Used by tests
 * and to synthesise inputs; the estimator itself never stores the jitter.
 *   out       device, [n_draws][T][d_out]; DUST_F32 or DUST_BF16 values
 *             (Rademacher/Gaussian) or DUST_U32 words (RAW_WORDS; stream 0,
 *             or stream 1 with DUST_WORD_STREAM1; DUST_ANTITHETIC ignored).
 *   draw_begin >= 0, n_draws in [0, DUST_MAX_DRAWS], T >= 0, d_out >= 0,
 *   T * d_out <= 2^32 (else DUST_ERR_RANGE). Empty sizes launch nothing.
 */
dust_status dust_noise(void* out, dust_dtype out_dtype, uint64_t seed,
                       dust_noise_kind kind, int64_t draw_begin, int64_t n_draws,
                       int64_t T, int64_t d_out, uint32_t flags, void* stream);

/*
 * dust_jitter_apply — the jittered forward's output perturbation, in place:
 * y[t][c] += sigma * a_t^(draw)[c] (same section; the jitter is added after
 * the layer's product, i.e. the split form of "Scaling To Unfathomable
 * Depth", section "Kernel Recipes").
 *   y      device, T rows of d_out values with row stride ld_y >= d_out
 *          (elements); DUST_F32 or DUST_BF16 (bf16 rounded to nearest even).
 *   kind   DUST_NOISE_RADEMACHER, DUST_NOISE_GAUSSIAN or
 *          DUST_NOISE_RADEMACHER_PACKED; draw >= 0.
 */
dust_status dust_jitter_apply(void* y, dust_dtype y_dtype, int64_t ld_y, int64_t T,
                              int64_t d_out, uint64_t seed, dust_noise_kind kind,
                              int64_t draw, float sigma, uint32_t flags, void* stream);

/*
 * dust_forward_jitter — the jittered forward of a linear layer for several
 * draws at once: the product y = X W^T is formed once on the tensor cores
 * and each draw's output y + sigma * a_t^(draw) is written from it ("Dust:
 * every token is a member of the population", section "Perturb the
 * activations, not the weights": each population member runs the layer with
 * its own jitter on the output; split form of "Scaling To Unfathomable
 * Depth", section "Kernel Recipes"):
 *   Y[s][t][c] = y[t][c]                                   s < clean
 *   Y[s][t][c] = y[t][c] + sigma * a_t^(draw_begin + k)[c]  s = clean + k
 * y is accumulated in fp32 from bf16 products; each output is rounded once
 * to bf16 (nearest even) after the jitter is added in fp32.
 *   X      device, bf16 [T][d_in] row-major.   W  device, bf16 [d_out][d_in].
 *   Y      device, bf16 [clean + n_draws][T][d_out], written (not read).
 *          X, W, Y 16-byte aligned; d_in > 0 and d_out multiples of 8
 *          (else DUST_ERR_UNSUPPORTED). Caller owns all three.
 *   kind   DUST_NOISE_RADEMACHER, DUST_NOISE_GAUSSIAN or
 *          DUST_NOISE_RADEMACHER_PACKED; flags 0 or DUST_ANTITHETIC.
 *   clean  0 or 1; n_draws in [0, DUST_MAX_DRAWS]; draw_begin >= 0 with
 *          draw_begin + n_draws <= 2^31; T * d_out <= 2^32 (DUST_ERR_RANGE).
 * Asynchronous on `stream`; a bounded device wait that runs out is reported
 * by dust_last_error as DUST_ERR_TIMEOUT.
 */
dust_status dust_forward_jitter(const void* X, const void* W, int64_t T, int64_t d_in,
                                int64_t d_out, uint64_t seed, dust_noise_kind kind,
                                int64_t draw_begin, int64_t n_draws, float sigma,
                                uint32_t flags, int32_t clean, void* Y, void* stream);

/*
 * dust_local_score — loss changes of draws scored locally: for blocks whose
 * output does not reach the loss (attention internals), each jittered draw k
 * is scored at token s against the block output's estimated error ("Dust:
 * every token is a member of the population", "What the released code
 * actually does", step 4: c_s = -<g_s, delta_o_s>). Returned as the loss
 * change delta[k][s] = <g_s, delta_o[k][s]>, the input dust_credit_scan and
 * dust_estimate_gW take (their reduction -delta is the page's c_s; keys and
 * values then use gamma 0.98 over later tokens, queries gamma 0).
 *   g        device [T][d], the block output's estimated error, DUST_F32 or
 *            DUST_BF16.
 *   delta_o  device [K][T][d], the change of the block output under each
 *            draw, DUST_F32 or DUST_BF16.
 *   delta    device f32 [K][T], written.
 * Sums run in fp32 in a fixed order (deterministic).
 */
dust_status dust_local_score(const void* g, dust_dtype g_dtype, const void* delta_o,
                             dust_dtype o_dtype, int64_t K, int64_t T, int64_t d,
                             float* delta, void* stream);

/*
 * dust_scatter_gE_workspace / dust_scatter_gE — embedding reassembly ("Dust:
 * every token is a member of the population", "What the released code
 * actually does", step 7: the error estimate becomes a weight gradient by "a
 * scatter-add for an embedding"): gE[v][c] = scale * sum over the tokens t
 * with ids[t] = v of g[t][c].
 *   g         device [T][d], DUST_F32 or DUST_BF16 (finite values).
 *   ids       device int32 [T]; ids outside [0, V) are skipped and make
 *             dust_last_error report DUST_ERR_INVALID_ARG.
 *   gE        device f32 [V][d]; overwritten, or accumulated into with
 *             DUST_ACCUMULATE (the only flag).
 *   workspace device, >= dust_scatter_gE_workspace(T, V, d) bytes, 256-byte
 *             aligned (about 8 V d + 4 T + 8 V bytes); contents on entry are
 *             ignored.
 * Deterministic whatever the order in which tokens arrive: sums are kept in
 * 64-bit fixed point with a step of 2^-s chosen per call so that
 * max|g| * (largest count of one id) * 2^s < 2^61; each term is rounded once
 * to that step, and the result is rounded to fp32 at the end.
 */
dust_status dust_scatter_gE_workspace(size_t* bytes, int64_t T, int64_t V, int64_t d);
dust_status dust_scatter_gE(const void* g, dust_dtype g_dtype, const int32_t* ids, int64_t T,
                            int64_t d, int64_t V, float scale, uint32_t flags, float* gE,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * dust_estimate_gE_workspace / dust_estimate_gE — the whole path for an
 * embedding E [V][d] whose looked-up rows are jittered: centring and the
 * credit scan of delta (as dust_credit_scan), the reward weighting into an
 * fp32 error g [T][d] (as dust_error_estimate; d plays d_out), and the
 * scatter-add of g into gE by token id (as dust_scatter_gE).
 *   ids          device int32 [T]; delta device f32 [K][T]; seq_offsets as
 *                for dust_credit_scan.
 *   kind         a value noise kind; flags DUST_CENTER, DUST_ANTITHETIC,
 *                DUST_ACCUMULATE. Other arguments as for dust_estimate_gW.
 *   workspace    device, >= dust_estimate_gE_workspace(...) bytes, 256-byte
 *                aligned.
 */
dust_status dust_estimate_gE_workspace(size_t* bytes, int64_t T, int64_t d, int64_t V,
                                       int64_t K);
dust_status dust_estimate_gE(const int32_t* ids, int64_t T, int64_t V, const float* delta,
                             int64_t K, int64_t d, const int32_t* seq_offsets, int64_t n_seq,
                             uint64_t seed, dust_noise_kind kind, int64_t draw_begin,
                             float sigma, float gamma, float scale, uint32_t flags, float* gE,
                             void* workspace, size_t ws_bytes, void* stream);

/*
 * dust_credit_scan_workspace / dust_credit_scan — centring and the reverse
 * credit scan on their own (the r_t equation; centring as described above).
 *   delta       device f32 [K][T] loss changes.
 *   seq_offsets device i32 [n_seq + 1]: 0 = o_0 < o_1 < ... < o_n_seq = T
 *               (each sequence non-empty); the scan restarts at every
 *               sequence. n_seq >= 1 when T > 0.
 *   gamma       credit decay, finite, |gamma| <= 1.
 *   flags       DUST_CENTER or 0.
 *   r           device f32 [T][K] (token-major): r[t][i] = r_t^(i).
 *   workspace   device, >= the size reported by dust_credit_scan_workspace,
 *               256-byte aligned.
 */
dust_status dust_credit_scan_workspace(size_t* bytes, int64_t K, int64_t T);
dust_status dust_credit_scan(const float* delta, int64_t K, int64_t T,
                             const int32_t* seq_offsets, int64_t n_seq, float gamma,
                             uint32_t flags, float* r, void* workspace, size_t ws_bytes,
                             void* stream);

/*
 * dust_credit_scan_noalloc — the same centring + credit scan as
 * dust_credit_scan, for callers that cannot allocate device memory (for
 * example a plugin whose host framework's pooling allocator owns all device
 * memory, or a latency-critical loop where cudaMalloc/cudaFree may
 * synchronise the device). The paper has no counterpart: this is a memory
 * management variant of the library, not a step of the method.
 * Its scratch is a fixed array of dust_credit_scan_noalloc_capacity() bytes
 * (8 MiB) built into the library as a static device variable, held by every
 * GPU that loads it until the process exits; it calls no cudaMalloc or
 * cudaFree. The caller still passes delta, seq_offsets and r (same meaning,
 * layout and results as dust_credit_scan). A call needing more scratch than
 * the capacity (4 T + 8 (K + 1) ceil(T/256) bytes, each of its four parts
 * rounded up to 256) returns DUST_ERR_RANGE.
 * The first call on a device looks up the array's device address with that
 * device current; make it before any stream capture. All calls share the
 * array: calls whose GPU work overlaps (several streams or host threads on
 * one device) race. Each call writes every scratch word it reads, so no
 * clearing between calls is needed.
 */
size_t dust_credit_scan_noalloc_capacity(void);
dust_status dust_credit_scan_noalloc(const float* delta, int64_t K, int64_t T,
                                     const int32_t* seq_offsets, int64_t n_seq, float gamma,
                                     uint32_t flags, float* r, void* stream);

/*
 * dust_error_estimate — reward-weighted noise on its own (the g_t equation):
 * g[t][c] = -(1/(K sigma)) sum_{i<K} r[t][i] a_t^(draw_begin+i)[c].
 *   r      device f32 [T][K] (the output of dust_credit_scan).
 *   g      device [T][d_out], DUST_F32 or DUST_BF16 (rounded to nearest even).
 *   sigma  finite, non-zero.
 */
dust_status dust_error_estimate(const float* r, int64_t K, int64_t T, int64_t d_out,
                                uint64_t seed, dust_noise_kind kind, int64_t draw_begin,
                                float sigma, uint32_t flags, void* g, dust_dtype g_dtype,
                                void* stream);

/*
 * dust_contract_workspace / dust_contract — the contraction on its own (the
 * G_W equation): GW[c][j] = scale * sum_t g[t][c] x[t][j].
 *   g       device [T][d_out]; X device [T][d_in]; both DUST_BF16 (tensor
 *           cores, fp32 accumulation; needs d_in % 8 == 0, d_out % 8 == 0 and
 *           16-byte aligned bases, otherwise CUDA cores) or both DUST_F32
 *           (CUDA cores, fp32).
 *   flags   DUST_ACCUMULATE, DUST_FORCE_SIMT.
 *   gW      device f32 [d_out][d_in], 16-byte aligned.
 *   workspace as for dust_estimate_gW (split-token partials).
 */
dust_status dust_contract_workspace(size_t* bytes, int64_t T, int64_t d_in, int64_t d_out,
                                    dust_dtype dtype, uint32_t flags);
dust_status dust_contract(const void* g, const void* X, dust_dtype dtype, int64_t T,
                          int64_t d_in, int64_t d_out, float scale, uint32_t flags, float* gW,
                          void* workspace, size_t ws_bytes, void* stream);

/*
 * dust_estimate_gW_workspace / dust_estimate_gW — the whole path, delta and X
 * to the weight gradient GW (the three equations above, in one call).
 *   X           device [T][d_in], DUST_BF16 (tensor-core path, fp32
 *               accumulation) or DUST_F32 (CUDA-core fp32 path). 16-byte
 *               aligned base; for DUST_BF16 the tensor-core paths also need
 *               d_in % 8 == 0 and d_out % 8 == 0 (otherwise the CUDA-core
 *               contraction runs).
 *   delta       device f32 [K][T]; seq_offsets as for dust_credit_scan.
 *   kind        DUST_NOISE_RADEMACHER, DUST_NOISE_GAUSSIAN or
 *               DUST_NOISE_RADEMACHER_PACKED.
 *   draw_begin  absolute index of the first draw (>= 0).
 *   sigma       finite, non-zero; gamma finite, |gamma| <= 1; scale finite.
 *   flags       DUST_CENTER, DUST_ANTITHETIC, DUST_ACCUMULATE and at most one
 *               of DUST_FORCE_UNFUSED / DUST_FORCE_FUSED / DUST_FORCE_SIMT.
 *   gW          device f32 [d_out][d_in], W's layout, 16-byte aligned;
 *               overwritten, or accumulated into with DUST_ACCUMULATE.
 *   workspace   device, >= dust_estimate_gW_workspace(...) bytes, 256-byte
 *               aligned; contents on entry are ignored.
 * The result is a deterministic function of the inputs (no floating-point
 * atomics): two calls with the same arguments give bit-identical gW.
 * With gamma = 0 the credit scan is the identity (r = c); for K <= 32 the
 * weighting kernel then centres delta itself and no scan kernel runs, with
 * the same bits as the scan path (the per-token mean is summed in the same
 * order). Sharding: calls over disjoint whole sequences (the other rows of X
 * zero or excluded), or over disjoint draw ranges (draw_begin; delta centred
 * over all K beforehand, DUST_CENTER off, scale = the range's share of K),
 * accumulate (DUST_ACCUMULATE) to the unsharded estimate.
 * Graph replay: from the second call with identical arguments (every pointer
 * and scalar) on the current device, the call's launches are captured once
 * into a CUDA graph and later calls launch that graph on `stream`; it reads
 * and writes the same buffers, so it sees their current contents. Up to 16
 * argument sets are kept per device (least recently used dropped). Bypassed
 * while dust_profile_enable(1) is on.
 */
dust_status dust_estimate_gW_workspace(size_t* bytes, int64_t T, int64_t d_in,
                                       int64_t d_out, int64_t K, dust_dtype x_dtype,
                                       uint32_t flags);
dust_status dust_estimate_gW(const void* X, dust_dtype x_dtype, int64_t T, int64_t d_in,
                             const float* delta, int64_t K, int64_t d_out,
                             const int32_t* seq_offsets, int64_t n_seq, uint64_t seed,
                             dust_noise_kind kind, int64_t draw_begin, float sigma,
                             float gamma, float scale, uint32_t flags, float* gW,
                             void* workspace, size_t ws_bytes, void* stream);

/* The contraction path dust_estimate_gW would take for these arguments
 * (a dust_path value), or a negative dust_status on invalid arguments. */
int32_t dust_estimate_gW_path(int64_t T, int64_t d_in, int64_t d_out, int64_t K,
                              dust_dtype x_dtype, uint32_t flags);

/*
 * dust_estimate_gW_sites — dust_estimate_gW for several layers ("sites") in
 * one stream-ordered pass, as in the page's section "What the released code
 * actually does" (one update covers every linear layer): sites[i] is computed
 * exactly as dust_estimate_gW would compute it with that site's arguments and
 * the shared x_dtype, kind, draw_begin, scale and flags, and the results are
 * bit-identical to such calls made one after another. What differs is the
 * order on the device: the sites run on internal compute lanes of the current
 * device (streams created on first use, never destroyed), site i on lane
 * i mod L, each lane with a companion stream of the device's highest priority
 * for its sites' contraction kernels. All of them start after everything
 * enqueued on `stream` before this call, and `stream` waits for all of them
 * at its end (on error paths too). So one site's contraction (tensor cores)
 * runs beside later sites' weighting (transcendental and integer pipes). The
 * same delta or seq_offsets may serve several sites (Dust's loss changes are
 * one per token and draw for the whole model).
 *
 * Because sites run concurrently, what a site writes (its gW, and its
 * workspace) must not overlap any buffer of another site (X, delta,
 * seq_offsets, gW or workspace): checked on the host, DUST_ERR_INVALID_ARG
 * otherwise. Every argument of every site is checked before anything is
 * enqueued. At most 4096 sites (DUST_ERR_RANGE). Graph replay as for
 * dust_estimate_gW: from the second call with identical arguments (the whole
 * site array included), the call is captured once into a CUDA graph, lanes
 * and all, and later calls launch that graph on `stream`; the graph keeps
 * each kernel's stream priority (the lanes' and the contraction streams'),
 * whatever the priority of `stream`. Concurrent calls on one device are
 * serialised on the host while they enqueue.
 */
typedef struct {
    const void* X;                   /* device [T][d_in], x_dtype */
    int64_t T, d_in, d_out;
    const float* delta;              /* device f32 [K][T] loss changes */
    int64_t K;
    const int32_t* seq_offsets;      /* device i32 [n_seq + 1] */
    int64_t n_seq;
    uint64_t seed;                   /* this site's noise seed */
    float sigma, gamma;
    float* gW;                       /* device f32 [d_out][d_in] */
    void* workspace;                 /* device, dust_estimate_gW_workspace bytes */
    size_t ws_bytes;
} dust_site;

dust_status dust_estimate_gW_sites(const dust_site* sites, int64_t n_sites, dust_dtype x_dtype,
                                   dust_noise_kind kind, int64_t draw_begin, float scale,
                                   uint32_t flags, void* stream);
/* The number L of compute lanes per device (fixed when the library is built). */
int32_t dust_estimate_gW_sites_lanes(void);

/*
 * dust_estimate_gW_host — the same computation from HOST buffers: copies
 * X_host -> X_dev, delta_host -> delta_dev and seq_offsets_host -> seq_dev,
 * runs dust_estimate_gW, and copies gW_dev -> gW_host. With DUST_ACCUMULATE,
 * gW_host is first copied to gW_dev. X, the large input, is copied on an
 * internal copy stream of the current device (created on first use, never
 * destroyed) that starts after earlier work on `stream`; the scan and the
 * weighting run on `stream` meanwhile, and `stream` waits for the copy
 * before the contraction (on error paths too), so everything this call
 * does is complete once `stream` is. Concurrent calls on one device share
 * the copy stream. Host buffers should be page-locked (else the copies are
 * synchronous) and must stay valid until the stream has completed; the
 * caller synchronises before reading gW_host. Device staging buffers are
 * caller-owned with the sizes of the host ones.
 */
dust_status dust_estimate_gW_host(const void* X_host, void* X_dev, dust_dtype x_dtype,
                                  int64_t T, int64_t d_in, const float* delta_host,
                                  float* delta_dev, int64_t K, int64_t d_out,
                                  const int32_t* seq_offsets_host, int32_t* seq_dev,
                                  int64_t n_seq, uint64_t seed, dust_noise_kind kind,
                                  int64_t draw_begin, float sigma, float gamma, float scale,
                                  uint32_t flags, float* gW_host, float* gW_dev,
                                  void* workspace, size_t ws_bytes, void* stream);

/*
 * dust_estimate_gW_host_sites — dust_estimate_gW_host for several layers
 * ("sites") in one stream-ordered pass, as in the page's section "What the
 * released code actually does" (one update covers every linear layer):
 * sites[i] is computed exactly as dust_estimate_gW_host would compute it with
 * that site's arguments and the shared x_dtype, kind, draw_begin, scale and
 * flags, and the results are bit-identical to such calls made one after
 * another. What differs is the copying and the order on the device: the
 * inputs of later sites travel host -> device while earlier sites compute,
 * and with more than one site the sites compute on the compute lanes of
 * dust_estimate_gW_sites (site i on lane i mod L). Site 0's loss changes and
 * offsets are copied on `stream`; then, on the internal copy stream and after
 * everything enqueued on `stream` before this call, X of site 0 and, for each
 * later site, its loss changes, offsets and X, in site order. Each site's
 * kernels wait for its own loss changes before they start and for its X
 * before the contraction. Every copy and every kernel of the call has
 * completed when the call's work on `stream` has (also on error paths).
 *
 * Because the copy stream writes a site's staging buffers (X_dev of every
 * site; delta_dev and seq_dev of sites after the first) while earlier sites
 * compute, those buffers must not overlap any device buffer of the call
 * (any site's X_dev, delta_dev, seq_dev, gW_dev or workspace); and because
 * sites compute concurrently, a site's workspace and gW_dev must not overlap
 * a buffer of another site. Checked on the host, DUST_ERR_INVALID_ARG
 * otherwise. Every argument of every site is checked before anything is
 * enqueued. At most 4096 sites (DUST_ERR_RANGE).
 * Results: every site but the last writes gW_dev, which an internal return
 * stream copies to gW_host while later sites compute (gW_dev of those sites
 * is therefore also read out of stream order and falls under the overlap
 * rule); the last site follows dust_estimate_gW_host's rule (gW_host written
 * in place over the host link when page-locked and device-mapped, else
 * through gW_dev and a copy on `stream`).
 */
typedef struct {
    const void* X_host;              /* host [T][d_in], x_dtype; page-locked for overlap */
    void* X_dev;                     /* device staging [T][d_in] */
    int64_t T, d_in, d_out;
    const float* delta_host;         /* host [K][T] loss changes */
    float* delta_dev;                /* device staging [K][T] */
    int64_t K;
    const int32_t* seq_offsets_host; /* host [n_seq + 1] */
    int32_t* seq_dev;                /* device staging [n_seq + 1] */
    int64_t n_seq;
    uint64_t seed;                   /* this site's noise seed */
    float sigma, gamma;
    float* gW_host;                  /* host [d_out][d_in] result */
    float* gW_dev;                   /* device [d_out][d_in] */
    void* workspace;                 /* device, dust_estimate_gW_workspace bytes */
    size_t ws_bytes;
} dust_host_site;

dust_status dust_estimate_gW_host_sites(const dust_host_site* sites, int64_t n_sites,
                                        dust_dtype x_dtype, dust_noise_kind kind,
                                        int64_t draw_begin, float scale, uint32_t flags,
                                        void* stream);

/*
 * Per-kernel timing for benchmarks (no counterpart on the pages: this is
 * measurement plumbing). While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on its stream; dust_profile_read
 * waits for the recorded events, returns per-kernel launch counts and summed
 * durations, and clears the record. Process-global state: enable it only in
 * a single-threaded benchmark. At most 65536 launches are recorded between
 * reads (later launches are not timed).
 */
typedef struct {
    char name[32];       /* kernel family, e.g. "weight", "gemm_tc", "scan" */
    int64_t launches;
    double total_ms;
} dust_profile_entry;

dust_status dust_profile_enable(int32_t on);
/* Writes up to max_entries entries; returns how many were written (>= 0) or a
 * negative dust_status. */
int32_t dust_profile_read(dust_profile_entry* out, int32_t max_entries);

/*
 * Pipe-rate probes for rooflines (no counterpart on the pages: measurement
 * plumbing). dust_pipe_probe enqueues on `stream` one launch of a
 * throughput kernel that keeps every SM's schedulers busy with independent
 * chains of one kind of operation, written in inline PTX:
 *   DUST_PIPE_XU     lg2.approx, sqrt.approx, sin.approx, cos.approx
 *                    (the transcendentals of a Box-Muller pair), counted ops
 *                    = those four instructions;
 *   DUST_PIPE_ALU    two shr.b32 and one lop3.b32 per step (the integer ALU
 *                    pipe), ops = all three;
 *   DUST_PIPE_FMA    fma.rn.f32, ops = FLOP (2 per FMA);
 *   DUST_PIPE_ISSUE  three fma.rn.f32 per lop3.b32, ops = lane instructions
 *                    (neither pipe binds before instruction issue does).
 * Each chain is nonlinear in its own state, so the assembler cannot fold
 * steps together.
 *
 * *ops receives the number of counted operations the launch performs; the
 * caller times the launch with CUDA events on `stream` and divides. `sink`
 * is a device float buffer of at least dust_pipe_probe_threads() elements:
 * each thread stores its result there only when the result's bits match a
 * fixed NaN pattern, which keeps the chains live (in practice almost never).
 * `steps` (1 .. 2^30, rounded up to a multiple of 4, which *ops counts)
 * sets the launch's length: about 2^14 steps take a few milliseconds on a
 * GB300. Returns DUST_ERR_INVALID_ARG for an unknown pipe, a bad step count
 * or a null pointer.
 */
typedef enum {
    DUST_PIPE_XU = 0,
    DUST_PIPE_ALU = 1,
    DUST_PIPE_FMA = 2,
    DUST_PIPE_ISSUE = 3
} dust_pipe;

dust_status dust_pipe_probe(int32_t pipe, int64_t steps, double* ops, void* sink,
                            void* stream);
/* Threads of one probe launch (SM count x 4 CTAs x 512), i.e. the size of
 * `sink` in floats; a negative dust_status if the device cannot be queried. */
int32_t dust_pipe_probe_threads(void);

/*
 * dust_debug_inject_timeout — test hook for the device-side failure path (no
 * counterpart on the pages). With on != 0, the next tensor-core contraction
 * launched by this process (dust_contract or the unfused dust_estimate_gW
 * path) makes its MMA thread wait on an mbarrier that no thread ever arrives
 * at. The wait gives up after its 1 s limit, the kernel lets its issued TMA
 * copies land, frees its tensor memory and returns without writing gW, and
 * dust_last_error then reports DUST_ERR_TIMEOUT; the CUDA context stays
 * usable. No fault, trap or hang is involved. One-shot; process-global.
 */
dust_status dust_debug_inject_timeout(int32_t on);

/*
 * dust_last_error — synchronise `stream`, then return and clear the device
 * status word (DUST_OK; DUST_ERR_TIMEOUT when a kernel's bounded wait ran out
 * since the last call; DUST_ERR_INVALID_ARG when dust_scatter_gE or
 * dust_estimate_gE met a token id outside [0, V)). DUST_ERR_CUDA if the
 * synchronisation failed.
 */
dust_status dust_last_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DUST_H */
