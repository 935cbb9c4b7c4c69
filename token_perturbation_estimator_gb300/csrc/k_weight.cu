// Reward weighting with in-register noise regeneration:
//   g[t][c] = -(1/(K sigma)) sum_i r_t^(i) a_t^(i)[c]
// ("Dust: every token is a member of the population", section "Perturb the
// activations, not the weights", the g_t equation). The jitter a is rebuilt
// from the hash for every (draw, token, channel) and used once; nothing of it
// is stored.
//
// Mapping: one warp per token, CPT channels per lane (CPT/2 Box-Muller pairs
// or CPT signs; packed signs: the 32 channels of one hash word; Gaussian with
// d_out a multiple of 1024: 32 channels), 8 tokens x 32 lanes' channels per
// CTA. The per-token rewards are already multiplied by -1/(K sigma); for
// antithetic pairs they are the pair's reward difference, one per base draw.
// They and the per-draw keys are staged in shared memory 64 draws at a time
// and read as warp-wide broadcasts. Source 2 (below) is the exception: its
// rewards are shuffled from lane to lane and its keys come from the host. The
// per-channel counters are pre-folded once per thread, so each element-draw
// costs the hash tail plus one FMA (Rademacher: the sign bit is xor-ed into
// the reward's sign bit).
//
// Reward sources (SRC): the credit scan's token-major rewards r [T][K]
// (0), the same plus the scan's chunk carry P[t] carry[chunk][i] (1), or,
// when gamma = 0 and the scan is the identity (r_t = c_t), the loss changes
// themselves, Delta [K][T], centred over the draws here (2): c = -(Delta -
// mean), the mean of a token's K changes summed in draw order as the scan
// does. Source 2 takes K <= 32 (the library uses it up to K = 32, beyond
// which the longer prologue costs more than the scan): each warp loads its
// own token's K loss changes, one per lane, and centres them with shuffles,
// so no CTA barrier is taken (the narrow Gaussian lanes, short of registers,
// stage them through shared memory instead, CTA-wide).
#include "internal.cuh"
#include "noise.cuh"

namespace dust {

namespace {

#ifndef DUST_WEIGHT_CPT
#define DUST_WEIGHT_CPT 16
#endif
// Resident CTAs per SM that the register allocation must allow, per noise
// kind (narrow Gaussian lanes: 48 registers; Rademacher: 64). The narrow
// Gaussian lanes now serve only channel counts that are not a multiple of
// 1024 (the sweep's 512- and 1536-channel sites): there 5 CTAs per SM
// measured 0.65 % faster than 6 on the 1536-channel site with the scan's
// rewards (1439 -> 1430 us) and the same on the 512-channel sites.
#ifndef DUST_WEIGHT_MINB_G
#define DUST_WEIGHT_MINB_G 5
#endif
#ifndef DUST_WEIGHT_MINB_R
#define DUST_WEIGHT_MINB_R 4
#endif
// Gaussian with 32 channels per lane (16 Box-Muller pairs per draw, for d_out
// a multiple of 1024 and at most 64 noise draws per token): the per-draw
// reads and the per-thread setup and store spread over twice the pairs, at 3
// resident CTAs per SM.
#ifndef DUST_WEIGHT_MINB_GW
#define DUST_WEIGHT_MINB_GW 3
#endif
#ifndef DUST_WEIGHT_UNROLL
#define DUST_WEIGHT_UNROLL 2
#endif
// Loss changes read by each warp for its own token and centred with warp
// shuffles (no CTA barrier), for reward source 2 (K <= 32); 0: staged
// through shared memory by the whole CTA.
#ifndef DUST_WEIGHT_WARP_SRC
#define DUST_WEIGHT_WARP_SRC 1
#endif
constexpr bool kWarpSrc = DUST_WEIGHT_WARP_SRC != 0;
constexpr int kMinBlocksG = DUST_WEIGHT_MINB_G;
constexpr int kMinBlocksR = DUST_WEIGHT_MINB_R;
constexpr int kUnrollW = DUST_WEIGHT_UNROLL;
// Gaussian draw-loop unroll: the wide lanes (few draws) take 4 (measured:
// weighting 135.5 -> 133.4 us on the up-projection); the narrow ones keep 2
// (4 cost qkv's 16-draw weighting 2 %).
constexpr int unroll_of(int cpt) { return cpt == 32 ? 4 : kUnrollW; }
constexpr int kTok = 8;                 // tokens per CTA (one per warp)
constexpr int kCpt = DUST_WEIGHT_CPT;   // channels per lane (8 or 16)
constexpr int kCptWide = 32;            // channels per lane: packed signs, wide Gaussian
constexpr int kGroup = 64;              // draws staged per pass
static_assert(kCpt % 8 == 0, "channels per lane must be a multiple of 8");
constexpr int min_blocks(int kind, int cpt) {
    return kind == 1 ? (cpt == kCptWide ? DUST_WEIGHT_MINB_GW : kMinBlocksG) : kMinBlocksR;
}

template <typename OutT>
__device__ __forceinline__ void store8(OutT* g, int64_t row, int64_t d_out, int64_t c0,
                                       const float* acc, bool vec);

template <>
__device__ __forceinline__ void store8<float>(float* g, int64_t row, int64_t d_out, int64_t c0,
                                              const float* acc, bool vec) {
    float* p = g + row * d_out + c0;
    if (vec) {
        reinterpret_cast<float4*>(p)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (c0 + j < d_out) p[j] = acc[j];
    }
}

template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* g, int64_t row,
                                                      int64_t d_out, int64_t c0,
                                                      const float* acc, bool vec) {
    __nv_bfloat16* p = g + row * d_out + c0;
    if (vec) {
        __nv_bfloat162 h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
        *reinterpret_cast<uint4*>(p) = *reinterpret_cast<uint4*>(h);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (c0 + j < d_out) p[j] = __float2bfloat16_rn(acc[j]);
    }
}

// Folded stream keys of up to 32 base draws, made on the host for reward
// source 2 and read in the draw loop with a warp-uniform index.
struct DrawKeys {
    uint2 k[32];
};

// One draw's contribution to a lane's channels: rr is the draw's weighted
// reward for the token, key its folded stream keys.
template <int KIND, int CPT, int NF>
__device__ __forceinline__ void add_draw(float (&acc)[CPT], const uint32_t (&nf)[NF], float rr,
                                         uint2 key) {
    if (KIND == 1) {
#pragma unroll
        for (int p = 0; p < CPT / 2; ++p) {
            const float f0 = unit_ff(key.x, nf[p]);
            const float f1 = unit_ff(key.y, nf[p]);
            const float tr = rr * neg_radius(f0);
            float sn, cs;
            __sincosf(centred_angle(f1), &sn, &cs);
            acc[2 * p] = fmaf(tr, cs, acc[2 * p]);
            acc[2 * p + 1] = fmaf(tr, sn, acc[2 * p + 1]);
        }
    } else if (KIND == 3) {
        const uint32_t rb = __float_as_uint(rr);
        const uint32_t w = word_ff(key.x, nf[0]);
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[j] += __uint_as_float(rb ^ packed_sign_bit(w, j));
    } else {
        const uint32_t rb = __float_as_uint(rr);
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[j] += __uint_as_float(rb ^ sign_ff(key.x, nf[j]));
    }
}

template <int KIND, int CPT, int SRC, bool ANTI, typename OutT>
__global__ void __launch_bounds__(256, min_blocks(KIND, CPT))
    k_weight(const float* __restrict__ r, const float* __restrict__ P,
             const float* __restrict__ carry, int64_t K, int64_t T, int64_t d_out, uint32_t skey,
             int64_t draw_begin, float coef, OutT* __restrict__ g, bool vec_ok, int center,
             const DrawKeys keys) {
    __shared__ uint2 s_key[kGroup];  // folded keys of streams 0 and 1
    __shared__ float s_r[kTok][kGroup];
    __shared__ float s_raw[SRC == 2 ? kTok : 1][kGroup + 1];  // Delta of the CTA's tokens
    __shared__ float s_mean[kTok];
    __shared__ float s_part[SRC == 2 ? kTok : 1][kGroup / 8];
    pdl_wait();
    pdl_trigger();

    // Channels per lane: one 32-sign word for the packed signs.
    constexpr int cpt = CPT;
    static_assert(KIND != 3 || CPT == 32, "packed signs: one word per lane");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t tb = static_cast<int64_t>(blockIdx.x) * kTok;
    const int64_t t = tb + warp;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * (32 * cpt) + lane * cpt;
    const bool active = (t < T) && (c0 < d_out);

    // Pre-folded counters: pairs for the Gaussian, single channels for signs,
    // the group's first channel for packed signs.
    constexpr int kNf = (KIND == 1) ? cpt / 2 : (KIND == 3 ? 1 : cpt);
    uint32_t nf[kNf];
    const uint32_t base = static_cast<uint32_t>(t * d_out + c0);
#pragma unroll
    for (int j = 0; j < kNf; ++j) nf[j] = fold16(base + (KIND == 1 ? 2u * j : j));

    float acc[cpt];
#pragma unroll
    for (int j = 0; j < cpt; ++j) acc[j] = 0.0f;

    // With antithetic pairs, draws 2b and 2b + 1 carry +a and -a of base draw
    // b, so each base draw's noise is evaluated once, weighted by the
    // difference of the pair's rewards: the loop runs over Kb = K / 2 base
    // draws (draw_begin is even).
    // (Not for the narrow Gaussian lanes: their 40-register budget would spill.)
    if constexpr (SRC == 2 && kWarpSrc && !(KIND == 1 && CPT != kCptWide)) {
        // Lane k holds the token's loss change of draw k (K <= 32). The mean
        // over the draws is summed in the credit scan's order (sums of 8
        // draws in draw order, then those sums in order), so the result
        // equals the scan path's bit for bit. Lane b then holds base draw b's
        // weighted reward, broadcast draw by draw.
        constexpr unsigned kAll = 0xffffffffu;
        const int kk = static_cast<int>(K);
        const bool tok_ok = t < T;  // the same for the whole warp
        float dv = 0.0f;
        if (tok_ok && lane < kk) dv = r[static_cast<int64_t>(lane) * T + t];
        float mean = 0.0f;
        if (center && kk > 1) {
            for (int q = 0; 8 * q < kk; ++q) {
                const int hi = (8 * q + 8 < kk) ? 8 * q + 8 : kk;
                float part = 0.0f;
                for (int k = 8 * q; k < hi; ++k) part += __shfl_sync(kAll, dv, k);
                mean += part;
            }
            mean /= static_cast<float>(kk);
        }
        const int kb = ANTI ? kk / 2 : kk;
        const int i0 = ANTI ? 2 * lane : lane;
        const float d0 = __shfl_sync(kAll, dv, i0 & 31);
        const float d1 = __shfl_sync(kAll, dv, (i0 + 1) & 31);
        float v = 0.0f;
        if (lane < kb) {
            const float r0 = -(d0 - mean);
            if (ANTI) {
                const float r1 = -(d1 - mean);
                v = (r0 - r1) * coef;
            } else {
                v = r0 * coef;
            }
        }
        if (tok_ok) {
            // Lanes past d_out run the loop too (no memory access in it) so
            // that every shuffle has the whole warp; they store nothing.
            if (KIND == 1) {
#pragma unroll unroll_of(CPT)
                for (int k = 0; k < kb; ++k)
                    add_draw<KIND, cpt, kNf>(acc, nf, __shfl_sync(kAll, v, k), keys.k[k]);
            } else if (KIND == 3) {
#pragma unroll 8
                for (int k = 0; k < kb; ++k)
                    add_draw<KIND, cpt, kNf>(acc, nf, __shfl_sync(kAll, v, k), keys.k[k]);
            } else {
#pragma unroll 2
                for (int k = 0; k < kb; ++k)
                    add_draw<KIND, cpt, kNf>(acc, nf, __shfl_sync(kAll, v, k), keys.k[k]);
            }
        }
    } else {
    if (SRC == 2) {
        // The CTA's loss changes, then each token's mean over its K draws
        // (centring), summed in draw order.
        const int kk = static_cast<int>(K);
        for (int e = tid; e < kTok * kk; e += blockDim.x) {
            const int k = e / kTok, tok = e - k * kTok;
            s_raw[tok][k] = (tb + tok < T) ? r[static_cast<int64_t>(k) * T + tb + tok] : 0.0f;
        }
        __syncthreads();
        // Sums of 8 draws each in draw order (one thread per token and batch),
        // then the batch sums in order: the credit scan's order.
        const int nb = (kk + 7) / 8;
        if (center && kk > 1 && tid < kTok * nb) {
            const int tok = tid / nb, q = tid - tok * nb;
            float part = 0.0f;
            for (int k = 8 * q; k < 8 * q + 8 && k < kk; ++k) part += s_raw[tok][k];
            s_part[tok][q] = part;
        }
        __syncthreads();
        if (tid < kTok) {
            float mean = 0.0f;
            if (center && kk > 1) {
                for (int q = 0; q < nb; ++q) mean += s_part[tid][q];
                mean /= static_cast<float>(kk);
            }
            s_mean[tid] = mean;
        }
        __syncthreads();
    }
    auto reward = [&](int tok, int64_t i) {
        if (SRC == 2) return -(s_raw[SRC == 2 ? tok : 0][i] - s_mean[tok]);
        const int64_t tt = tb + tok;
        float v = r[tt * K + i];
        if (SRC == 1) v = fmaf(P[tt], carry[(tt / kScanChunk) * K + i], v);
        return v;
    };
    const int64_t Kb = ANTI ? K / 2 : K;
    const int64_t b_begin = ANTI ? draw_begin / 2 : draw_begin;
    for (int64_t g0 = 0; g0 < Kb; g0 += kGroup) {
        const int gn = static_cast<int>(Kb - g0 < kGroup ? Kb - g0 : kGroup);
        if (tid < gn) {
            const int64_t bi = b_begin + g0 + tid;
            s_key[tid] = make_uint2(fold16(draw_key(skey, bi, 0)),
                                    KIND == 1 ? fold16(draw_key(skey, bi, 1)) : 0u);
        }
        for (int e = tid; e < kTok * gn; e += blockDim.x) {
            const int tok = e / gn, k = e - tok * gn;
            float v = 0.0f;
            if (tb + tok < T) {
                if (ANTI) {
                    const int64_t i = 2 * (g0 + k);
                    v = (reward(tok, i) - reward(tok, i + 1)) * coef;
                } else {
                    v = reward(tok, g0 + k) * coef;
                }
            }
            s_r[tok][k] = v;
        }
        __syncthreads();
        if (active) {
            if (KIND == 1) {
#pragma unroll unroll_of(CPT)
                for (int k = 0; k < gn; ++k) add_draw<KIND, cpt, kNf>(acc, nf, s_r[warp][k], s_key[k]);
            } else if (KIND == 3) {
#pragma unroll 8  // 2: 813 us, 4: 774 us, 8: 766 us on the 4096^2 layer, 64 draws
                for (int k = 0; k < gn; ++k) add_draw<KIND, cpt, kNf>(acc, nf, s_r[warp][k], s_key[k]);
            } else {
#pragma unroll 2
                for (int k = 0; k < gn; ++k) add_draw<KIND, cpt, kNf>(acc, nf, s_r[warp][k], s_key[k]);
            }
        }
        __syncthreads();
    }
    }
    if (active) {
        const bool vec = vec_ok;  // 16-byte aligned rows (host-checked)
#pragma unroll
        for (int q = 0; q < cpt / 8; ++q) {
            const int64_t cq = c0 + 8 * q;
            if (cq < d_out) store8<OutT>(g, t, d_out, cq, acc + 8 * q, vec && cq + 8 <= d_out);
        }
    }
}

template <int KIND, int CPT, int SRC>
cudaError_t launch_kind(const float* r, const ScanBuffers& b, int64_t K, int64_t T, int64_t d_out,
                        uint32_t skey, int64_t draw_begin, float coef, bool anti, int center,
                        void* g, int g_bf16, cudaStream_t s) {
    constexpr int ch = 32 * CPT;  // channels per CTA
    DrawKeys keys = {};
    if (SRC == 2) {  // K <= 32 (checked by the caller)
        const int64_t kb = anti ? K / 2 : K;
        const int64_t b0 = anti ? draw_begin / 2 : draw_begin;
        for (int64_t i = 0; i < kb; ++i)
            keys.k[i] = make_uint2(fold16(draw_key(skey, b0 + i, 0)),
                                   KIND == 1 ? fold16(draw_key(skey, b0 + i, 1)) : 0u);
    }
    dim3 grid(static_cast<unsigned>((T + kTok - 1) / kTok),
              static_cast<unsigned>((d_out + ch - 1) / ch));
    const bool vec_ok = (d_out % 8 == 0) && (reinterpret_cast<uintptr_t>(g) % 16 == 0);
    ProfScope ps(kStageWeight, s);
    auto go = [&](auto kernel, auto* out) {
        return launch_pdl_shared(kernel, grid, dim3(256), 0, s, r, b.P, b.carry, K, T, d_out,
                                 skey, draw_begin, coef, out, vec_ok, center, keys);
    };
    auto* gb = static_cast<__nv_bfloat16*>(g);
    auto* gf = static_cast<float*>(g);
    if (g_bf16)
        return anti ? go(k_weight<KIND, CPT, SRC, true, __nv_bfloat16>, gb)
                    : go(k_weight<KIND, CPT, SRC, false, __nv_bfloat16>, gb);
    return anti ? go(k_weight<KIND, CPT, SRC, true, float>, gf)
                : go(k_weight<KIND, CPT, SRC, false, float>, gf);
}

template <int KIND, int CPT>
cudaError_t launch_src(const float* delta, const ScanBuffers& b, bool fix, int64_t K, int64_t T,
                       int64_t d_out, uint32_t skey, int64_t draw_begin, float coef, bool anti,
                       int center, void* g, int g_bf16, cudaStream_t s) {
    if (delta) {
        if (K > 32) return cudaErrorInvalidValue;  // one loss change per lane
        return launch_kind<KIND, CPT, 2>(delta, b, K, T, d_out, skey, draw_begin, coef, anti,
                                         center, g, g_bf16, s);
    }
    if (fix)
        return launch_kind<KIND, CPT, 1>(b.r, b, K, T, d_out, skey, draw_begin, coef, anti, 0, g,
                                         g_bf16, s);
    return launch_kind<KIND, CPT, 0>(b.r, b, K, T, d_out, skey, draw_begin, coef, anti, 0, g,
                                     g_bf16, s);
}

}  // namespace

cudaError_t launch_weight(const ScanBuffers& b, bool fix, int64_t K, int64_t T, int64_t d_out,
                          uint64_t seed, int kind, int64_t draw_begin, float coef, bool anti,
                          void* g, int g_bf16, cudaStream_t s, const float* delta, bool center) {
    if (T == 0 || d_out == 0) return cudaSuccess;
    const uint32_t skey = seed_key(seed);
    const int c = center ? 1 : 0;
    // Wide Gaussian lanes where the CTAs of 1024 channels are whole: the
    // per-draw shared-memory or shuffle reads and the per-thread setup and
    // store spread over twice the pairs. Measured on 8 to 64 noise draws
    // (weighting: up-projection K 8 139 -> 135.5 us, K 16 257 -> 250 us,
    // K 64 957 -> 942 us; 4096^2 K 64 3775 -> 3739 us; qkv K 16 373 -> 368 us);
    // longer draw loops keep the narrow lanes.
    const int64_t noise_draws = anti ? K / 2 : K;
    if (kind == 1 && d_out % (32 * kCptWide) == 0 && noise_draws <= 64)
        return launch_src<1, kCptWide>(delta, b, fix, K, T, d_out, skey, draw_begin, coef, anti, c,
                                       g, g_bf16, s);
    if (kind == 1)
        return launch_src<1, kCpt>(delta, b, fix, K, T, d_out, skey, draw_begin, coef, anti, c, g,
                                   g_bf16, s);
    if (kind == 3)
        return launch_src<3, kCptWide>(delta, b, fix, K, T, d_out, skey, draw_begin, coef, anti, c,
                                       g, g_bf16, s);
    return launch_src<0, kCpt>(delta, b, fix, K, T, d_out, skey, draw_begin, coef, anti, c, g,
                               g_bf16, s);
}

}  // namespace dust
