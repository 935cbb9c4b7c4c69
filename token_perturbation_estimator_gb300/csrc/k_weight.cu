// Reward weighting with in-register noise regeneration:
//   g[t][c] = -(1/(K sigma)) sum_i r_t^(i) a_t^(i)[c]
// ("Dust: every token is a member of the population", section "Perturb the
// activations, not the weights", the g_t equation). The jitter a is rebuilt
// from the hash for every (draw, token, channel) and used once; nothing of it
// is stored.
//
// Mapping: one warp per token, 8 channels per lane (4 Box-Muller pairs or 8
// signs), 8 tokens x 256 channels per CTA. The per-draw keys and the
// per-token rewards (already multiplied by -1/(K sigma) and, for antithetic
// draws, by the pair sign) are staged in shared memory 64 draws at a time and
// read as warp-wide broadcasts. The per-channel counters are pre-folded once
// per thread, so each element-draw costs the hash tail plus one FMA
// (Rademacher: the sign bit is xor-ed into the reward's sign bit).
#include "internal.cuh"
#include "noise.cuh"

namespace dust {

namespace {

constexpr int kTok = 8;     // tokens per CTA (one per warp)
constexpr int kCh = 256;    // channels per CTA (8 per lane)
constexpr int kGroup = 64;  // draws staged per pass

template <typename OutT>
__device__ __forceinline__ void store8(OutT* g, int64_t row, int64_t d_out, int64_t c0,
                                       const float (&acc)[8], bool vec);

template <>
__device__ __forceinline__ void store8<float>(float* g, int64_t row, int64_t d_out, int64_t c0,
                                              const float (&acc)[8], bool vec) {
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
                                                      const float (&acc)[8], bool vec) {
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

template <int KIND, bool FIX, typename OutT>
__global__ void __launch_bounds__(256) k_weight(const float* __restrict__ r,
                                                const float* __restrict__ P,
                                                const float* __restrict__ carry, int64_t K,
                                                int64_t T, int64_t d_out, uint32_t skey,
                                                int64_t draw_begin, float coef, bool anti,
                                                OutT* __restrict__ g) {
    __shared__ uint32_t s_k0[kGroup];
    __shared__ uint32_t s_k1[kGroup];
    __shared__ float s_r[kTok][kGroup];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t tb = static_cast<int64_t>(blockIdx.x) * kTok;
    const int64_t t = tb + warp;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kCh + lane * 8;
    const bool active = (t < T) && (c0 < d_out);

    // Pre-folded counters: pairs for the Gaussian, single channels for signs.
    uint32_t nf[8];
    const uint32_t base = static_cast<uint32_t>(t * d_out + c0);
#pragma unroll
    for (int j = 0; j < 8; ++j) nf[j] = fold16(base + (KIND == 1 ? 2u * (j & 3) : j));

    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;

    for (int64_t g0 = 0; g0 < K; g0 += kGroup) {
        const int gn = static_cast<int>(K - g0 < kGroup ? K - g0 : kGroup);
        if (tid < gn) {
            const int64_t i = draw_begin + g0 + tid;
            const int64_t bi = base_draw(i, anti);
            s_k0[tid] = fold16(draw_key(skey, bi, 0));
            if (KIND == 1) s_k1[tid] = fold16(draw_key(skey, bi, 1));
        }
        for (int e = tid; e < kTok * gn; e += blockDim.x) {
            const int tok = e / gn, k = e - tok * gn;
            const int64_t tt = tb + tok;
            float v = 0.0f;
            if (tt < T) {
                v = r[tt * K + g0 + k];
                if (FIX) v = fmaf(P[tt], carry[(tt / kScanChunk) * K + g0 + k], v);
                v *= coef;
                if (anti && ((draw_begin + g0 + k) & 1)) v = -v;
            }
            s_r[tok][k] = v;
        }
        __syncthreads();
        if (active) {
            if (KIND == 1) {
#pragma unroll 2
                for (int k = 0; k < gn; ++k) {
                    const float rr = s_r[warp][k];
                    const uint32_t k0 = s_k0[k], k1 = s_k1[k];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const float f0 = unit_ff(k0, nf[p]);
                        const float f1 = unit_ff(k1, nf[p]);
                        const float tr = rr * neg_radius(f0);
                        float sn, cs;
                        __sincosf(6.28318530717958648f * (f1 - 1.5f), &sn, &cs);
                        acc[2 * p] = fmaf(tr, cs, acc[2 * p]);
                        acc[2 * p + 1] = fmaf(tr, sn, acc[2 * p + 1]);
                    }
                }
            } else {
#pragma unroll 2
                for (int k = 0; k < gn; ++k) {
                    const uint32_t rb = __float_as_uint(s_r[warp][k]);
                    const uint32_t k0 = s_k0[k];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[j] += __uint_as_float(rb ^ sign_ff(k0, nf[j]));
                }
            }
        }
        __syncthreads();
    }
    if (active) {
        const bool vec = ((d_out & 7) == 0) && (c0 + 8 <= d_out);
        store8<OutT>(g, t, d_out, c0, acc, vec);
    }
}

template <int KIND, bool FIX>
cudaError_t launch_kind(const ScanBuffers& b, int64_t K, int64_t T, int64_t d_out, uint32_t skey,
                        int64_t draw_begin, float coef, bool anti, void* g, int g_bf16,
                        cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((T + kTok - 1) / kTok),
              static_cast<unsigned>((d_out + kCh - 1) / kCh));
    ProfScope ps(kStageWeight, s);
    if (g_bf16)
        k_weight<KIND, FIX, __nv_bfloat16><<<grid, 256, 0, s>>>(
            b.r, b.P, b.carry, K, T, d_out, skey, draw_begin, coef, anti,
            static_cast<__nv_bfloat16*>(g));
    else
        k_weight<KIND, FIX, float><<<grid, 256, 0, s>>>(b.r, b.P, b.carry, K, T, d_out, skey,
                                                        draw_begin, coef, anti,
                                                        static_cast<float*>(g));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_weight(const ScanBuffers& b, bool fix, int64_t K, int64_t T, int64_t d_out,
                          uint64_t seed, int kind, int64_t draw_begin, float coef, bool anti,
                          void* g, int g_bf16, cudaStream_t s) {
    if (T == 0 || d_out == 0) return cudaSuccess;
    const uint32_t skey = seed_key(seed);
    if (kind == 1)
        return fix ? launch_kind<1, true>(b, K, T, d_out, skey, draw_begin, coef, anti, g, g_bf16, s)
                   : launch_kind<1, false>(b, K, T, d_out, skey, draw_begin, coef, anti, g, g_bf16, s);
    return fix ? launch_kind<0, true>(b, K, T, d_out, skey, draw_begin, coef, anti, g, g_bf16, s)
               : launch_kind<0, false>(b, K, T, d_out, skey, draw_begin, coef, anti, g, g_bf16, s);
}

}  // namespace dust
