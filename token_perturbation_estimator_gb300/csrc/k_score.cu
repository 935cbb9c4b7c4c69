// Local scores of blocks whose output does not reach the loss ("Dust: every
// token is a member of the population", section "What the released code
// actually does", step 4): for every draw k and token s,
//     delta[k][s] = <g_s, delta_o[k][s]>,
// the first-order loss change whose reduction is the page's score
// c_s = -<g_s, delta_o_s>; the credit scan then sums the later tokens' scores
// decayed by gamma (keys, values, gates) or keeps the token's own (queries).
//
// Bound by HBM: each (k, s) row of delta_o is read once and used once. A warp
// takes one token's g row and several draws' rows, its 16-byte vector loads
// issued before the products; each row's partial sums are reduced by warp
// shuffles in a fixed order (deterministic).
#include "internal.cuh"

namespace dust {

namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Eight consecutive elements, kept as loaded (one 16-byte vector of bf16 or
// two of f32) and widened only inside the products, so that the registers
// stay few and many warps stay resident.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        u = __ldg(reinterpret_cast<const uint4*>(p));
    }
    __device__ __forceinline__ float at(int k) const {
        const uint32_t w = (k < 2) ? u.x : (k < 4) ? u.y : (k < 6) ? u.z : u.w;
        return __uint_as_float((k & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = __ldg(reinterpret_cast<const float4*>(p));
        b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ float at(int k) const {
        const float4& h = (k < 4) ? a : b;
        const int m = k & 3;
        return m == 0 ? h.x : m == 1 ? h.y : m == 2 ? h.z : h.w;
    }
};

// Vector path: a warp takes one token and kDraws draws at a time; each lane
// holds kVec 8-element vectors of the token's g row and of each draw's
// delta_o row per pass (d <= 512 in one pass), all loaded before the first
// product, so that one warp keeps kDraws rows of HBM reads in flight.
constexpr int kVec = 2;

template <typename TO> constexpr int draws_per_warp() { return sizeof(TO) == 2 ? 4 : 2; }

#ifndef DUST_SCORE_MINB
#define DUST_SCORE_MINB 3  // resident CTAs per SM the registers must allow
#endif

template <typename TG, typename TO>
__global__ void __launch_bounds__(256, DUST_SCORE_MINB) k_local_score(const TG* __restrict__ g,
                                                     const TO* __restrict__ dO, int64_t K,
                                                     int64_t T, int64_t d, float* __restrict__ out,
                                                     int vec) {
    pdl_wait();
    pdl_trigger();
    constexpr int kD = draws_per_warp<TO>();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t n_kb = (K + kD - 1) / kD;
    for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         w < T * n_kb; w += warps) {
        const int64_t t = w / n_kb;
        const int64_t k0 = (w - t * n_kb) * kD;
        const TG* gr = g + t * d;
        float acc[kD];
#pragma unroll
        for (int r = 0; r < kD; ++r) acc[r] = 0.0f;
        if (vec) {  // d % 8 == 0 and both bases 16-byte aligned (host-checked)
            for (int64_t j0 = 0; j0 < d; j0 += 256 * kVec) {
                Raw8<TG> a[kVec];
                Raw8<TO> b[kD][kVec];
#pragma unroll
                for (int v = 0; v < kVec; ++v) {
                    const int64_t j = j0 + 256 * v + 8 * lane;
                    if (j >= d) continue;
                    a[v].load(gr + j);
#pragma unroll
                    for (int r = 0; r < kD; ++r)
                        if (k0 + r < K) b[r][v].load(dO + ((k0 + r) * T + t) * d + j);
                }
#pragma unroll
                for (int v = 0; v < kVec; ++v) {
                    if (j0 + 256 * v + 8 * lane >= d) continue;
#pragma unroll
                    for (int r = 0; r < kD; ++r) {
                        if (k0 + r >= K) continue;
#pragma unroll
                        for (int u = 0; u < 8; ++u) acc[r] = fmaf(a[v].at(u), b[r][v].at(u), acc[r]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < kD; ++r) {
                if (k0 + r >= K) continue;
                const TO* orow = dO + ((k0 + r) * T + t) * d;
                for (int64_t j = lane; j < d; j += 32)
                    acc[r] = fmaf(to_f(gr[j]), to_f(orow[j]), acc[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < kD; ++r) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
            if (lane == 0 && k0 + r < K) out[(k0 + r) * T + t] = acc[r];
        }
    }
}

template <typename TG, typename TO>
cudaError_t launch_typed(const void* g, const void* dO, int64_t K, int64_t T, int64_t d,
                         float* out, cudaStream_t s) {
    const int64_t warps = T * ((K + draws_per_warp<TO>() - 1) / draws_per_warp<TO>());
    int64_t blocks = (warps + 7) / 8;
    if (blocks > 152 * 16) blocks = 152 * 16;
    const int vec = (d % 8 == 0) && (reinterpret_cast<uintptr_t>(g) % 16 == 0) &&
                    (reinterpret_cast<uintptr_t>(dO) % 16 == 0);
    ProfScope ps(kStageScore, s);
    return launch_pdl(k_local_score<TG, TO>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                      s, static_cast<const TG*>(g), static_cast<const TO*>(dO), K, T, d, out,
                      vec);
}

}  // namespace

cudaError_t launch_local_score(const void* g, int g_bf16, const void* dO, int o_bf16, int64_t K,
                               int64_t T, int64_t d, float* out, cudaStream_t s) {
    if (K * T == 0) return cudaSuccess;
    if (g_bf16 && o_bf16) return launch_typed<__nv_bfloat16, __nv_bfloat16>(g, dO, K, T, d, out, s);
    if (g_bf16) return launch_typed<__nv_bfloat16, float>(g, dO, K, T, d, out, s);
    if (o_bf16) return launch_typed<float, __nv_bfloat16>(g, dO, K, T, d, out, s);
    return launch_typed<float, float>(g, dO, K, T, d, out, s);
}

}  // namespace dust
