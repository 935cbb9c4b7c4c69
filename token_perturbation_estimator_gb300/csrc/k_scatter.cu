// Embedding reassembly ("Dust: every token is a member of the population",
// "What the released code actually does", step 7: "a scatter-add for an
// embedding"): gE[v][c] = scale * sum_{t : ids[t] = v} g[t][c].
//
// Deterministic without sorting: the sums are accumulated in 64-bit fixed
// point, where addition is associative, so the atomics' arrival order cannot
// change a bit of the result. The fixed-point step 2^-s is chosen per call
// from the data: with M = max |g| and C = the largest number of tokens
// sharing one id, every term is below 2^61 / C in units of 2^-s, so no sum
// can overflow, and each term is rounded once, to within 2^-s / 2, far below
// the fp32 rounding of the output.
//
//   k_scatter_stats    per-id token counts (with the largest), max |g|, and a
//                      flag for ids outside [0, V);
//   k_scatter_add      g -> round(g 2^s) added into acc[id][c];
//   k_scatter_finish   gE = scale * acc 2^-s (+ gE when accumulating).
#include "internal.cuh"

namespace dust {

namespace {

struct ScatterHeader {
    unsigned int max_abs_bits;  // bit pattern of max |g| (non-negative floats order as ints)
    int max_count;
    unsigned int bad_ids;
    int pad;
};

template <typename TG>
__device__ __forceinline__ float load_g(const TG* g, int64_t i);
template <>
__device__ __forceinline__ float load_g<float>(const float* g, int64_t i) { return g[i]; }
template <>
__device__ __forceinline__ float load_g<__nv_bfloat16>(const __nv_bfloat16* g, int64_t i) {
    return __bfloat162float(g[i]);
}

// One warp per token: its id's count and the row's max |g|.
template <typename TG>
__global__ void __launch_bounds__(256) k_scatter_stats(const TG* __restrict__ g,
                                                       const int32_t* __restrict__ ids, int64_t T,
                                                       int64_t d, int64_t V, int* __restrict__ counts,
                                                       ScatterHeader* __restrict__ hdr,
                                                       unsigned int* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T;
         t += warps) {
        const int64_t v = ids[t];
        if (v < 0 || v >= V) {
            if (lane == 0) {
                atomicOr(&hdr->bad_ids, 1u);
                atomicExch(status, 1u /* DUST_ERR_INVALID_ARG */);
            }
            continue;
        }
        float m = 0.0f;
        for (int64_t c = lane; c < d; c += 32) m = fmaxf(m, fabsf(load_g(g, t * d + c)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) {
            const int n = atomicAdd(&counts[v], 1) + 1;
            atomicMax(&hdr->max_count, n);
            atomicMax(&hdr->max_abs_bits, __float_as_uint(m));
        }
    }
}

// The fixed-point exponent s: M C 2^s < 2^61 (0 when g is all zero).
__device__ __forceinline__ int scatter_shift(const ScatterHeader* hdr) {
    const double m = static_cast<double>(__uint_as_float(hdr->max_abs_bits));
    const int c = hdr->max_count;
    if (!(m > 0.0) || c <= 0) return 0;
    int e = 0;
    frexp(m * static_cast<double>(c), &e);  // m c < 2^e
    return 61 - e;
}

// One warp per token: its row's fixed-point values added into its id's row.
template <typename TG>
__global__ void __launch_bounds__(256) k_scatter_add(const TG* __restrict__ g,
                                                     const int32_t* __restrict__ ids, int64_t T,
                                                     int64_t d, int64_t V,
                                                     const ScatterHeader* __restrict__ hdr,
                                                     unsigned long long* __restrict__ acc) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const double step = ldexp(1.0, scatter_shift(hdr));
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T;
         t += warps) {
        const int64_t v = ids[t];
        if (v < 0 || v >= V) continue;
        for (int64_t c = lane; c < d; c += 32) {
            const float x = load_g(g, t * d + c);
            if (x == 0.0f) continue;
            const long long f = __double2ll_rn(static_cast<double>(x) * step);
            atomicAdd(&acc[v * d + c], static_cast<unsigned long long>(f));
        }
    }
}

__global__ void __launch_bounds__(256) k_scatter_finish(const unsigned long long* __restrict__ acc,
                                                        int64_t n, const ScatterHeader* __restrict__ hdr,
                                                        float scale, int accumulate,
                                                        float* __restrict__ gE) {
    pdl_wait();
    pdl_trigger();
    const double unit = ldexp(1.0, -scatter_shift(hdr)) * static_cast<double>(scale);
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float v = static_cast<float>(static_cast<double>(static_cast<long long>(acc[q])) * unit);
        gE[q] = accumulate ? gE[q] + v : v;
    }
}

size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

unsigned grid_for(int64_t n, int64_t per_block, int64_t cap) {
    int64_t b = (n + per_block - 1) / per_block;
    if (b > cap) b = cap;
    return static_cast<unsigned>(b < 1 ? 1 : b);
}

}  // namespace

size_t scatter_workspace_bytes(int64_t V, int64_t d) {
    return a256(sizeof(ScatterHeader)) + a256(sizeof(int) * static_cast<size_t>(V)) +
           a256(sizeof(unsigned long long) * static_cast<size_t>(V * d));
}

cudaError_t launch_scatter_gE(const void* g, int g_bf16, const int32_t* ids, int64_t T,
                              int64_t d, int64_t V, float scale, bool accumulate, float* gE,
                              void* workspace, cudaStream_t s) {
    char* w = static_cast<char*>(workspace);
    auto* hdr = reinterpret_cast<ScatterHeader*>(w);
    auto* counts = reinterpret_cast<int*>(w + a256(sizeof(ScatterHeader)));
    auto* acc = reinterpret_cast<unsigned long long*>(w + a256(sizeof(ScatterHeader)) +
                                                      a256(sizeof(int) * static_cast<size_t>(V)));
    unsigned int* st = status_word();
    if (!st) return cudaErrorUnknown;
    cudaError_t e = cudaMemsetAsync(workspace, 0, scatter_workspace_bytes(V, d), s);
    if (e != cudaSuccess) return e;
    {
        ProfScope ps(kStageScatter, s);
        const unsigned gs = grid_for(T, 8, 152 * 16);
        e = g_bf16 ? launch_pdl(k_scatter_stats<__nv_bfloat16>, dim3(gs), dim3(256), 0, s,
                                static_cast<const __nv_bfloat16*>(g), ids, T, d, V, counts, hdr, st)
                   : launch_pdl(k_scatter_stats<float>, dim3(gs), dim3(256), 0, s,
                                static_cast<const float*>(g), ids, T, d, V, counts, hdr, st);
        if (e != cudaSuccess) return e;
        const unsigned ga = grid_for(T, 8, 152 * 16);
        e = g_bf16 ? launch_pdl(k_scatter_add<__nv_bfloat16>, dim3(ga), dim3(256), 0, s,
                                static_cast<const __nv_bfloat16*>(g), ids, T, d, V,
                                static_cast<const ScatterHeader*>(hdr), acc)
                   : launch_pdl(k_scatter_add<float>, dim3(ga), dim3(256), 0, s,
                                static_cast<const float*>(g), ids, T, d, V,
                                static_cast<const ScatterHeader*>(hdr), acc);
        if (e != cudaSuccess) return e;
        const unsigned gf = grid_for(V * d, 256, 152 * 32);
        e = launch_pdl(k_scatter_finish, dim3(gf), dim3(256), 0, s,
                       static_cast<const unsigned long long*>(acc), V * d,
                       static_cast<const ScatterHeader*>(hdr), scale, accumulate ? 1 : 0, gE);
    }
    return e;
}

}  // namespace dust
