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
//   k_scatter_starts   each id's first slot in the token list grouped by id;
//   k_scatter_place    every token into a slot of its id's run;
//   k_scatter_runs     per warp, the runs of a 32-slot range summed in
//                      registers (round(g 2^s) per term) and added into
//                      acc[id][c] once per run;
//   k_scatter_finish   gE = scale * acc 2^-s (+ gE when accumulating).
#include "internal.cuh"

namespace dust {

namespace {

struct ScatterHeader {
    unsigned int max_abs_bits;  // bit pattern of max |g| (non-negative floats order as ints)
    int max_count;
    unsigned int bad_ids;  // tokens with an id outside [0, V)
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

// x 2^s rounded to the nearest integer (ties up), from the float's bits with
// integer operations only (no FP64: this GPU's FP64 rate is a small fraction
// of its integer rate). Callers guarantee |x| 2^s < 2^61.
__device__ __forceinline__ long long to_fixed(float x, int s) {
    const uint32_t b = __float_as_uint(x);
    const uint32_t ex = (b >> 23) & 0xFFu;
    const long long m = (ex ? (b & 0x7FFFFFu) | 0x800000u : (b & 0x7FFFFFu));
    const int k = (ex ? static_cast<int>(ex) : 1) - 150 + s;  // x 2^s = m 2^k
    long long r;
    if (k >= 0) {
        r = m << k;
    } else if (k > -40) {
        r = (m + (1ll << (-k - 1))) >> (-k);
    } else {
        r = 0;
    }
    return (b >> 31) ? -r : r;
}

// A 64-bit integer times u in fp32 (hi * 2^32 + lo, one fused multiply-add).
__device__ __forceinline__ float from_fixed(long long q, float u) {
    const float hi = static_cast<float>(static_cast<int>(q >> 32));
    const float lo = static_cast<float>(static_cast<uint32_t>(q & 0xFFFFFFFFll));
    return fmaf(hi, 4294967296.0f * u, lo * u);
}

// Block-wide max of v (all threads of the block call it).
__device__ __forceinline__ float block_max(float v, float* s_red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    v = (threadIdx.x < (blockDim.x >> 5)) ? s_red[threadIdx.x] : 0.0f;
    if (warp == 0)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;  // valid in thread 0
}

// Per-id token counts (thread per token, the largest count reduced per
// block), tokens with an id outside [0, V) counted, and max |g| over all
// elements (16-byte loads when aligned, reduced per block): one atomic per
// block for each maximum, so no address is contended.
template <typename TG>
__global__ void __launch_bounds__(256) k_scatter_stats(const TG* __restrict__ g,
                                                       const int32_t* __restrict__ ids, int64_t T,
                                                       int64_t d, int64_t V, int* __restrict__ counts,
                                                       ScatterHeader* __restrict__ hdr,
                                                       unsigned int* __restrict__ status, int vec) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_red[8];
    const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t gn = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int cmax = 0;
    for (int64_t t = gt; t < T; t += gn) {
        const int64_t v = ids[t];
        if (v < 0 || v >= V) {
            atomicAdd(&hdr->bad_ids, 1u);
            atomicExch(status, 1u /* DUST_ERR_INVALID_ARG */);
            continue;
        }
        const int n = atomicAdd(&counts[v], 1) + 1;
        cmax = n > cmax ? n : cmax;
    }
    float m = 0.0f;
    const int64_t n = T * d;
    if (vec) {  // 16-byte aligned base and n % (16 / sizeof(TG)) == 0 (host-checked)
        constexpr int kPer = 16 / sizeof(TG);
        const uint4* p = reinterpret_cast<const uint4*>(g);
        for (int64_t q = gt; q < n / kPer; q += gn) {
            const uint4 u = __ldg(p + q);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (sizeof(TG) == 2) {
                    m = fmaxf(m, fabsf(__uint_as_float(w[k] << 16)));
                    m = fmaxf(m, fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
                } else {
                    m = fmaxf(m, fabsf(__uint_as_float(w[k])));
                }
            }
        }
    } else {
        for (int64_t q = gt; q < n; q += gn) m = fmaxf(m, fabsf(load_g(g, q)));
    }
    // the ids of bad tokens are skipped later; their rows may still raise m,
    // which only makes the fixed-point step finer than needed
    const float bm = block_max(m, s_red);
    if (threadIdx.x == 0) atomicMax(&hdr->max_abs_bits, __float_as_uint(bm));
    cmax = __reduce_max_sync(0xffffffffu, cmax);
    if ((threadIdx.x & 31) == 0 && cmax > 0) atomicMax(&hdr->max_count, cmax);
}

// The fixed-point exponent s: M C 2^s < 2^61 (0 when g is all zero).
__device__ __forceinline__ int scatter_shift(const ScatterHeader* hdr) {
    const double m = static_cast<double>(__uint_as_float(hdr->max_abs_bits));
    const int c = hdr->max_count;
    if (!(m > 0.0) || c <= 0) return 0;
    int e = 0;
    frexp(m * static_cast<double>(c), &e);  // m c < 2^e
    // at most 2^100 (steps below 2^-100 would only resolve values that far
    // below any fp32 output; keeps 2^-s normal in fp32)
    return 61 - e < 100 ? 61 - e : 100;
}

// Exclusive scan of the per-id counts into the first slot of each id's run
// in the grouped token list (one CTA: each thread scans a contiguous block of
// ids, then the block totals are scanned).
__global__ void __launch_bounds__(1024) k_scatter_starts(const int* __restrict__ counts,
                                                         int64_t V, int* __restrict__ cursor) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_tot[1024];
    const int tid = threadIdx.x;
    const int64_t per = (V + 1023) / 1024;
    const int64_t lo = tid * per, hi = (lo + per < V) ? lo + per : V;
    int sum = 0;
    for (int64_t v = lo; v < hi; ++v) sum += counts[v];
    s_tot[tid] = sum;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan of the block totals
        const int x = tid >= off ? s_tot[tid - off] : 0;
        __syncthreads();
        s_tot[tid] += x;
        __syncthreads();
    }
    int run = tid > 0 ? s_tot[tid - 1] : 0;
    for (int64_t v = lo; v < hi; ++v) {
        cursor[v] = run;
        run += counts[v];
    }
}

// Tokens grouped by id: token t goes to a free slot of its id's run.
__global__ void __launch_bounds__(256) k_scatter_place(const int32_t* __restrict__ ids, int64_t T,
                                                       int64_t V, int* __restrict__ cursor,
                                                       int* __restrict__ perm) {
    pdl_wait();
    pdl_trigger();
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t v = ids[t];
        if (v < 0 || v >= V) continue;
        perm[atomicAdd(&cursor[v], 1)] = static_cast<int>(t);
    }
}

// One warp per kRange consecutive slots of the grouped list and 64 columns
// (2 per lane): the rows of a run of one id are summed in registers in
// fixed point, and each run that the warp sees is added once into acc (an
// id whose run spans several warps' ranges gets one addition per warp).
constexpr int kRange = 32;

template <typename TG>
__global__ void __launch_bounds__(256) k_scatter_runs(const TG* __restrict__ g,
                                                      const int32_t* __restrict__ ids,
                                                      const int* __restrict__ perm, int64_t T,
                                                      int64_t d,
                                                      const ScatterHeader* __restrict__ hdr,
                                                      unsigned long long* __restrict__ acc) {
    pdl_wait();
    pdl_trigger();
    constexpr int kAhead = 8;  // rows whose loads are issued together
    constexpr int kCols = 2;   // columns per lane
    const int lane = threadIdx.x & 31;
    const int sh = scatter_shift(hdr);
    const int64_t n = T - static_cast<int64_t>(hdr->bad_ids);
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t passes = (d + 32 * kCols - 1) / (32 * kCols);
    for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         w < ((n + kRange - 1) / kRange) * passes; w += warps) {
        const int64_t r0 = (w / passes) * kRange;
        const int64_t c0 = (w % passes) * (32 * kCols);
        const int len = static_cast<int>((r0 + kRange < n) ? kRange : n - r0);
        // the range's token indices and ids, one per lane
        int t_l = 0, v_l = -1;
        if (lane < len) {
            t_l = perm[r0 + lane];
            v_l = ids[t_l];
        }
        long long sum[kCols];
#pragma unroll
        for (int u = 0; u < kCols; ++u) sum[u] = 0;
        int cur = -1;
        for (int p0 = 0; p0 < len; p0 += kAhead) {
            float x[kAhead][kCols];
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int64_t t = __shfl_sync(0xffffffffu, t_l, (p0 + a) & 31);
#pragma unroll
                for (int u = 0; u < kCols; ++u) {
                    const int64_t c = c0 + 32 * u + lane;
                    x[a][u] = (p0 + a < len && c < d) ? load_g(g, t * d + c) : 0.0f;
                }
            }
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                const int v = __shfl_sync(0xffffffffu, v_l, (p0 + a) & 31);
                if (p0 + a >= len) break;
                if (v != cur) {
                    if (cur >= 0) {
#pragma unroll
                        for (int u = 0; u < kCols; ++u) {
                            const int64_t c = c0 + 32 * u + lane;
                            if (c < d && sum[u] != 0)
                                atomicAdd(&acc[static_cast<int64_t>(cur) * d + c],
                                          static_cast<unsigned long long>(sum[u]));
                            sum[u] = 0;
                        }
                    }
                    cur = v;
                }
#pragma unroll
                for (int u = 0; u < kCols; ++u) sum[u] += to_fixed(x[a][u], sh);
            }
        }
        if (cur >= 0) {
#pragma unroll
            for (int u = 0; u < kCols; ++u) {
                const int64_t c = c0 + 32 * u + lane;
                if (c < d && sum[u] != 0)
                    atomicAdd(&acc[static_cast<int64_t>(cur) * d + c],
                              static_cast<unsigned long long>(sum[u]));
            }
        }
    }
}

__global__ void __launch_bounds__(256) k_scatter_finish(const unsigned long long* __restrict__ acc,
                                                        int64_t n, const ScatterHeader* __restrict__ hdr,
                                                        float scale, int accumulate,
                                                        float* __restrict__ gE) {
    pdl_wait();
    pdl_trigger();
    const float unit = ldexpf(scale, -scatter_shift(hdr));
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float v = from_fixed(static_cast<long long>(acc[q]), unit);
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

// Workspace: header | counts [V] | cursor [V] | perm [T] | acc [V][d].
size_t scatter_workspace_bytes(int64_t T, int64_t V, int64_t d) {
    return a256(sizeof(ScatterHeader)) + 2 * a256(sizeof(int) * static_cast<size_t>(V)) +
           a256(sizeof(int) * static_cast<size_t>(T)) +
           a256(sizeof(unsigned long long) * static_cast<size_t>(V * d));
}

cudaError_t launch_scatter_gE(const void* g, int g_bf16, const int32_t* ids, int64_t T,
                              int64_t d, int64_t V, float scale, bool accumulate, float* gE,
                              void* workspace, cudaStream_t s) {
    char* w = static_cast<char*>(workspace);
    auto* hdr = reinterpret_cast<ScatterHeader*>(w);
    w += a256(sizeof(ScatterHeader));
    auto* counts = reinterpret_cast<int*>(w);
    w += a256(sizeof(int) * static_cast<size_t>(V));
    auto* cursor = reinterpret_cast<int*>(w);
    w += a256(sizeof(int) * static_cast<size_t>(V));
    auto* perm = reinterpret_cast<int*>(w);
    w += a256(sizeof(int) * static_cast<size_t>(T));
    auto* acc = reinterpret_cast<unsigned long long*>(w);
    unsigned int* st = status_word();
    if (!st) return cudaErrorUnknown;
    // header and counts, then the accumulator (cursor and perm are written first)
    cudaError_t e = cudaMemsetAsync(workspace, 0,
                                    a256(sizeof(ScatterHeader)) +
                                        a256(sizeof(int) * static_cast<size_t>(V)), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(acc, 0, sizeof(unsigned long long) * static_cast<size_t>(V * d), s);
    if (e != cudaSuccess) return e;
    const auto* chdr = static_cast<const ScatterHeader*>(hdr);
    {
        ProfScope ps(kStageScatter, s);
        const unsigned gw = grid_for(T * d / 8 + 1, 256, 152 * 8);
        const int per = g_bf16 ? 8 : 4;
        const int vec = (reinterpret_cast<uintptr_t>(g) % 16 == 0) && ((T * d) % per == 0);
        e = g_bf16 ? launch_pdl(k_scatter_stats<__nv_bfloat16>, dim3(gw), dim3(256), 0, s,
                                static_cast<const __nv_bfloat16*>(g), ids, T, d, V, counts, hdr, st,
                                vec)
                   : launch_pdl(k_scatter_stats<float>, dim3(gw), dim3(256), 0, s,
                                static_cast<const float*>(g), ids, T, d, V, counts, hdr, st, vec);
        if (e == cudaSuccess)
            e = launch_pdl(k_scatter_starts, dim3(1), dim3(1024), 0, s,
                           static_cast<const int*>(counts), V, cursor);
        if (e == cudaSuccess)
            e = launch_pdl(k_scatter_place, dim3(grid_for(T, 256, 152 * 8)), dim3(256), 0, s, ids,
                           T, V, cursor, perm);
        if (e != cudaSuccess) return e;
        // one warp per (32-slot range, 64-column pass); the valid count is
        // known on the device only, so the grid covers all T tokens
        const int64_t units = ((T + kRange - 1) / kRange) * ((d + 63) / 64);
        const unsigned gr = grid_for(units, 8, 152 * 16);
        e = g_bf16 ? launch_pdl(k_scatter_runs<__nv_bfloat16>, dim3(gr), dim3(256), 0, s,
                                static_cast<const __nv_bfloat16*>(g), ids,
                                static_cast<const int*>(perm), T, d, chdr, acc)
                   : launch_pdl(k_scatter_runs<float>, dim3(gr), dim3(256), 0, s,
                                static_cast<const float*>(g), ids, static_cast<const int*>(perm),
                                T, d, chdr, acc);
        if (e != cudaSuccess) return e;
        const unsigned gf = grid_for(V * d, 256, 152 * 32);
        e = launch_pdl(k_scatter_finish, dim3(gf), dim3(256), 0, s,
                       static_cast<const unsigned long long*>(acc), V * d, chdr, scale,
                       accumulate ? 1 : 0, gE);
    }
    return e;
}

}  // namespace dust
