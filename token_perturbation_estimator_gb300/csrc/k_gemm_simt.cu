// CUDA-core contraction GW[c][j] = scale * sum_t g[t][c] x[t][j] ("Dust: every
// token is a member of the population", section "Perturb the activations, not
// the weights", the G_W equation), in fp32 FFMA. It serves the fp32 path and
// shapes the tensor-core kernels do not take. Deterministic: the token range
// is cut into fixed slices whose fp32 partials are summed in slice order.
#include "internal.cuh"

namespace dust {

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16;

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename TG, typename TX>
__global__ void __launch_bounds__(256) k_gemm_simt(const TG* __restrict__ g,
                                                   const TX* __restrict__ X, int64_t T,
                                                   int64_t d_in, int64_t d_out, int64_t slice,
                                                   float* __restrict__ out, float scale,
                                                   int mode) {
    pdl_wait();
    pdl_trigger();
    __shared__ float sg[kBK][kBM];
    __shared__ float sx[kBK][kBN];
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int64_t cb = static_cast<int64_t>(blockIdx.y) * kBM;
    const int64_t jb = static_cast<int64_t>(blockIdx.x) * kBN;
    const int64_t s = blockIdx.z;
    const int64_t t_lo = s * slice;
    const int64_t t_hi = (t_lo + slice < T) ? t_lo + slice : T;

    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;

    for (int64_t t0 = t_lo; t0 < t_hi; t0 += kBK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid * 4 + q;
            const int tt = e / kBM, cc = e % kBM;
            const int64_t t = t0 + tt;
            float vg = 0.0f, vx = 0.0f;
            if (t < t_hi) {
                if (cb + cc < d_out) vg = ld(g + t * d_out + cb + cc);
                if (jb + cc < d_in) vx = ld(X + t * d_in + jb + cc);
            }
            sg[tt][cc] = vg;
            sx[tt][cc] = vx;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[q] = sg[k][ty * 4 + q];
                b[q] = sx[k][tx * 4 + q];
            }
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(a[p], b[q], acc[p][q]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int64_t c = cb + ty * 4 + p;
        if (c >= d_out) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t j = jb + tx * 4 + q;
            if (j >= d_in) continue;
            if (mode == 0) {
                out[(s * d_out + c) * d_in + j] = acc[p][q];
            } else if (mode == 1) {
                out[c * d_in + j] = scale * acc[p][q];
            } else {
                out[c * d_in + j] += scale * acc[p][q];
            }
        }
    }
}

// gW[q] = scale * sum_{s<S} partials[s][q] (+ gW[q]), the sum in slice
// order. Vectorised form: each thread sums U float4 outputs per round, with
// the loads of SB slices of all U outputs issued before any sum, so that a
// thread keeps about 8 loads in flight however few slices there are (the
// reduction is bound by L2 latency: with one output per thread a 3-slice
// reduction over 3072 x 1024 outputs ran as 10 waves of one round trip each),
// at 3 CTAs per SM.
template <int U, int SB>
__global__ void __launch_bounds__(256, 3) k_reduce_v4(const float4* __restrict__ p4, int64_t S,
                                                   int64_t n4, float scale, int accumulate,
                                                   float4* __restrict__ g4) {
    pdl_wait();
    pdl_trigger();
    const int64_t threads = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (int64_t base = tid; base < n4; base += U * threads) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t q = base + u * threads;
            v[u] = q < n4 ? p4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int64_t s0 = 1; s0 < S; s0 += SB) {
            float4 w[U][SB];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t q = base + u * threads;
#pragma unroll
                for (int j = 0; j < SB; ++j)
                    if (s0 + j < S && q < n4) w[u][j] = p4[(s0 + j) * n4 + q];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
#pragma unroll
                for (int j = 0; j < SB; ++j) {
                    if (s0 + j >= S) break;
                    v[u].x += w[u][j].x;
                    v[u].y += w[u][j].y;
                    v[u].z += w[u][j].z;
                    v[u].w += w[u][j].w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t q = base + u * threads;
            if (q >= n4) break;
            float4 o = make_float4(scale * v[u].x, scale * v[u].y, scale * v[u].z, scale * v[u].w);
            if (accumulate) {
                const float4 a = g4[q];
                o = make_float4(a.x + o.x, a.y + o.y, a.z + o.z, a.w + o.w);
            }
            g4[q] = o;
        }
    }
}

__global__ void __launch_bounds__(256) k_reduce(const float* __restrict__ part, int64_t S,
                                                int64_t n, float scale, int accumulate,
                                                float* __restrict__ gW) {
    pdl_wait();
    pdl_trigger();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (int64_t q = tid; q < n; q += stride) {
        float v = 0.0f;
        for (int64_t s = 0; s < S; ++s) v += part[s * n + q];
        gW[q] = accumulate ? gW[q] + scale * v : scale * v;
    }
}

int64_t slices_for(int64_t T, int64_t d_in, int64_t d_out) {
    const int64_t tiles = ((d_out + kBM - 1) / kBM) * ((d_in + kBN - 1) / kBN);
    int64_t S = (2 * 152 + tiles - 1) / tiles;
    const int64_t max_s = (T + 63) / 64;
    if (S > max_s) S = max_s;
    if (S > 64) S = 64;
    return S < 1 ? 1 : S;
}

template <typename TG, typename TX>
cudaError_t run(const void* g, const void* X, int64_t T, int64_t d_in, int64_t d_out,
                float scale, bool accumulate, float* gW, float* partials, cudaStream_t s) {
    const int64_t S = slices_for(T, d_in, d_out);
    int64_t slice = (T + S - 1) / S;
    slice = (slice + kBK - 1) / kBK * kBK;
    const int64_t S_used = (T + slice - 1) / slice;
    dim3 grid(static_cast<unsigned>((d_in + kBN - 1) / kBN),
              static_cast<unsigned>((d_out + kBM - 1) / kBM), static_cast<unsigned>(S_used));
    if (S_used == 1) {
        ProfScope ps(kStageGemmSimt, s);
        return launch_pdl(k_gemm_simt<TG, TX>, grid, dim3(256), 0, s,
                          static_cast<const TG*>(g), static_cast<const TX*>(X), T, d_in, d_out,
                          slice, gW, scale, accumulate ? 2 : 1);
    }
    cudaError_t e;
    {
        ProfScope ps(kStageGemmSimt, s);
        e = launch_pdl(k_gemm_simt<TG, TX>, grid, dim3(256), 0, s, static_cast<const TG*>(g),
                       static_cast<const TX*>(X), T, d_in, d_out, slice, partials, scale, 0);
    }
    if (e != cudaSuccess) return e;
    return launch_reduce(partials, S_used, d_out * d_in, scale, accumulate, gW, s);
}

}  // namespace

cudaError_t launch_reduce(const float* partials, int64_t S, int64_t n, float scale,
                          bool accumulate, float* gW, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int vec4 = ((n & 3) == 0) && (reinterpret_cast<uintptr_t>(gW) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(partials) % 16 == 0);
    ProfScope ps(kStageReduce, s);
    if (!vec4) {
        int64_t rg = (n + 255) / 256;
        if (rg > 152 * 16) rg = 152 * 16;
        return launch_pdl_shared(k_reduce, dim3(static_cast<unsigned>(rg)), dim3(256), 0, s,
                                 partials, S, n, scale, accumulate ? 1 : 0, gW);
    }
    // Outputs per thread and slices per batch: about 8 loads in flight per
    // thread; one CTA of 256 threads per U x 256 outputs, at most 8 per SM.
    const int64_t n4 = n / 4;
    const float4* p4 = reinterpret_cast<const float4*>(partials);
    float4* g4 = reinterpret_cast<float4*>(gW);
    const int acc = accumulate ? 1 : 0;
    auto go = [&](auto kernel, int U) {
        int64_t rg = (n4 + 256 * U - 1) / (256 * U);
        if (rg > 152 * 8) rg = 152 * 8;
        return launch_pdl_shared(kernel, dim3(static_cast<unsigned>(rg)), dim3(256), 0, s, p4,
                                 S, n4, scale, acc, g4);
    };
    if (S <= 3) return go(k_reduce_v4<4, 2>, 4);
    if (S <= 5) return go(k_reduce_v4<2, 4>, 2);
    return go(k_reduce_v4<1, 8>, 1);
}

size_t simt_gemm_workspace_bytes(int64_t T, int64_t d_in, int64_t d_out) {
    const int64_t S = slices_for(T, d_in, d_out);
    return S > 1 ? sizeof(float) * static_cast<size_t>(S * d_out * d_in) : 0;
}

cudaError_t launch_simt_gemm(const void* g, int g_bf16, const void* X, int x_bf16, int64_t T,
                             int64_t d_in, int64_t d_out, float scale, bool accumulate,
                             float* gW, float* partials, cudaStream_t s) {
    if (d_in == 0 || d_out == 0) return cudaSuccess;
    if (g_bf16 && x_bf16)
        return run<__nv_bfloat16, __nv_bfloat16>(g, X, T, d_in, d_out, scale, accumulate, gW,
                                                 partials, s);
    if (!g_bf16 && !x_bf16)
        return run<float, float>(g, X, T, d_in, d_out, scale, accumulate, gW, partials, s);
    if (g_bf16)
        return run<__nv_bfloat16, float>(g, X, T, d_in, d_out, scale, accumulate, gW, partials, s);
    return run<float, __nv_bfloat16>(g, X, T, d_in, d_out, scale, accumulate, gW, partials, s);
}

}  // namespace dust
