// Materialising noise kernel (dust_noise) and the forward's jitter
// y += sigma * a (dust_jitter_apply). Both walk channel pairs so one
// Box-Muller evaluation serves both channels of a pair.
#include <mutex>

#include "internal.cuh"
#include "noise.cuh"

namespace dust {

namespace {

__device__ unsigned int g_status = 0;

template <int OUT>  // 0 f32, 1 bf16, 2 u32 words
__global__ void __launch_bounds__(256) k_noise(void* __restrict__ out, uint32_t skey, int kind,
                                               int64_t draw_begin, int64_t n_draws, int64_t T,
                                               int64_t d_out, bool anti, uint32_t stream) {
    const int64_t pairs = (d_out + 1) >> 1;
    const int64_t total = n_draws * T * pairs;
    for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < total;
         q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = q / pairs;       // k * T + t
        const int64_t p = (q - row * pairs) * 2;
        const int64_t k = row / T;
        const int64_t t = row - k * T;
        const int64_t i = draw_begin + k;
        const bool has_odd = p + 1 < d_out;
        const uint32_t n0 = static_cast<uint32_t>(t * d_out + p);
        const int64_t o = row * d_out + p;
        if (OUT == 2) {
            const uint32_t kf = fold16(draw_key(skey, i, stream));
            uint32_t* w = static_cast<uint32_t*>(out);
            w[o] = word_ff(kf, fold16(n0));
            if (has_odd) w[o + 1] = word_ff(kf, fold16(n0 + 1));
            continue;
        }
        float v0, v1 = 0.0f;
        if (kind == 0) {
            v0 = noise_value(0, skey, i, n0, n0, false, anti);
            if (has_odd) v1 = noise_value(0, skey, i, n0 + 1, n0, true, anti);
        } else if (kind == 3) {
            // p is even, so p and p + 1 share their 32-channel group's word
            const int64_t bi = anti ? (i >> 1) : i;
            const uint32_t sg = (anti && (i & 1)) ? 0x80000000u : 0u;
            const int j = static_cast<int>(p & 31);
            const uint32_t w = word_ff(fold16(draw_key(skey, bi, 0)), fold16(n0 - j));
            v0 = __uint_as_float(0x3F800000u | (packed_sign_bit(w, j) ^ sg));
            v1 = __uint_as_float(0x3F800000u | (packed_sign_bit(w, j + 1) ^ sg));
        } else {
            float sgn = 1.0f;
            int64_t bi = i;
            if (anti) {
                sgn = (i & 1) ? -1.0f : 1.0f;
                bi = i >> 1;
            }
            const uint32_t nf = fold16(n0);
            const float f0 = unit_ff(fold16(draw_key(skey, bi, 0)), nf);
            const float f1 = unit_ff(fold16(draw_key(skey, bi, 1)), nf);
            gauss_pair(f0, f1, v0, v1);
            v0 *= sgn;
            v1 *= sgn;
        }
        if (OUT == 0) {
            float* f = static_cast<float*>(out);
            f[o] = v0;
            if (has_odd) f[o + 1] = v1;
        } else {
            __nv_bfloat16* h = static_cast<__nv_bfloat16*>(out);
            h[o] = __float2bfloat16_rn(v0);
            if (has_odd) h[o + 1] = __float2bfloat16_rn(v1);
        }
    }
}

template <bool BF16>
__global__ void __launch_bounds__(256) k_jitter(void* __restrict__ y, int64_t ld_y, int64_t T,
                                                int64_t d_out, uint32_t skey, int kind,
                                                int64_t draw, float sigma, bool anti) {
    const int64_t pairs = (d_out + 1) >> 1;
    const int64_t total = T * pairs;
    float sgn = 1.0f;
    int64_t bi = draw;
    if (anti) {
        sgn = (draw & 1) ? -1.0f : 1.0f;
        bi = draw >> 1;
    }
    const uint32_t kf0 = fold16(draw_key(skey, bi, 0));
    const uint32_t kf1 = fold16(draw_key(skey, bi, 1));
    const float ss = sgn * sigma;
    for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < total;
         q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = q / pairs;
        const int64_t p = (q - t * pairs) * 2;
        const bool has_odd = p + 1 < d_out;
        const uint32_t n0 = static_cast<uint32_t>(t * d_out + p);
        float a0, a1 = 0.0f;
        if (kind == 0) {
            a0 = __uint_as_float(0x3F800000u | sign_ff(kf0, fold16(n0)));
            a1 = __uint_as_float(0x3F800000u | sign_ff(kf0, fold16(n0 + 1)));
        } else if (kind == 3) {
            const int j = static_cast<int>(p & 31);
            const uint32_t w = word_ff(kf0, fold16(n0 - j));
            a0 = __uint_as_float(0x3F800000u | packed_sign_bit(w, j));
            a1 = __uint_as_float(0x3F800000u | packed_sign_bit(w, j + 1));
        } else {
            const uint32_t nf = fold16(n0);
            gauss_pair(unit_ff(kf0, nf), unit_ff(kf1, nf), a0, a1);
        }
        const int64_t o = t * ld_y + p;
        if (BF16) {
            __nv_bfloat16* h = static_cast<__nv_bfloat16*>(y);
            h[o] = __float2bfloat16_rn(fmaf(ss, a0, __bfloat162float(h[o])));
            if (has_odd) h[o + 1] = __float2bfloat16_rn(fmaf(ss, a1, __bfloat162float(h[o + 1])));
        } else {
            float* f = static_cast<float*>(y);
            f[o] = fmaf(ss, a0, f[o]);
            if (has_odd) f[o + 1] = fmaf(ss, a1, f[o + 1]);
        }
    }
}

__global__ void k_zero(float* __restrict__ p, int64_t n) {
    for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n;
         q += (int64_t)gridDim.x * blockDim.x)
        p[q] = 0.0f;
}

int grid_for(int64_t work, int per_block) {
    int64_t b = (work + per_block - 1) / per_block;
    const int64_t cap = 152 * 32;  // grid-stride beyond 32 waves of 152 SMs
    if (b > cap) b = cap;
    return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_noise(void* out, int out_kind, uint64_t seed, int kind, int64_t draw_begin,
                         int64_t n_draws, int64_t T, int64_t d_out, uint32_t flags,
                         cudaStream_t s) {
    const int64_t total = n_draws * T * ((d_out + 1) >> 1);
    if (total == 0) return cudaSuccess;
    const uint32_t skey = seed_key(seed);
    const bool anti = (flags & 2u) != 0;
    const uint32_t stream = (flags & 32u) ? 1u : 0u;
    const int grid = grid_for(total, 256);
    ProfScope ps(kStageNoise, s);
    if (out_kind == 2)
        k_noise<2><<<grid, 256, 0, s>>>(out, skey, kind, draw_begin, n_draws, T, d_out, false, stream);
    else if (out_kind == 1)
        k_noise<1><<<grid, 256, 0, s>>>(out, skey, kind, draw_begin, n_draws, T, d_out, anti, 0);
    else
        k_noise<0><<<grid, 256, 0, s>>>(out, skey, kind, draw_begin, n_draws, T, d_out, anti, 0);
    return cudaGetLastError();
}

cudaError_t launch_jitter(void* y, int y_bf16, int64_t ld_y, int64_t T, int64_t d_out,
                          uint64_t seed, int kind, int64_t draw, float sigma, uint32_t flags,
                          cudaStream_t s) {
    const int64_t total = T * ((d_out + 1) >> 1);
    if (total == 0) return cudaSuccess;
    const uint32_t skey = seed_key(seed);
    const bool anti = (flags & 2u) != 0;
    const int grid = grid_for(total, 256);
    ProfScope ps(kStageJitter, s);
    if (y_bf16)
        k_jitter<true><<<grid, 256, 0, s>>>(y, ld_y, T, d_out, skey, kind, draw, sigma, anti);
    else
        k_jitter<false><<<grid, 256, 0, s>>>(y, ld_y, T, d_out, skey, kind, draw, sigma, anti);
    return cudaGetLastError();
}

unsigned int* status_word() {
    constexpr int kMaxDev = 64;
    static unsigned int* cache[kMaxDev] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int*>(p);
    }
    return cache[dev];
}

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
    struct Entry {
        const void* kernel;
        int dev;
        int bytes;
    };
    constexpr int kMaxEntries = 256;
    static Entry done[kMaxEntries];
    static int n_done = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].kernel == kernel && done[i].dev == dev && done[i].bytes >= bytes)
            return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (n_done < kMaxEntries) done[n_done++] = Entry{kernel, dev, bytes};
    return cudaSuccess;
}

cudaError_t ensure_shared_carveout(const void* kernel) {
    struct Entry {
        const void* kernel;
        int dev;
    };
    constexpr int kMaxEntries = 256;
    static Entry done[kMaxEntries];
    static int n_done = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].kernel == kernel && done[i].dev == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (n_done < kMaxEntries) done[n_done++] = Entry{kernel, dev};
    return cudaSuccess;
}

cudaError_t launch_zero(float* p, int64_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    ProfScope ps(kStageZero, s);
    k_zero<<<grid_for(n, 256), 256, 0, s>>>(p, n);
    return cudaGetLastError();
}

}  // namespace dust
