// Centring of the loss reductions and the segmented reverse credit scan
//   r[t] = c[t] + m[t] * r[t+1],  m[t] = 0 at a sequence's last token, else gamma,
// ("Dust: every token is a member of the population", section "Perturb the
// activations, not the weights", the r_t equation, restarted per sequence).
//
// The recurrence is affine in r[t+1], and affine maps compose associatively,
// so it is scanned in three levels:
//   lane   : 8 consecutive tokens, serial;
//   warp   : 32 lanes (a 256-token chunk) by a shuffle scan of the lane maps;
//   chunks : one thread per draw walks the chunk maps from the end (k_carry).
// A chunk's tokens then take r_true[t] = r_local[t] + P[t] * carry[chunk],
// with P[t] the product of m from t to the chunk's last token.
#include "internal.cuh"

namespace dust {

namespace {

constexpr int kDrawGroup = 32;       // draws staged in shared memory at once
constexpr int64_t kCoopOffsets = 4096;  // up to this many sequences, scan all offsets
constexpr size_t kCarrySmem = 96 * 1024;  // chunk summaries staged by k_carry

// m[t] for the 256 tokens of a chunk: 0 where t is the last token of its
// sequence (t + 1 is an offset in seq_offsets[1..n_seq]) or t >= T.
__device__ float decay_of(int64_t t, int64_t T, const int32_t* __restrict__ so, int64_t n_seq,
                          float gamma) {
    if (t >= T - 1) return 0.0f;
    const int64_t key = t + 1;
    int64_t lo = 1, hi = n_seq;  // search seq_offsets[1..n_seq]
    while (lo <= hi) {
        const int64_t mid = (lo + hi) >> 1;
        const int64_t v = so[mid];
        if (v == key) return 0.0f;
        if (v < key) lo = mid + 1; else hi = mid - 1;
    }
    return gamma;
}

__global__ void __launch_bounds__(256) k_scan_local(const float* __restrict__ delta, int64_t K,
                                                    int64_t T, const int32_t* __restrict__ so,
                                                    int64_t n_seq, float gamma, int center,
                                                    float* __restrict__ r, float* __restrict__ P,
                                                    float* __restrict__ A, float* __restrict__ B,
                                                    float* __restrict__ carry,
                                                    unsigned int* __restrict__ ticket) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_m[kScanChunk];
    __shared__ float s_c[kDrawGroup][kScanChunk + 1];

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t chunk = blockIdx.x;
    const int64_t t0 = chunk * kScanChunk;
    const int64_t t = t0 + tid;

    if (n_seq <= kCoopOffsets) {
        // Mark the chunk's sequence ends from all offsets at once (independent
        // loads) rather than by a chain of dependent binary-search loads.
        __shared__ unsigned char s_end[kScanChunk];
        s_end[tid] = 0;
        __syncthreads();
        for (int64_t q = 1 + tid; q <= n_seq; q += blockDim.x) {
            const int64_t e = static_cast<int64_t>(so[q]) - 1 - t0;
            if (e >= 0 && e < kScanChunk) s_end[e] = 1;
        }
        __syncthreads();
        s_m[tid] = (t >= T - 1 || s_end[tid]) ? 0.0f : gamma;
    } else {
        s_m[tid] = decay_of(t, T, so, n_seq, gamma);
    }
    // Loads are issued in batches of independent registers before they are
    // used, so a thread waits for one memory latency per batch rather than one
    // per draw. The sum's order: each batch of 8 draws summed in draw order,
    // then the batch sums in order (the weighting kernel's direct path, which
    // centres without a scan, sums in the same order, so both give the same
    // bits).
    float mean = 0.0f;
    if (center && K > 1 && t < T) {
        for (int64_t i0 = 0; i0 < K; i0 += 8) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (i0 + j < K) ? delta[(i0 + j) * T + t] : 0.0f;
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + j < K) part += v[j];
            mean += part;
        }
        mean /= static_cast<float>(K);
    }
    __syncthreads();

    // Lane maps of the decay products (draw-independent): P for the lane's 8
    // tokens, then the suffix over the lanes after it.
    float mloc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) mloc[j] = s_m[lane * 8 + j];
    float Bl = 1.0f;
#pragma unroll
    for (int j = 7; j >= 0; --j) Bl *= mloc[j];
    // Inclusive suffix product of Bl over lanes >= lane.
    float Bsuf = Bl;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_down_sync(0xffffffffu, Bsuf, off);
        if (lane + off < 32) Bsuf *= o;
    }
    float Bnext = __shfl_down_sync(0xffffffffu, Bsuf, 1);
    if (lane == 31) Bnext = 1.0f;
    if (warp == 0) {
        float p = Bnext;
        for (int j = 7; j >= 0; --j) {
            p *= mloc[j];
            const int64_t tt = t0 + lane * 8 + j;
            if (tt < T) P[tt] = p;
        }
        if (lane == 0) B[chunk] = Bsuf;
    }

    for (int64_t g0 = 0; g0 < K; g0 += kDrawGroup) {
        const int gn = static_cast<int>(K - g0 < kDrawGroup ? K - g0 : kDrawGroup);
        // Load the group's centred reductions c = -(delta - mean), all loads
        // of the group in flight at once.
        {
            float v[kDrawGroup];
#pragma unroll
            for (int k = 0; k < kDrawGroup; ++k)
                v[k] = (k < gn && t < T) ? delta[(g0 + k) * T + t] : 0.0f;
#pragma unroll
            for (int k = 0; k < kDrawGroup; ++k)
                if (k < gn) s_c[k][tid] = (t < T) ? -(v[k] - mean) : 0.0f;
        }
        __syncthreads();
        for (int k = warp; k < gn; k += 8) {
            float cl[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cl[j] = s_c[k][lane * 8 + j];
            float x = 0.0f;
#pragma unroll
            for (int j = 7; j >= 0; --j) x = cl[j] + mloc[j] * x;
            // Suffix composition of the lane maps (x_l, Bl).
            float As = x, Bs = Bl;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float oA = __shfl_down_sync(0xffffffffu, As, off);
                const float oB = __shfl_down_sync(0xffffffffu, Bs, off);
                if (lane + off < 32) {
                    As = fmaf(Bs, oA, As);
                    Bs *= oB;
                }
            }
            float carry = __shfl_down_sync(0xffffffffu, As, 1);
            if (lane == 31) carry = 0.0f;
            x = carry;
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                x = cl[j] + mloc[j] * x;
                s_c[k][lane * 8 + j] = x;
            }
            if (lane == 0) A[chunk * K + g0 + k] = As;
        }
        __syncthreads();
        // Write r_local token-major: r[t][g0 + k].
        for (int e = tid; e < gn * kScanChunk; e += blockDim.x) {
            const int tok = e / gn, k = e - tok * gn;
            const int64_t tt = t0 + tok;
            if (tt < T) r[tt * K + g0 + k] = s_c[k][tok];
        }
        __syncthreads();
    }
    if (!ticket) return;
    // The last CTA to finish runs the carry pass over all chunk summaries
    // (the host picks this form only when they fit in s_c).
    __shared__ unsigned int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int64_t nc = gridDim.x;
    float* sA = &s_c[0][0];
    float* sB = sA + nc * K;
    for (int64_t e = tid; e < nc * K; e += blockDim.x) sA[e] = __ldcg(A + e);
    for (int64_t e = tid; e < nc; e += blockDim.x) sB[e] = __ldcg(B + e);
    __syncthreads();
    for (int64_t i = tid; i < K; i += blockDim.x) {
        float c = 0.0f;
        carry[(nc - 1) * K + i] = 0.0f;
        for (int64_t j = nc - 1; j >= 1; --j) {
            c = fmaf(sB[j], c, sA[j * K + i]);
            carry[(j - 1) * K + i] = c;
        }
    }
}

// carry[j][i] = A[j+1][i] + B[j+1] * carry[j+1][i], carry[last] = 0.
// The summaries are first staged in shared memory by all threads (when they
// fit), so the serial chain of each draw runs at shared-memory latency.
__global__ void __launch_bounds__(256) k_carry(const float* __restrict__ A,
                                               const float* __restrict__ B, int64_t K,
                                               int64_t n_chunks, float* __restrict__ carry,
                                               int staged) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float s_sum[];  // [n_chunks][K] A, then [n_chunks] B
    const float* sA = A;
    const float* sB = B;
    if (staged) {
        float* dA = s_sum;
        float* dB = s_sum + n_chunks * K;
        for (int64_t e = threadIdx.x; e < n_chunks * K; e += blockDim.x) dA[e] = A[e];
        for (int64_t e = threadIdx.x; e < n_chunks; e += blockDim.x) dB[e] = B[e];
        __syncthreads();
        sA = dA;
        sB = dB;
    }
    for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
        float c = 0.0f;
        carry[(n_chunks - 1) * K + i] = 0.0f;
        for (int64_t j = n_chunks - 1; j >= 1; --j) {
            c = fmaf(sB[j], c, sA[j * K + i]);
            carry[(j - 1) * K + i] = c;
        }
    }
}

__global__ void __launch_bounds__(256) k_fixup(float* __restrict__ r, const float* __restrict__ P,
                                               const float* __restrict__ carry, int64_t K,
                                               int64_t T) {
    pdl_wait();
    pdl_trigger();
    const int64_t n = K * T;
    for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n;
         q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = q / K, i = q - t * K;
        r[q] = fmaf(P[t], carry[(t / kScanChunk) * K + i], r[q]);
    }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

// Every buffer keeps at least 16 bytes of slack after it, so that a copy
// rounded up to 16 bytes never leaves the workspace.
size_t scan_workspace_bytes(int64_t K, int64_t T) {
    const int64_t nc = (T + kScanChunk - 1) / kScanChunk;
    return align256(sizeof(float) * K * T + 16) + align256(sizeof(float) * T + 16) +
           2 * align256(sizeof(float) * nc * K + 16) + align256(sizeof(float) * nc + 16);
}

ScanBuffers scan_carve(void* ws, int64_t K, int64_t T) {
    ScanBuffers b;
    b.n_chunks = (T + kScanChunk - 1) / kScanChunk;
    char* p = static_cast<char*>(ws);
    b.r = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * K * T + 16);
    b.P = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * T + 16);
    b.A = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * b.n_chunks * K + 16);
    b.carry = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * b.n_chunks * K + 16);
    b.B = reinterpret_cast<float*>(p);
    return b;
}

cudaError_t launch_scan(const float* delta, int64_t K, int64_t T, const int32_t* seq_offsets,
                        int64_t n_seq, float gamma, bool center, const ScanBuffers& b,
                        cudaStream_t s, unsigned int* ticket) {
    if (T == 0 || K == 0) return cudaSuccess;
    // Carry pass inside the scan kernel's last CTA when the chunk summaries
    // fit in its shared staging buffer and a zeroed ticket word is provided.
    const bool merged =
        ticket && b.n_chunks * (K + 1) <= static_cast<int64_t>(kDrawGroup) * (kScanChunk + 1);
    cudaError_t e;
    {
    ProfScope ps(kStageScanLocal, s);
    e = launch_pdl(k_scan_local, dim3(static_cast<unsigned>(b.n_chunks)), dim3(256), 0, s, delta,
                   K, T, seq_offsets, n_seq, gamma, center ? 1 : 0, b.r, b.P, b.A, b.B, b.carry,
                   merged ? ticket : nullptr);
    }
    if (e != cudaSuccess || merged) return e;
    const size_t smem = sizeof(float) * static_cast<size_t>(b.n_chunks * (K + 1));
    const int staged = smem <= kCarrySmem ? 1 : 0;
    static cudaError_t attr = cudaFuncSetAttribute(
        k_carry, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kCarrySmem));
    if (attr != cudaSuccess) return attr;
    ProfScope ps(kStageScanCarry, s);
    return launch_pdl(k_carry, dim3(1), dim3(256), staged ? smem : 0, s, b.A, b.B, K, b.n_chunks,
                      b.carry, staged);
}

cudaError_t launch_scan_fixup(const ScanBuffers& b, int64_t K, int64_t T, cudaStream_t s) {
    const int64_t n = K * T;
    if (n == 0) return cudaSuccess;
    int64_t grid = (n + 255) / 256;
    if (grid > 152 * 32) grid = 152 * 32;
    ProfScope ps(kStageScanFixup, s);
    return launch_pdl(k_fixup, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, b.r, b.P,
                      b.carry, K, T);
}

}  // namespace dust
