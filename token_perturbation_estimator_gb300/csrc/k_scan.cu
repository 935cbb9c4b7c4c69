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
//
// Precision of the decay products. A product of k factors gamma rounded to
// fp32 after every factor drifts by up to about k/2 units in the last place,
// and the drift of the chunk product B (the same for every full chunk)
// compounds along the chunk carries: at gamma = 0.9999 over 300,000 tokens
// that alone gave 3e-5 relative error in r. So P and B are multiplied out in
// fp64 and each rounded once; B is kept as an fp32 pair hi + lo (hi the
// rounded product, lo the rounded remainder), and each carry step applies
// both, so the rounding of B no longer compounds. What remains is fp32
// rounding of the sums, which does not drift.
#include "internal.cuh"

namespace dust {

namespace {

constexpr int kDrawGroup = 32;       // draws staged in shared memory at once
constexpr int64_t kCoopOffsets = 4096;  // up to this many sequences, scan all offsets
constexpr size_t kCarrySmem = 96 * 1024;  // chunk summaries staged by k_carry
// Chunks whose decay products (hi + lo pairs) the scan kernel's last CTA can
// stage beside the draw summaries for the merged carry pass.
constexpr int64_t kMergedChunks = 512;

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

// dst[e] = src[e] for e < n, by the whole CTA, loads batched 8 deep (read
// through L2: src was written by other CTAs of this grid or the previous one).
__device__ __forceinline__ void stage_cg(float* dst, const float* __restrict__ src, int64_t n) {
    for (int64_t e0 = threadIdx.x; e0 < n; e0 += 8 * static_cast<int64_t>(blockDim.x)) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t e = e0 + u * static_cast<int64_t>(blockDim.x);
            v[u] = e < n ? __ldcg(src + e) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t e = e0 + u * static_cast<int64_t>(blockDim.x);
            if (e < n) dst[e] = v[u];
        }
    }
}

// carry[j][i] = A[j+1][i] + B[j+1] * carry[j+1][i], carry[last] = 0, one
// thread per draw, with B[j] = hi + lo (Bp[2j], Bp[2j+1]) applied as two
// fused steps so that B's rounding does not compound.
__device__ __forceinline__ void carry_walk(const float* A, const float* Bp, int64_t K,
                                           int64_t nc, float* __restrict__ carry) {
    for (int64_t i = threadIdx.x; i < K; i += blockDim.x) {
        float c = 0.0f;
        carry[(nc - 1) * K + i] = 0.0f;
        // Unrolled so that the loads of later steps are issued ahead of the
        // serial chain of fused multiply-adds.
#pragma unroll 8
        for (int64_t j = nc - 1; j >= 1; --j) {
            c = fmaf(Bp[2 * j + 1], c, fmaf(Bp[2 * j], c, A[j * K + i]));
            carry[(j - 1) * K + i] = c;
        }
    }
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
    // The first draw group's loss changes (all of them when K <= 32) are
    // loaded once, every load in flight together, and serve both the mean
    // and the scan. Later draws' loads are issued in batches of independent
    // registers, so a thread waits for one memory latency per batch rather
    // than one per draw. The sum's order: each batch of 8 draws summed in
    // draw order, then the batch sums in order (the weighting kernel's direct
    // path, which centres without a scan, sums in the same order, so both
    // give the same bits).
    const int gn0 = static_cast<int>(K < kDrawGroup ? K : kDrawGroup);
    float v0[kDrawGroup];
#pragma unroll
    for (int k = 0; k < kDrawGroup; ++k) v0[k] = (k < gn0 && t < T) ? delta[k * T + t] : 0.0f;
    float mean = 0.0f;
    if (center && K > 1 && t < T) {
#pragma unroll
        for (int b = 0; b < kDrawGroup / 8; ++b) {
            if (8 * b < K) {
                float part = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (8 * b + j < K) part += v0[8 * b + j];
                mean += part;
            }
        }
        for (int64_t i0 = kDrawGroup; i0 < K; i0 += 8) {
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

    // Lane map of the decay (draw-independent): the lane's product Bl of its
    // 8 factors, for the per-draw composition below.
    float mloc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) mloc[j] = s_m[lane * 8 + j];
    float Bl = 1.0f;
#pragma unroll
    for (int j = 7; j >= 0; --j) Bl *= mloc[j];

    for (int64_t g0 = 0; g0 < K; g0 += kDrawGroup) {
        const int gn = static_cast<int>(K - g0 < kDrawGroup ? K - g0 : kDrawGroup);
        // Load the group's centred reductions c = -(delta - mean), all loads
        // of the group in flight at once.
        {
            float v[kDrawGroup];
            if (g0 == 0) {
#pragma unroll
                for (int k = 0; k < kDrawGroup; ++k) v[k] = v0[k];
            } else {
#pragma unroll
                for (int k = 0; k < kDrawGroup; ++k)
                    v[k] = (k < gn && t < T) ? delta[(g0 + k) * T + t] : 0.0f;
            }
            // In the first group warp 0 multiplies out the chunk's decay
            // products in fp64 (a chain of about 20 dependent double-precision
            // steps): the suffix over the lanes after each lane, P for the
            // lane's 8 tokens, and the chunk product B as an fp32 pair.
            if (g0 == 0 && warp == 0) {
                double Bl_d = 1.0;
#pragma unroll
                for (int j = 7; j >= 0; --j) Bl_d *= static_cast<double>(mloc[j]);
                double Bsuf = Bl_d;  // inclusive suffix product over lanes >= lane
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const double o = __shfl_down_sync(0xffffffffu, Bsuf, off);
                    if (lane + off < 32) Bsuf *= o;
                }
                double p = __shfl_down_sync(0xffffffffu, Bsuf, 1);
                if (lane == 31) p = 1.0;
#pragma unroll
                for (int j = 7; j >= 0; --j) {
                    p *= static_cast<double>(mloc[j]);
                    const int64_t tt = t0 + lane * 8 + j;
                    if (tt < T) P[tt] = static_cast<float>(p);
                }
                if (lane == 0) {
                    const float hi = static_cast<float>(Bsuf);
                    B[2 * chunk] = hi;
                    B[2 * chunk + 1] = static_cast<float>(Bsuf - static_cast<double>(hi));
                }
            }
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
    // (the host picks this form only when the draw summaries fit in s_c and
    // the chunk products in s_B).
    __shared__ unsigned int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int64_t nc = gridDim.x;
    __shared__ float s_B[2 * kMergedChunks];
    float* sA = &s_c[0][0];
    stage_cg(sA, A, nc * K);
    stage_cg(s_B, B, 2 * nc);
    __syncthreads();
    carry_walk(sA, s_B, K, nc, carry);
}

// The carry pass as its own one-CTA kernel (see carry_walk). The summaries
// are first staged in shared memory by all threads (when they fit), so the
// serial chain of each draw runs at shared-memory latency.
__global__ void __launch_bounds__(256) k_carry(const float* __restrict__ A,
                                               const float* __restrict__ B, int64_t K,
                                               int64_t n_chunks, float* __restrict__ carry,
                                               int staged) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float s_sum[];  // [n_chunks][K] A, then [n_chunks][2] B
    if (staged) {
        float* dA = s_sum;
        float* dB = s_sum + n_chunks * K;
        stage_cg(dA, A, n_chunks * K);
        stage_cg(dB, B, 2 * n_chunks);
        __syncthreads();
        carry_walk(dA, dB, K, n_chunks, carry);
    } else {
        carry_walk(A, B, K, n_chunks, carry);
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
           2 * align256(sizeof(float) * nc * K + 16) + align256(sizeof(float) * 2 * nc + 16);
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
    const bool merged = ticket && b.n_chunks <= kMergedChunks &&
                        b.n_chunks * K <= static_cast<int64_t>(kDrawGroup) * (kScanChunk + 1);
    cudaError_t e;
    {
    ProfScope ps(kStageScanLocal, s);
    e = launch_pdl_shared(k_scan_local, dim3(static_cast<unsigned>(b.n_chunks)), dim3(256), 0, s,
                          delta, K, T, seq_offsets, n_seq, gamma, center ? 1 : 0, b.r, b.P, b.A,
                          b.B, b.carry, merged ? ticket : nullptr);
    }
    if (e != cudaSuccess || merged) return e;
    const size_t smem = sizeof(float) * static_cast<size_t>(b.n_chunks * (K + 2));
    const int staged = smem <= kCarrySmem ? 1 : 0;
    const cudaError_t attr =
        ensure_smem_limit(reinterpret_cast<const void*>(k_carry), static_cast<int>(kCarrySmem));
    if (attr != cudaSuccess) return attr;
    ProfScope ps(kStageScanCarry, s);
    return launch_pdl_shared(k_carry, dim3(1), dim3(256), staged ? smem : 0, s, b.A, b.B, K,
                             b.n_chunks, b.carry, staged);
}

cudaError_t launch_scan_fixup(const ScanBuffers& b, int64_t K, int64_t T, cudaStream_t s) {
    const int64_t n = K * T;
    if (n == 0) return cudaSuccess;
    int64_t grid = (n + 255) / 256;
    if (grid > 152 * 32) grid = 152 * 32;
    ProfScope ps(kStageScanFixup, s);
    return launch_pdl_shared(k_fixup, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, b.r,
                             b.P, b.carry, K, T);
}

}  // namespace dust
