// Fused reward weighting + tensor-core contraction for layers with d_in <= 512:
//   g[t][c]  = -(1/(K sigma)) sum_i r_t^(i) a_t^(i)[c]     (made in shared memory)
//   GW[c][j] = scale * sum_t g[t][c] x[t][j]               (tcgen05, TMEM)
// ("Dust: every token is a member of the population", section "Perturb the
// activations, not the weights", the g_t and G_W equations).
//
// One CTA owns 128 output channels, the whole d_in (the fp32 accumulator is
// 128 lanes x up to 512 TMEM columns) and one slice of the tokens. Per stage
// of kBK tokens (32 by default):
//   warp 0, one thread: bulk-copies the stage's rewards (chunk-local scan
//     rows, decay products, the chunk's carry row) into shared memory on one
//     mbarrier, and the X tile [kBK tokens x d_in] by TMA on another;
//   warp 1, one thread: issues the MMAs (M 128, N <= 256 per instruction,
//     K 16) and commits the stage back to the loader and the producers;
//   warps 2.. (producers): regenerate the jitter of kBK tokens x 128 channels
//     x K draws in registers, weight it by the staged rewards, round g to
//     bf16 and store it in the 128-byte-swizzled MN-major layout the MMA reads.
// g never leaves the SM and the producers issue no global loads in their
// loop. After the last stage the producer warps drain TMEM, transpose through
// shared memory and write the slice's fp32 partial (or GW itself when there
// is one slice) with coalesced stores. All waits are bounded (1 s) and record
// DUST_ERR_TIMEOUT in the device status word instead of hanging.
#include <cuda.h>

#include <mutex>

#include "internal.cuh"
#include "noise.cuh"
#include "tc_common.cuh"

namespace dust {

bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                    uint32_t box_rows);

namespace {

#ifndef DUST_FUSED_PW
#define DUST_FUSED_PW 16      // producer warps
#endif
#ifndef DUST_FUSED_TPW
#define DUST_FUSED_TPW 2      // tokens per producer warp and stage
#endif
#ifndef DUST_FUSED_STAGES
#define DUST_FUSED_STAGES 4
#endif
#ifndef DUST_FUSED_UNROLL
#define DUST_FUSED_UNROLL 2   // draws interleaved per producer thread
#endif
constexpr int kBM = 128;                      // channels per CTA
constexpr int kPW = DUST_FUSED_PW;
constexpr int kTokPerWarp = DUST_FUSED_TPW;
constexpr int kBK = kPW * kTokPerWarp;        // tokens per stage
constexpr int kStages = DUST_FUSED_STAGES;
constexpr int kUnroll = DUST_FUSED_UNROLL;
constexpr int kDrawChunk = 32 / kTokPerWarp;  // draws whose rewards one shuffle round covers
constexpr int kThreads = 64 + 32 * kPW;
constexpr int kMaxDin = 512;
constexpr int kMaxDraws = 64;                 // K limit of this kernel
constexpr int kGTileBytes = kBM * kBK * 2;                // bf16 g tile
constexpr int kXBoxBytes = 64 * kBK * 2;                  // 64 columns x kBK tokens of X
constexpr int kXTileBytes = (kMaxDin / 64) * kXBoxBytes;
constexpr int kRwRBytes = kBK * kMaxDraws * 4;            // chunk-local scan rows
constexpr int kRwPBytes = kBK * 4;                        // decay products
constexpr int kRwCBytes = (kMaxDraws + 4) * 4;            // carry row (16-byte rounded)
constexpr int kRwBytes = (kRwRBytes + kRwPBytes + kRwCBytes + 1023) / 1024 * 1024;
constexpr int kStageBytes = kGTileBytes + kXTileBytes + kRwBytes;
constexpr int kSmemBytes = kStages * kStageBytes + kMaxDraws * 8 + 1024 + 256;
static_assert(kBK % 16 == 0, "a stage must hold whole MMA K steps of 16 tokens");
static_assert(kScanChunk % kBK == 0, "a stage must not straddle a scan chunk");
static_assert(kPW % 4 == 0, "producer warps must cover the four TMEM lane quarters");
static_assert(32 % kTokPerWarp == 0 && kDrawChunk <= 32, "tokens per warp must divide the warp");
static_assert(kThreads <= 1024, "one CTA");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kStageBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kPW * 32 * 33 * 4 <= kStages * kStageBytes, "epilogue transpose buffers");

struct Ctl {
    uint64_t full[kStages];   // X landed + all producer warps stored g
    uint64_t empty[kStages];  // the MMAs of the stage have read it
    uint64_t rw[kStages];     // the stage's rewards landed
    uint64_t done;
    uint32_t tmem;
    int abort;
    int issued;
    int consumed;
};

struct FusedArgs {
    const float* r;      // [T][K] chunk-local scan
    const float* P;      // [T]
    const float* carry;  // [n_chunks][K]
    int64_t K, T, d_in, d_out, slice;
    uint32_t skey;
    int64_t draw_begin;
    float coef, scale;
    int anti, mode;
    float* out;
    unsigned int* status;
};

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Bulk copy global -> shared (16-byte aligned, multiple of 16 bytes),
// completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(tc::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    k_fused(const __grid_constant__ CUtensorMap tmX, const FusedArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint2* s_keys = reinterpret_cast<uint2*>(smem + kStages * kStageBytes);
    Ctl* ctl = reinterpret_cast<Ctl*>(s_keys + kMaxDraws);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kBM;
    const int64_t t_lo = static_cast<int64_t>(blockIdx.y) * a.slice;
    const int64_t t_hi = (t_lo + a.slice < a.T) ? t_lo + a.slice : a.T;
    const int n_k = static_cast<int>((t_hi - t_lo + kBK - 1) / kBK);
    const int nbx = static_cast<int>((a.d_in + 63) / 64);     // X boxes per stage
    const int n_pad = nbx * 64;                                 // padded d_in
    const int n_half = n_pad > 256 ? 2 : 1;
    const uint32_t tmem_cols = n_pad > 256 ? 512u : (n_pad > 128 ? 256u : (n_pad > 64 ? 128u : 64u));
    const int K = static_cast<int>(a.K);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&ctl->full[i], 1 + kPW);  // X loader + one arrive per producer warp
            tc::mbar_init(&ctl->empty[i], 1);
            tc::mbar_init(&ctl->rw[i], 1);
        }
        tc::mbar_init(&ctl->done, 1);
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->consumed = 0;
        tc::fence_mbar_init();
    }
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
        const int64_t bi = base_draw(a.draw_begin + i, a.anti != 0);
        s_keys[i] = make_uint2(fold16(draw_key(a.skey, bi, 0)), fold16(draw_key(a.skey, bi, 1)));
    }
    if (warp == 1) {
        tc::tmem_alloc(&ctl->tmem, tmem_cols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    volatile int* abort_flag = &ctl->abort;
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            tc::prefetch_tmap(&tmX);
            int it = 0;
            for (; it < n_k; ++it) {
                const int st = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!tc::mbar_wait_sleep(&ctl->empty[st], ph ^ 1) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                unsigned char* base = smem + st * kStageBytes;
                const int64_t tb = t_lo + static_cast<int64_t>(it) * kBK;
                const int64_t left = a.T - tb;
                const uint32_t ntok = static_cast<uint32_t>(left < kBK ? left : kBK);
                // rewards: r rows, P, and the chunk's carry row (rounded to 16 B)
                unsigned char* rw = base + kGTileBytes + kXTileBytes;
                const uint32_t rb = round16(ntok * K * 4);
                const uint32_t pb = round16(ntok * 4);
                const uint64_t cbyte = static_cast<uint64_t>(tb / kScanChunk) * K * 4;
                const uint64_t cstart = cbyte & ~static_cast<uint64_t>(15);
                const uint32_t cb = round16(static_cast<uint32_t>(cbyte - cstart) + K * 4);
                tc::mbar_arrive_expect_tx(&ctl->rw[st], rb + pb + cb);
                bulk_g2s(rw, a.r + tb * K, rb, &ctl->rw[st]);
                bulk_g2s(rw + kRwRBytes, a.P + tb, pb, &ctl->rw[st]);
                bulk_g2s(rw + kRwRBytes + kRwPBytes,
                         reinterpret_cast<const unsigned char*>(a.carry) + cstart, cb,
                         &ctl->rw[st]);
                // X tile
                const int32_t y = static_cast<int32_t>(tb);
                tc::mbar_arrive_expect_tx(&ctl->full[st], nbx * kXBoxBytes);
                for (int q = 0; q < nbx; ++q)
                    tc::tma_load_2d(base + kGTileBytes + q * kXBoxBytes, &tmX, 64 * q, y,
                                    &ctl->full[st]);
            }
            ctl->issued = it;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id0 = tc::idesc_bf16_mn(kBM, n_pad > 256 ? 256 : n_pad);
            const uint32_t id1 = tc::idesc_bf16_mn(kBM, n_pad > 256 ? n_pad - 256 : 16);
            int it = 0;
            for (; it < n_k; ++it) {
                const int st = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!tc::mbar_wait_sleep(&ctl->full[st], ph) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t gs = tc::smem_u32(smem + st * kStageBytes);
                const uint32_t xs = gs + kGTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t ad = tc::sdesc_sw128(gs + kk * 2048, kBK * 128, 1024);
                    const uint64_t b0 = tc::sdesc_sw128(xs + kk * 2048, kXBoxBytes, 1024);
                    tc::mma_bf16(tmem, ad, b0, id0, (it | kk) != 0 ? 1u : 0u);
                    if (n_half == 2) {
                        const uint64_t b1 =
                            tc::sdesc_sw128(xs + 4 * kXBoxBytes + kk * 2048, kXBoxBytes, 1024);
                        tc::mma_bf16(tmem + 256, ad, b1, id1, (it | kk) != 0 ? 1u : 0u);
                    }
                }
                tc::mma_commit(&ctl->empty[st]);
            }
            ctl->consumed = it;
            tc::mma_commit(&ctl->done);
        }
    } else {
        // ---------------- producers: kTokPerWarp tokens x 4 channels per thread
        const int pw = warp - 2;
        const int64_t c0 = m0 + 4 * lane;  // first of this lane's 4 channels
        // smem byte offsets of this lane's 8 bytes in a token row of the g tile
        const int blk = lane >> 4;
        const int chunk16 = (lane & 15) >> 1;
        const int sub8 = (lane & 1) * 8;
        // Lane l builds the reward of token row pw * kTokPerWarp + l / kDrawChunk,
        // draw i0 + l % kDrawChunk; the draw loop broadcasts it by shuffles.
        const int tok = lane / kDrawChunk;
        const int dl = lane % kDrawChunk;
        const int trow = pw * kTokPerWarp + tok;
        for (int it = 0; it < n_k; ++it) {
            const int st = it % kStages;
            const uint32_t ph = (it / kStages) & 1;
            const int64_t t0 = t_lo + static_cast<int64_t>(it) * kBK;
            const int64_t tb = t0 + pw * kTokPerWarp;
            const unsigned char* rw = smem + st * kStageBytes + kGTileBytes + kXTileBytes;
            const float* s_r = reinterpret_cast<const float*>(rw);
            const float* s_P = reinterpret_cast<const float*>(rw + kRwRBytes);
            const float* s_c = reinterpret_cast<const float*>(rw + kRwRBytes + kRwPBytes) +
                               (((t0 / kScanChunk) * K) & 3);  // row start within 16 B
            float acc[kTokPerWarp][4];
#pragma unroll
            for (int j = 0; j < kTokPerWarp; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[j][c] = 0.0f;
            uint32_t nf[kTokPerWarp][4];
#pragma unroll
            for (int j = 0; j < kTokPerWarp; ++j) {
                const uint32_t base = static_cast<uint32_t>((tb + j) * a.d_out + c0);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    nf[j][c] = fold16(base + (KIND == 1 ? 2u * (c >> 1) : static_cast<uint32_t>(c)));
            }
            const bool landed = tc::mbar_wait(&ctl->rw[st], ph);
            if (!__all_sync(0xffffffffu, landed) || *abort_flag) {
                *abort_flag = 1;
                break;
            }
            if (tb < t_hi) {
                for (int i0 = 0; i0 < K; i0 += kDrawChunk) {
                    float v = 0.0f;
                    const int dr = i0 + dl;
                    if (t0 + trow < t_hi && dr < K) {
                        v = fmaf(s_P[trow], s_c[dr], s_r[trow * K + dr]) * a.coef;
                        if (a.anti && ((a.draw_begin + dr) & 1)) v = -v;
                    }
                    const int kn = (K - i0 < kDrawChunk) ? K - i0 : kDrawChunk;
#pragma unroll kUnroll
                    for (int k = 0; k < kn; ++k) {
                        const uint2 key = s_keys[i0 + k];
                        float rr[kTokPerWarp];
#pragma unroll
                        for (int j = 0; j < kTokPerWarp; ++j)
                            rr[j] = __shfl_sync(0xffffffffu, v, j * kDrawChunk + k);
                        if (KIND == 1) {
#pragma unroll
                            for (int j = 0; j < kTokPerWarp; ++j)
#pragma unroll
                                for (int p = 0; p < 2; ++p) {
                                    const float f0 = unit_ff(key.x, nf[j][2 * p]);
                                    const float f1 = unit_ff(key.y, nf[j][2 * p]);
                                    const float tr = rr[j] * neg_radius(f0);
                                    float sn, cs;
                                    __sincosf(centred_angle(f1), &sn, &cs);
                                    acc[j][2 * p] = fmaf(tr, cs, acc[j][2 * p]);
                                    acc[j][2 * p + 1] = fmaf(tr, sn, acc[j][2 * p + 1]);
                                }
                        } else {
#pragma unroll
                            for (int j = 0; j < kTokPerWarp; ++j) {
                                const uint32_t rb = __float_as_uint(rr[j]);
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    acc[j][c] += __uint_as_float(rb ^ sign_ff(key.x, nf[j][c]));
                            }
                        }
                    }
                }
            }
            // Channels past d_out and tokens past the slice contribute zero.
#pragma unroll
            for (int j = 0; j < kTokPerWarp; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (c0 + c >= a.d_out || tb + j >= t_hi) acc[j][c] = 0.0f;
            const bool ready = tc::mbar_wait(&ctl->empty[st], ph ^ 1);
            if (!__all_sync(0xffffffffu, ready) || *abort_flag) {
                *abort_flag = 1;
                break;
            }
            const uint32_t gs = tc::smem_u32(smem + st * kStageBytes);
#pragma unroll
            for (int j = 0; j < kTokPerWarp; ++j) {
                const int row = pw * kTokPerWarp + j;  // token row within the stage
                const uint32_t addr = gs + blk * (kBK * 128) + row * 128 +
                                      ((chunk16 ^ (row & 7)) << 4) + sub8;
                st_shared_v2(addr, pack_bf16(acc[j][0], acc[j][1]), pack_bf16(acc[j][2], acc[j][3]));
            }
            // Each lane makes its own stores visible to the tensor core's
            // async proxy; the warp then arrives once.
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl->full[st]);
        }
        // ---------------- epilogue: TMEM -> shared (transpose) -> partial tile
        const bool ok = tc::mbar_wait(&ctl->done, 0);
        tc::tc_fence_after();
        if (!ok) *abort_flag = 1;
        if (ok && !*abort_flag && n_k > 0) {
            // The stage ring is idle now; each producer warp gets a 32 x 33
            // float transpose buffer in it.
            float* tbuf = reinterpret_cast<float*>(smem) + pw * (32 * 33);
            const int q = warp & 3;  // TMEM lane quarter this warp may read
            const int64_t row0 = m0 + 32 * q;
            // column blocks of 32 handled by this warp: pw / 4, pw / 4 + kPW / 4, ...
            for (int cb = pw >> 2; cb * 32 < n_pad; cb += kPW / 4) {
                float vv[32];
                tc::tmem_ld_32x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + cb * 32, vv);
#pragma unroll
                for (int u = 0; u < 32; ++u) tbuf[lane * 33 + u] = vv[u];  // row lane, column u
                __syncwarp();
                const int64_t col = static_cast<int64_t>(cb) * 32 + lane;
                if (col < a.d_in) {
                    for (int rr = 0; rr < 32; ++rr) {
                        const int64_t row = row0 + rr;
                        if (row >= a.d_out) break;
                        const float v = tbuf[rr * 33 + lane];
                        float* dst = (a.mode == 0)
                                         ? a.out + (static_cast<int64_t>(blockIdx.y) * a.d_out + row) *
                                                       a.d_in + col
                                         : a.out + row * a.d_in + col;
                        if (a.mode == 0) *dst = v;
                        else if (a.mode == 1) *dst = a.scale * v;
                        else *dst += a.scale * v;
                    }
                }
                __syncwarp();
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        // Let every bulk copy already issued land before the CTA exits.
        for (int it = ctl->consumed; it < ctl->issued; ++it) {
            tc::mbar_wait(&ctl->full[it % kStages], (it / kStages) & 1);
            tc::mbar_wait(&ctl->rw[it % kStages], (it / kStages) & 1);
        }
        atomicExch(a.status, 5u /* DUST_ERR_TIMEOUT */);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, tmem_cols);
    }
}

int64_t fused_slices(int64_t T, int64_t d_out) {
    const int64_t tiles = (d_out + kBM - 1) / kBM;
    int64_t S = 152 / tiles;
    const int64_t max_s = (T + 2 * kBK - 1) / (2 * kBK);
    if (S > max_s) S = max_s;
    return S < 1 ? 1 : S;
}

}  // namespace

bool fused_supported(int64_t d_in, int64_t d_out, int64_t K) {
    return d_in > 0 && d_in <= kMaxDin && d_in % 8 == 0 && d_out > 0 && d_out % 8 == 0 &&
           K >= 1 && K <= kMaxDraws;
}

size_t fused_workspace_bytes(int64_t T, int64_t d_in, int64_t d_out) {
    const int64_t S = fused_slices(T, d_out);
    return S > 1 ? sizeof(float) * static_cast<size_t>(S * d_out * d_in) : 0;
}

cudaError_t launch_fused(const ScanBuffers& b, const void* X, int64_t K, int64_t T, int64_t d_in,
                         int64_t d_out, uint64_t seed, int kind, int64_t draw_begin, float coef,
                         bool anti, float scale, bool accumulate, float* gW, float* partials,
                         cudaStream_t s) {
    CUtensorMap tx;
    if (!make_tmap_bf16(&tx, X, T, d_in, kBK)) return cudaErrorInvalidValue;
    cudaError_t attr_err =
        ensure_smem_limit(reinterpret_cast<const void*>(k_fused<0>), kSmemBytes);
    if (attr_err == cudaSuccess)
        attr_err = ensure_smem_limit(reinterpret_cast<const void*>(k_fused<1>), kSmemBytes);
    if (attr_err != cudaSuccess) return attr_err;
    unsigned int* st = status_word();
    if (!st) return cudaErrorUnknown;
    const int64_t S = fused_slices(T, d_out);
    int64_t slice = (T + S - 1) / S;
    slice = (slice + kBK - 1) / kBK * kBK;
    const int64_t S_used = (T + slice - 1) / slice;
    FusedArgs fa;
    fa.r = b.r;
    fa.P = b.P;
    fa.carry = b.carry;
    fa.K = K;
    fa.T = T;
    fa.d_in = d_in;
    fa.d_out = d_out;
    fa.slice = slice;
    fa.skey = seed_key(seed);
    fa.draw_begin = draw_begin;
    fa.coef = coef;
    fa.scale = scale;
    fa.anti = anti ? 1 : 0;
    fa.mode = (S_used > 1) ? 0 : (accumulate ? 2 : 1);
    fa.out = (S_used > 1) ? partials : gW;
    fa.status = st;
    dim3 grid(static_cast<unsigned>((d_out + kBM - 1) / kBM), static_cast<unsigned>(S_used));
    cudaError_t e;
    {
        ProfScope ps(kStageFused, s);
        if (kind == 1)
            e = launch_pdl(k_fused<1>, grid, dim3(kThreads), kSmemBytes, s, tx, fa);
        else
            e = launch_pdl(k_fused<0>, grid, dim3(kThreads), kSmemBytes, s, tx, fa);
    }
    if (e != cudaSuccess || S_used == 1) return e;
    return launch_reduce(partials, S_used, d_out * d_in, scale, accumulate, gW, s);
}

}  // namespace dust
