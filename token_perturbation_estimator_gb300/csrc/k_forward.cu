// Jittered forward of a linear layer for several draws from one product:
//     Y[s][t][c] = y[t][c]                              s < clean
//     Y[s][t][c] = y[t][c] + sigma a_t^(draw_begin+k)[c]  s = clean + k
// with y = X W^T ("Dust: every token is a member of the population", section
// "Perturb the activations, not the weights": every population member runs
// the same layer and adds its own jitter to the output; the split form of
// "Scaling To Unfathomable Depth", section "Kernel Recipes", where the noise
// is added to the clean product instead of entering the weights).
//
// Persistent: one CTA per SM walks 128-token x kBN-channel tiles of y. Each
// tile's product is formed once on the tensor cores and every slice of the
// tile is written from TMEM, so X and W are read once per tile however many
// draws there are, and the jitter is regenerated in registers, never read:
//   warp 0, one thread: TMA loads of the X tile [128 x 64] and the W tile
//     [kBN x 64] per k-step (both K-major, 128-byte swizzle) into a ring;
//   warp 1, one thread: tcgen05.mma (M 128, N kBN, K 16) into one of two
//     TMEM accumulators, so the next tile's product overlaps this tile's
//     epilogue;
//   24 epilogue warps (16 for packed signs, whose arithmetic is light, so each
//     warp gets more staging buffers): each reads 32 tokens x 32 channels of y from TMEM
//     (its lane quarter), frees the accumulator after its last read, adds
//     sigma a per draw, rounds to bf16, stages the 32 x 32 block in shared
//     memory (64-byte swizzle, no bank conflicts) and writes it with a TMA
//     tensor store; two or three staging buffers per warp keep stores in
//     flight. The stores clip at T and d_out.
// All waits are bounded (1 s) and record DUST_ERR_TIMEOUT in the device
// status word instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "noise.cuh"
#include "tc_common.cuh"

namespace dust {

bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                    uint32_t box_rows);
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

namespace {

#ifndef DUST_FWD_BN
#define DUST_FWD_BN 256  // channels per tile (columns of one TMEM accumulator)
#endif
#ifndef DUST_FWD_EW
#define DUST_FWD_EW 24  // epilogue warps (Gaussian, per-channel signs)
#endif
#ifndef DUST_FWD_EW_PACKED
#define DUST_FWD_EW_PACKED 16  // (packed signs: light arithmetic, more staging buffers each)
#endif
#ifndef DUST_FWD_SUB_G
#define DUST_FWD_SUB_G 8  // TMEM columns an epilogue thread holds at a time (Gaussian)
#endif
#ifndef DUST_FWD_SUB_R
#define DUST_FWD_SUB_R 16  // (signs)
#endif
#ifndef DUST_FWD_DEEP_KSTEPS
#define DUST_FWD_DEEP_KSTEPS 32  // k-steps from which the deeper ring pays
#endif
constexpr int kBM = 128;
constexpr int kBN = DUST_FWD_BN;
constexpr int kBK = 64;  // d_in per k-step: one 128-byte swizzle row
constexpr int kEW = DUST_FWD_EW;
// Epilogue warps and threads of the kernel for a noise kind.
constexpr int ew_of(int kind) { return kind == 3 ? DUST_FWD_EW_PACKED : kEW; }
constexpr int threads_of(int kind) { return 64 + 32 * ew_of(kind); }
// Shared memory is split between the k-step ring and the epilogue's staging
// buffers in one of two ways, chosen per launch: 2 stages and 3 buffers per
// warp (short reductions, where the stores dominate), or 3 stages and 2
// buffers (long reductions, where the tensor cores need the deeper ring).
constexpr int kMaxStages = 3;
template <int KIND> constexpr int sub_cols() { return KIND == 1 ? DUST_FWD_SUB_G : DUST_FWD_SUB_R; }
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kBufBytes = 32 * 32 * 2;  // 32 tokens x 32 channels of bf16
constexpr int kSplitBytes = 3 * kStageBytes + 64 * 1024;  // ring + staging buffers
constexpr int kChunks = kBN / 32;
constexpr int kKeyTable = 64;           // per-draw keys kept in shared memory
constexpr int kSmemBytes = kSplitBytes + kKeyTable * 8 + 256 + 1024;
static_assert(kBN == 128 || kBN == 256, "two accumulators of kBN columns fit TMEM");
static_assert(kEW % 4 == 0 && DUST_FWD_EW_PACKED % 4 == 0,
              "epilogue warps cover the four TMEM lane quarters");
static_assert(kSplitBytes - 3 * kStageBytes >= kEW * kBufBytes &&
                  kSplitBytes - 3 * kStageBytes >= DUST_FWD_EW_PACKED * kBufBytes,
              "a staging buffer per warp");
static_assert(kStageBytes % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(threads_of(0) <= 1024 && threads_of(3) <= 1024, "one CTA");

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];   // accumulator holds a finished tile
    uint64_t tempty[2];  // every epilogue warp has read the accumulator
    uint64_t never;      // test hook: a barrier nothing completes
    uint32_t tmem;
    int abort;
    int issued;
    int consumed;
};

struct FwdArgs {
    int64_t T, d_in, d_out;
    int64_t n_tn, n_tiles;  // channel tiles, all tiles
    int stages, nbuf;       // k-step ring depth, staging buffers per epilogue warp
    uint32_t skey;
    int64_t draw_begin, n_draws;
    float sigma;
    int anti, clean, stall;
    unsigned int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Keys of draw (draw_begin + k) under the antithetic mapping, pre-folded, and
// the signed jitter scale of that draw.
__device__ __forceinline__ void draw_keys(const FwdArgs& a, const uint2* s_keys, int64_t k,
                                          uint32_t& kf0, uint32_t& kf1, float& ss) {
    const int64_t i = a.draw_begin + k;
    if (k < kKeyTable) {
        const uint2 kk = s_keys[k];
        kf0 = kk.x;
        kf1 = kk.y;
    } else {
        const int64_t bi = base_draw(i, a.anti != 0);
        kf0 = fold16(draw_key(a.skey, bi, 0));
        kf1 = fold16(draw_key(a.skey, bi, 1));
    }
    ss = (a.anti && (i & 1)) ? -a.sigma : a.sigma;
}

// Folded counter of channel c0 + j. With ALIGNED (n_row a multiple of 32,
// i.e. d_out a multiple of 32), adding j < 32 only sets low bits that are
// zero, so fold16(n_row + j) = fold16(n_row) ^ j.
template <bool ALIGNED>
__device__ __forceinline__ uint32_t counter_f(uint32_t n_row, uint32_t nf_row, uint32_t j) {
    return ALIGNED ? (nf_row ^ j) : fold16(n_row + j);
}

// Channels [c0 + j0, c0 + j0 + N) of one slice: pk[p] = bf16x2 of y + ss a
// for the channel pair (j0 + 2p, j0 + 2p + 1). n_row = t d_out + c0 is the
// counter of the 32-channel block's first channel (nf_row folded); w is the
// block's hash word (packed signs).
template <int KIND, bool ALIGNED, int N>
__device__ __forceinline__ void jitter_sub(const float (&y)[N], uint32_t n_row, uint32_t nf_row,
                                           int j0, uint32_t kf0, uint32_t kf1, uint32_t w,
                                           float ss, uint32_t (&pk)[N / 2]) {
    if (KIND == 1) {
#pragma unroll
        for (int p = 0; p < N / 2; ++p) {
            // Box-Muller as in gauss_pair, with sigma folded into the radius:
            // y + (ss rho) cos, y + (ss rho) sin.
            const uint32_t nf = counter_f<ALIGNED>(n_row, nf_row, j0 + 2u * p);
            const float sr = ss * neg_radius(unit_ff(kf0, nf));
            float sn, cs;
            __sincosf(centred_angle(unit_ff(kf1, nf)), &sn, &cs);
            pk[p] = pack_bf16(fmaf(sr, cs, y[2 * p]), fmaf(sr, sn, y[2 * p + 1]));
        }
    } else if (KIND == 3) {
        const uint32_t sb = __float_as_uint(ss);
#pragma unroll
        for (int p = 0; p < N / 2; ++p)
            pk[p] = pack_bf16(y[2 * p] + __uint_as_float(sb ^ packed_sign_bit(w, j0 + 2 * p)),
                              y[2 * p + 1] +
                                  __uint_as_float(sb ^ packed_sign_bit(w, j0 + 2 * p + 1)));
    } else {
        const uint32_t sb = __float_as_uint(ss);
#pragma unroll
        for (int p = 0; p < N / 2; ++p) {
            const uint32_t s0 = sign_ff(kf0, counter_f<ALIGNED>(n_row, nf_row, j0 + 2u * p));
            const uint32_t s1 = sign_ff(kf0, counter_f<ALIGNED>(n_row, nf_row, j0 + 2u * p + 1u));
            pk[p] = pack_bf16(y[2 * p] + __uint_as_float(sb ^ s0),
                              y[2 * p + 1] + __uint_as_float(sb ^ s1));
        }
    }
}

template <int KIND, bool ALIGNED>
__global__ void __launch_bounds__(threads_of(KIND), 1)
    k_forward(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
              const __grid_constant__ CUtensorMap tmY, const FwdArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int n_stages = a.stages;
    unsigned char* staging = smem + n_stages * kStageBytes;
    uint2* s_keys = reinterpret_cast<uint2*>(smem + kSplitBytes);
    Ctl* ctl = reinterpret_cast<Ctl*>(s_keys + kKeyTable);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_kb = static_cast<int>((a.d_in + kBK - 1) / kBK);

    if (threadIdx.x == 0) {
        for (int i = 0; i < n_stages; ++i) {
            tc::mbar_init(&ctl->full[i], 1);
            tc::mbar_init(&ctl->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ctl->tfull[i], 1);
            tc::mbar_init(&ctl->tempty[i], ew_of(KIND));
        }
        tc::mbar_init(&ctl->never, 1);
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->consumed = 0;
        tc::fence_mbar_init();
    }
    const int nk = a.n_draws < kKeyTable ? static_cast<int>(a.n_draws) : kKeyTable;
    for (int k = threadIdx.x; k < nk; k += blockDim.x) {
        const int64_t bi = base_draw(a.draw_begin + k, a.anti != 0);
        s_keys[k] = make_uint2(fold16(draw_key(a.skey, bi, 0)), fold16(draw_key(a.skey, bi, 1)));
    }
    if (warp == 1) {
        tc::tmem_alloc(&ctl->tmem, 2 * kBN);
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
            tc::prefetch_tmap(&tmW);
            int it = 0;  // k-steps issued, over all tiles of this CTA
            for (int64_t tile = blockIdx.x; tile < a.n_tiles && !*abort_flag; tile += gridDim.x) {
                const int32_t t0 = static_cast<int32_t>((tile / a.n_tn) * kBM);
                const int32_t n0 = static_cast<int32_t>((tile % a.n_tn) * kBN);
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int st = it % n_stages;
                    if (!tc::mbar_wait(&ctl->empty[st], ((it / n_stages) & 1) ^ 1) ||
                        *abort_flag) {
                        *abort_flag = 1;
                        break;
                    }
                    unsigned char* base = smem + st * kStageBytes;
                    tc::mbar_arrive_expect_tx(&ctl->full[st], kStageBytes);
                    tc::tma_load_2d(base, &tmX, kb * kBK, t0, &ctl->full[st]);
                    tc::tma_load_2d(base + kABytes, &tmW, kb * kBK, n0, &ctl->full[st]);
                }
            }
            ctl->issued = it;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_k(kBM, kBN);
            if (a.stall && !tc::mbar_wait(&ctl->never, 0)) *abort_flag = 1;
            int it = 0, j = 0;
            for (int64_t tile = blockIdx.x; tile < a.n_tiles && !*abort_flag;
                 tile += gridDim.x, ++j) {
                const int acc = j & 1;
                if (!tc::mbar_wait_sleep(&ctl->tempty[acc], ((j >> 1) & 1) ^ 1)) {
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d = tmem + acc * kBN;
                for (int kb = 0; kb < n_kb; ++kb, ++it) {
                    const int st = it % n_stages;
                    if (!tc::mbar_wait(&ctl->full[st], (it / n_stages) & 1) || *abort_flag) {
                        *abort_flag = 1;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t as = tc::smem_u32(smem + st * kStageBytes);
                    const uint32_t bs = as + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_bf16(d, tc::sdesc_sw128(as + 32 * kk, 16, 1024),
                                     tc::sdesc_sw128(bs + 32 * kk, 16, 1024), idesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                    tc::mma_commit(&ctl->empty[st]);
                }
                if (*abort_flag) break;
                tc::mma_commit(&ctl->tfull[acc]);
            }
            ctl->consumed = it;
        }
    } else {
        // ---------------- epilogue
        constexpr int kPerQuarter = ew_of(KIND) / 4;  // warps reading one TMEM lane quarter
        // The work of a tile's lane quarter is kChunks x n_slices items (one
        // 32-channel block of one slice each), dealt round robin to the
        // quarter's kPerQuarter warps; the deal continues across tiles so no
        // warp is always the one with an extra item. An item reloads its y
        // block from TMEM kSub columns at a time, so that a thread holds few
        // registers and many warps fit on the SM.
        const int ew = warp - 2;
        const int q = warp & 3;   // TMEM lane quarter this warp may read
        const int h = ew >> 2;    // this warp's place among the quarter's warps
        const int nbuf = a.nbuf;
        unsigned char* bufs = staging + ew * (nbuf * kBufBytes);
        const uint32_t swz = (lane >> 1) & 3;  // 64-byte swizzle of this lane's row
        constexpr int kSub = sub_cols<KIND>();
        const int n_slices = a.clean + static_cast<int>(a.n_draws);
        const int items = kChunks * n_slices;
        uint32_t used = 0;  // staging buffers this warp has filled
        int bi = 0;         // the next one, used % nbuf
        int rot = 0;        // items dealt before this tile, mod kPerQuarter
        int j = 0;
        for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++j) {
            const int acc = j & 1;
            const bool ok = tc::mbar_wait(&ctl->tfull[acc], (j >> 1) & 1);
            tc::tc_fence_after();
            if (!__all_sync(0xffffffffu, ok) || *abort_flag) {
                *abort_flag = 1;
                break;
            }
            const int64_t t0 = (tile / a.n_tn) * kBM;
            const int64_t n0 = (tile % a.n_tn) * kBN;
            const int64_t t = t0 + 32 * q + lane;
            const int32_t row_box = static_cast<int32_t>(t0 + 32 * q);
            const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + acc * kBN;
            // A lane quarter wholly past T has nothing to store (a tensor
            // store is never started outside the tensor).
            const bool rows_live = t0 + 32 * q < a.T;
            int it = h - rot;
            if (it < 0) it += kPerQuarter;
            rot = (rot + items) % kPerQuarter;
            for (; it < items; it += kPerQuarter) {
                const int cb = it % kChunks;
                const int s = it / kChunks;
                const int64_t c0 = n0 + 32 * cb;
                if (!rows_live || c0 >= a.d_out) continue;
                const uint32_t n_row = static_cast<uint32_t>(t * a.d_out + c0);
                const uint32_t nf_row = fold16(n_row);
                const bool clean_slice = s < a.clean;
                uint32_t kf0 = 0, kf1 = 0, w = 0;
                float ss = 0.0f;
                if (!clean_slice) {
                    draw_keys(a, s_keys, s - a.clean, kf0, kf1, ss);
                    if (KIND == 3) w = word_ff(kf0, nf_row);  // one word per 32-channel block
                }
                unsigned char* buf = bufs + bi * kBufBytes;
                bi = (bi + 1 == nbuf) ? 0 : bi + 1;
                if (used >= static_cast<uint32_t>(nbuf)) {
                    if (lane == 0) {
                        if (nbuf == 3) tc::bulk_wait_read<2>();
                        else if (nbuf == 2) tc::bulk_wait_read<1>();
                        else tc::bulk_wait_read<0>();
                    }
                    __syncwarp();
                }
                const uint32_t row = tc::smem_u32(buf) + lane * 64;
#pragma unroll
                for (int u = 0; u < 32 / kSub; ++u) {
                    float y[kSub];
                    tc::tmem_ld_32xN<kSub>(tq + 32 * cb + kSub * u, y);
                    uint32_t pk[kSub / 2];
                    if (clean_slice) {
#pragma unroll
                        for (int p = 0; p < kSub / 2; ++p) pk[p] = pack_bf16(y[2 * p], y[2 * p + 1]);
                    } else {
                        jitter_sub<KIND, ALIGNED, kSub>(y, n_row, nf_row, kSub * u, kf0, kf1, w,
                                                        ss, pk);
                    }
#pragma unroll
                    for (int v = 0; v < kSub / 8; ++v) {
                        const uint32_t piece = u * (kSub / 8) + v;  // 16-byte piece of the row
                        st_shared_v4(row + ((piece ^ swz) << 4), pk[4 * v], pk[4 * v + 1],
                                     pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_3d(&tmY, buf, static_cast<int32_t>(c0), row_box, s);
                    tc::bulk_commit();
                }
                ++used;
            }
            // This warp's reads of the accumulator are done: free it.
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl->tempty[acc]);
        }
        if (lane == 0) tc::bulk_wait_all();
        __syncwarp();
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        // Let every TMA load already issued land before the CTA exits.
        for (int it = ctl->consumed; it < ctl->issued; ++it)
            tc::mbar_wait(&ctl->full[it % n_stages], (it / n_stages) & 1);
        atomicExch(a.status, 5u /* DUST_ERR_TIMEOUT */);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 2 * kBN);
    }
}

// Y [slices][T][d_out] bf16 as a 3-D tensor map with 32 x 32 x 1 boxes and
// the 64-byte swizzle (a 32-channel bf16 row is 64 bytes).
bool make_tmap_slices(CUtensorMap* map, void* Y, int64_t slices, int64_t T, int64_t d_out) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d_out), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(slices)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d_out) * 2,
                             static_cast<cuuint64_t>(T) * static_cast<cuuint64_t>(d_out) * 2};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, Y, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    constexpr int kMaxDev = 64;
    static int cache[kMaxDev] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

template <int KIND, bool ALIGNED>
cudaError_t launch_kind(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty,
                        const FwdArgs& fa, dim3 grid, cudaStream_t s) {
    const cudaError_t attr =
        ensure_smem_limit(reinterpret_cast<const void*>(k_forward<KIND, ALIGNED>), kSmemBytes);
    if (attr != cudaSuccess) return attr;
    FwdArgs f = fa;
    const int nbuf = (kSplitBytes - f.stages * kStageBytes) / (ew_of(KIND) * kBufBytes);
    f.nbuf = nbuf > 3 ? 3 : nbuf;
    return launch_pdl(k_forward<KIND, ALIGNED>, grid, dim3(threads_of(KIND)), kSmemBytes, s, tx,
                      tw, ty, f);
}

}  // namespace

cudaError_t launch_forward(const void* X, const void* W, int64_t T, int64_t d_in, int64_t d_out,
                           uint64_t seed, int kind, int64_t draw_begin, int64_t n_draws,
                           float sigma, bool anti, int clean, void* Y, cudaStream_t s) {
    const int64_t slices = clean + n_draws;
    if (T * d_out * slices == 0) return cudaSuccess;
    CUtensorMap tx, tw, ty;
    if (!make_tmap_bf16(&tx, X, T, d_in, kBM) || !make_tmap_bf16(&tw, W, d_out, d_in, kBN) ||
        !make_tmap_slices(&ty, Y, slices, T, d_out))
        return cudaErrorInvalidValue;
    unsigned int* st = status_word();
    const int sms = sm_count();
    if (!st || sms <= 0) return cudaErrorUnknown;
    FwdArgs fa;
    fa.T = T;
    fa.d_in = d_in;
    fa.d_out = d_out;
    fa.n_tn = (d_out + kBN - 1) / kBN;
    fa.n_tiles = fa.n_tn * ((T + kBM - 1) / kBM);
    const bool deep = (d_in + kBK - 1) / kBK >= DUST_FWD_DEEP_KSTEPS;
    fa.stages = deep ? 3 : 2;
    fa.skey = seed_key(seed);
    fa.draw_begin = draw_begin;
    fa.n_draws = n_draws;
    fa.sigma = sigma;
    fa.anti = anti ? 1 : 0;
    fa.clean = clean;
    fa.stall = take_stall_injection() ? 1 : 0;
    fa.status = st;
    const dim3 grid(static_cast<unsigned>(fa.n_tiles < sms ? fa.n_tiles : sms));
    const bool aligned = d_out % 32 == 0;
    ProfScope ps(kStageForward, s);
    if (kind == 1)
        return aligned ? launch_kind<1, true>(tx, tw, ty, fa, grid, s)
                       : launch_kind<1, false>(tx, tw, ty, fa, grid, s);
    if (kind == 3)  // one hash word per 32-channel block: no per-channel counter
        return launch_kind<3, true>(tx, tw, ty, fa, grid, s);
    return aligned ? launch_kind<0, true>(tx, tw, ty, fa, grid, s)
                   : launch_kind<0, false>(tx, tw, ty, fa, grid, s);
}

}  // namespace dust
