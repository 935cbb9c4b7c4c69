// Tensor-core contraction GW[c][j] = scale * sum_t g[t][c] x[t][j] ("Dust:
// every token is a member of the population", section "Perturb the
// activations, not the weights", the G_W equation) with tcgen05 MMAs on
// sm_103a: bf16 operands, fp32 accumulation in TMEM.
//
// Operands are used as stored, both token-major ("MN-major" in tcgen05
// terms): A = g^T is read from g [T][d_out], B = X from X [T][d_in]. TMA
// brings 64 x 64 boxes with the 128-byte swizzle into a 4-stage ring; one
// thread issues the MMAs (M = 128 channels, N = 256 inputs, K = 16 tokens)
// and commits each stage back to the loader; four warps drain TMEM.
//
// Tile of one CTA: 128 channels x 256 inputs x one slice of the tokens. When
// the output tiles alone cannot fill the GPU, the tokens are cut into S
// fixed slices whose fp32 partials are summed afterwards in slice order, so
// the result does not depend on scheduling.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace dust {

namespace {

#ifndef DUST_GEMM_MT
#define DUST_GEMM_MT 1       // 128-row accumulators per CTA (1 or 2)
#endif
#ifndef DUST_GEMM_BN
#define DUST_GEMM_BN 256     // inputs per CTA tile (64..256)
#endif
#ifndef DUST_GEMM_BK
#define DUST_GEMM_BK 64      // tokens per stage
#endif
#ifndef DUST_GEMM_STAGES
#define DUST_GEMM_STAGES 4
#endif
constexpr int kMT = DUST_GEMM_MT;
constexpr int kBM = 128 * kMT, kBN = DUST_GEMM_BN, kBK = DUST_GEMM_BK, kStages = DUST_GEMM_STAGES;
constexpr int kBoxBytes = 64 * kBK * 2;                 // one 64-wide bf16 box of kBK rows
constexpr int kABytes = (kBM / 64) * kBoxBytes;
constexpr int kBBytes = (kBN / 64) * kBoxBytes;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr uint32_t kTmemCols = (kMT * kBN <= 256) ? 256u : 512u;
constexpr uint32_t kIdesc = tc::idesc_bf16_mn(128, kBN);
static_assert(kMT * kBN <= 512, "accumulators must fit the 512 TMEM columns");
static_assert(kBK % 16 == 0 && kBN % 64 == 0, "tile shape");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t done;
    uint64_t never;  // no thread ever arrives here (test hook for the bounded waits)
    uint32_t tmem;
    int abort;
    int issued;
    int consumed;
};

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              int64_t d_in, int64_t d_out, int64_t T, int64_t slice, float* __restrict__ out,
              float scale, int mode, unsigned int* __restrict__ status, int stall) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + kStages * kStageBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBN;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM;
    const int64_t t_lo = static_cast<int64_t>(blockIdx.z) * slice;
    const int64_t t_hi = (t_lo + slice < T) ? t_lo + slice : T;
    const int n_k = static_cast<int>((t_hi - t_lo + kBK - 1) / kBK);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&ctl->full[i], 1);
            tc::mbar_init(&ctl->empty[i], 1);
        }
        tc::mbar_init(&ctl->done, 1);
        tc::mbar_init(&ctl->never, 1);
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->consumed = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&ctl->tmem, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    volatile int* abort_flag = &ctl->abort;
    pdl_wait();  // g and X come from the kernels before this one
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmA);
        tc::prefetch_tmap(&tmB);
        int it = 0;
        for (; it < n_k; ++it) {
            const int st = it % kStages;
            const uint32_t ph = (it / kStages) & 1;
            if (!tc::mbar_wait(&ctl->empty[st], ph ^ 1) || *abort_flag) {
                *abort_flag = 1;
                break;
            }
            unsigned char* a = smem + st * kStageBytes;
            unsigned char* b = a + kABytes;
            const int32_t y = static_cast<int32_t>(t_lo + static_cast<int64_t>(it) * kBK);
            tc::mbar_arrive_expect_tx(&ctl->full[st], kStageBytes);
#pragma unroll
            for (int q = 0; q < kBM / 64; ++q)
                tc::tma_load_2d(a + q * kBoxBytes, &tmA, static_cast<int32_t>(m0 + 64 * q), y,
                                &ctl->full[st]);
#pragma unroll
            for (int q = 0; q < kBN / 64; ++q)
                tc::tma_load_2d(b + q * kBoxBytes, &tmB, static_cast<int32_t>(n0 + 64 * q), y,
                                &ctl->full[st]);
        }
        ctl->issued = it;
    } else if (warp == 1 && lane == 0) {
        // Test hook: wait on a barrier no one arrives at, so that the bounded
        // wait runs out and the kernel takes its timeout path.
        if (stall && !tc::mbar_wait(&ctl->never, 0)) *abort_flag = 1;
        int it = 0;
        for (; it < n_k && !*abort_flag; ++it) {
            const int st = it % kStages;
            const uint32_t ph = (it / kStages) & 1;
            if (!tc::mbar_wait(&ctl->full[st], ph) || *abort_flag) {
                *abort_flag = 1;
                break;
            }
            tc::tc_fence_after();
            const uint32_t a = tc::smem_u32(smem + st * kStageBytes);
            const uint32_t b = a + kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint64_t bd = tc::sdesc_sw128(b + kk * 2048, kBoxBytes, 1024);
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) {
                    const uint64_t ad =
                        tc::sdesc_sw128(a + 2 * mt * kBoxBytes + kk * 2048, kBoxBytes, 1024);
                    tc::mma_bf16(tmem + mt * kBN, ad, bd, kIdesc, (it | kk) != 0 ? 1u : 0u);
                }
            }
            tc::mma_commit(&ctl->empty[st]);
        }
        ctl->consumed = it;
        tc::mma_commit(&ctl->done);
    } else if (warp >= 2) {
        const bool ok = tc::mbar_wait(&ctl->done, 0);
        tc::tc_fence_after();
        if (!ok) *abort_flag = 1;
        if (ok && !*abort_flag && n_k > 0) {
            const int q = warp & 3;  // TMEM lane quarter this warp may access
#pragma unroll 1
            for (int mt = 0; mt < kMT; ++mt) {
                const int64_t row = m0 + 128 * mt + 32 * q + lane;
                float* dst = nullptr;
                if (row < d_out) {
                    dst = (mode == 0)
                              ? out + (static_cast<int64_t>(blockIdx.z) * d_out + row) * d_in
                              : out + row * d_in;
                }
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    float v[32];
                    tc::tmem_ld_32x32(
                        tmem + (static_cast<uint32_t>(32 * q) << 16) + mt * kBN + c * 32, v);
                    const int64_t j0 = n0 + c * 32;
                    if (!dst || j0 >= d_in) continue;
                    if (j0 + 32 <= d_in) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            float4 w4 = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2],
                                                    v[4 * u + 3]);
                            float4* p = reinterpret_cast<float4*>(dst + j0 + 4 * u);
                            if (mode == 0) {
                                *p = w4;
                            } else if (mode == 1) {
                                *p = make_float4(scale * w4.x, scale * w4.y, scale * w4.z,
                                                 scale * w4.w);
                            } else {
                                float4 o = *p;
                                *p = make_float4(o.x + scale * w4.x, o.y + scale * w4.y,
                                                 o.z + scale * w4.z, o.w + scale * w4.w);
                            }
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            if (j0 + u >= d_in) continue;
                            if (mode == 0) dst[j0 + u] = v[u];
                            else if (mode == 1) dst[j0 + u] = scale * v[u];
                            else dst[j0 + u] += scale * v[u];
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        // Let every TMA copy already issued land before the CTA exits.
        for (int it = ctl->consumed; it < ctl->issued; ++it)
            tc::mbar_wait(&ctl->full[it % kStages], (it / kStages) & 1);
        atomicExch(status, 5u /* DUST_ERR_TIMEOUT */);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int64_t tc_slices(int64_t T, int64_t d_in, int64_t d_out) {
    const int64_t tiles = ((d_out + kBM - 1) / kBM) * ((d_in + kBN - 1) / kBN);
    int64_t S = 152 / tiles;
    const int64_t max_s = (T + 4 * kBK - 1) / (4 * kBK);  // at least 4 k-steps per slice
    if (S > max_s) S = max_s;
    return S < 1 ? 1 : S;
}

}  // namespace

// A bf16 [rows][cols] row-major matrix as a 2-D tensor map with boxes of 64
// columns x box_rows rows and the 128-byte swizzle; false if the driver
// refuses it.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                    uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_gemm_supported(const void* g, const void* X, int64_t d_in, int64_t d_out) {
    return (d_in % 8 == 0) && (d_out % 8 == 0) && d_in > 0 && d_out > 0 &&
           (reinterpret_cast<uintptr_t>(g) % 16 == 0) &&
           (reinterpret_cast<uintptr_t>(X) % 16 == 0) && encode_fn() != nullptr;
}

size_t tc_gemm_workspace_bytes(int64_t T, int64_t d_in, int64_t d_out) {
    const int64_t S = tc_slices(T, d_in, d_out);
    return S > 1 ? sizeof(float) * static_cast<size_t>(S * d_out * d_in) : 0;
}

int64_t tc_gemm_tiles(int64_t d_in, int64_t d_out) {
    return ((d_out + kBM - 1) / kBM) * ((d_in + kBN - 1) / kBN);
}

cudaError_t launch_tc_gemm(const void* g, const void* X, int64_t T, int64_t d_in, int64_t d_out,
                           float scale, bool accumulate, float* gW, float* partials,
                           cudaStream_t s) {
    CUtensorMap ta, tb;
    if (!make_tmap_bf16(&ta, g, T, d_out, kBK) || !make_tmap_bf16(&tb, X, T, d_in, kBK))
        return cudaErrorInvalidValue;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    unsigned int* st = status_word();
    if (!st) return cudaErrorUnknown;
    const int64_t S = tc_slices(T, d_in, d_out);
    int64_t slice = (T + S - 1) / S;
    slice = (slice + kBK - 1) / kBK * kBK;
    const int64_t S_used = (T + slice - 1) / slice;
    dim3 grid(static_cast<unsigned>((d_in + kBN - 1) / kBN),
              static_cast<unsigned>((d_out + kBM - 1) / kBM), static_cast<unsigned>(S_used));
    cudaError_t e;
    const int mode = (S_used > 1) ? 0 : (accumulate ? 2 : 1);
    {
        ProfScope ps(kStageGemmTc, s);
        e = launch_pdl(k_gemm_tc, grid, dim3(kThreads), kSmemBytes, s, ta, tb, d_in, d_out, T,
                       slice, S_used > 1 ? partials : gW, scale, mode, st,
                       take_stall_injection() ? 1 : 0);
    }
    if (e != cudaSuccess || S_used == 1) return e;
    return launch_reduce(partials, S_used, d_out * d_in, scale, accumulate, gW, s);
}

}  // namespace dust
