// Tensor-core contraction GW[c][j] = scale * sum_t g[t][c] x[t][j] ("Dust:
// every token is a member of the population", section "Perturb the
// activations, not the weights", the G_W equation) with tcgen05 MMAs on
// sm_103a: bf16 operands, fp32 accumulation in TMEM.
//
// Operands are used as stored, both token-major ("MN-major" in tcgen05
// terms): A = g^T is read from g [T][d_out], B = X from X [T][d_in]. TMA
// brings 64 x 64 boxes with the 128-byte swizzle into a 4-stage ring; one
// thread issues the MMAs (M = 128 channels, N = 256 inputs, K = 16 tokens)
// and commits each stage back to the loader; four warps drain TMEM through
// the idle stage buffers, so that GW is stored along its rows.
//
// Tile of one CTA: 128 x MT channels x 256 inputs x one slice of the tokens,
// MT = 1 or 2 accumulators of 128 rows (MT = 2 uses all 512 TMEM columns and
// a 3-stage ring of 64 KB stages). The larger tile moves a third fewer
// operand bytes from L2 into shared memory per FLOP and loads shared memory
// less per MMA (measured: 4096^2 contraction 781 -> 623 us, qkv 1024 x 3072
// 104 -> 77 us); it is used where every token slice stays long (see
// tc_tile_rows). When the output tiles alone cannot fill the GPU, the tokens
// are cut into S fixed slices whose fp32 partials are summed in slice order,
// so the result does not depend on scheduling: inside a thread-block cluster
// of the S CTAs when all clusters fit at once (one 128-row accumulator at a
// time), else by a reduction kernel.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "tc_common.cuh"

namespace dust {

namespace {

#ifndef DUST_GEMM_BN
#define DUST_GEMM_BN 256     // inputs per CTA tile (64..256)
#endif
#ifndef DUST_GEMM_BK
#define DUST_GEMM_BK 64      // tokens per stage
#endif
#ifndef DUST_GEMM_CLUSTER_REDUCE
#define DUST_GEMM_CLUSTER_REDUCE 1  // reduce the token slices in a cluster (else partials)
#endif
#ifndef DUST_GEMM_PULL
#define DUST_GEMM_PULL 1  // slices pulled by the summing CTA (else pushed to it)
#endif
// The larger tile (two accumulators) where every token slice keeps at least
// this many tokens (0: never).
#ifndef DUST_GEMM_MT2_MIN_SLICE
#define DUST_GEMM_MT2_MIN_SLICE 4096
#endif
constexpr bool kClusterReduce = DUST_GEMM_CLUSTER_REDUCE != 0;
constexpr bool kPull = DUST_GEMM_PULL != 0;
constexpr int kBN = DUST_GEMM_BN, kBK = DUST_GEMM_BK;
constexpr int kBoxBytes = 64 * kBK * 2;                 // one 64-wide bf16 box of kBK rows
// Builds of the kernel, by what else shares its SM ("fit"):
//   0: 192 threads (warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue), no
//      register bound: the kernel alone on the SM;
//   1: the same at most 80 registers a thread, beside four weighting CTAs;
//   2: 128 threads at most 32 registers (warp 0 TMA, warp 1 MMA + TMEM, then
//      all four warps the epilogue), beside five weighting CTAs, which hold
//      61,440 of the SM's 65,536 registers: the 4,096 left are this CTA's.
constexpr int threads_of(int fit) { return fit == 2 ? 128 : 192; }
constexpr int min_ctas_of(int fit) { return fit == 0 ? 1 : fit == 1 ? 4 : 16; }
constexpr uint32_t kIdesc = tc::idesc_bf16_mn(128, kBN);
static_assert(kBK % 16 == 0 && kBN % 64 == 0, "tile shape");

// Shape of the kernel with MT accumulators of 128 rows.
template <int MT>
struct Cfg {
    static constexpr int kBM = 128 * MT;                       // channels per tile
    static constexpr int kStages = MT == 1 ? 4 : 3;            // stages in flight
    static constexpr int kABytes = (kBM / 64) * kBoxBytes;
    static constexpr int kBBytes = (kBN / 64) * kBoxBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;
    static constexpr uint32_t kTmemCols = (MT * kBN <= 256) ? 256u : 512u;
    static_assert(MT * kBN <= 512, "accumulators must fit the 512 TMEM columns");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

template <int MT>
struct Ctl {
    uint64_t full[Cfg<MT>::kStages];
    uint64_t empty[Cfg<MT>::kStages];
    uint64_t done;
    uint64_t never;  // no thread ever arrives here (test hook for the bounded waits)
    uint32_t tmem;
    int abort;
    int issued;
    int consumed;
};

// Cluster reduction of the token slices (modes 3 and 4). The S CTAs of one
// output tile (one per token slice, 2 <= S <= 8) form a cluster of S along z.
// After every CTA's main loop, CTA z sends row block d (ceil(128 / S) rows of
// its fp32 accumulator, fewer in the last block) into slot z of CTA d's
// shared memory; CTA d then sums its rows
// over the slots in slice order and writes scale * sum (+ GW when
// accumulating) to GW. The stage buffers, idle after the main loop, hold the
// slots. Every thread of every CTA passes both cluster barriers, also after a
// timeout, so no CTA of the cluster waits on one that left.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

constexpr int kRowPad = kBN + 4;  // floats per slot row (16-byte pad: conflict-free stores)
constexpr int kMaxClusterSlices = 8;  // portable cluster size
constexpr int kReduceBytes = Cfg<1>::kStages * Cfg<1>::kStageBytes;  // stage buffers, MT = 1
// S slots of ceil(128 / S) rows each; the most rows over S = 2..8 is 133 (S = 7).
static_assert(133 * kRowPad * 4 <= kReduceBytes, "slots fit in the stage buffers");
// The epilogue stages 128 accumulator rows at a time through the stage buffers.
static_assert(128 * kRowPad * 4 <= Cfg<2>::kStages * Cfg<2>::kStageBytes, "rows fit (MT = 2)");

__device__ void cluster_reduce(unsigned char* smem, uint32_t tmem, bool ok, int64_t m0,
                               int64_t n0, int64_t d_in, int64_t d_out, float* __restrict__ gW,
                               float scale, bool accumulate) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = static_cast<int>(gridDim.z);
    const int R = (128 + S - 1) / S;  // rows summed by each CTA (the last may have fewer)
    const uint32_t me = cluster_rank();
    const int R_me = (128 - static_cast<int>(me) * R < R) ? 128 - static_cast<int>(me) * R : R;
    float* slots = reinterpret_cast<float*>(smem);  // [S][R][kRowPad]
    cluster_sync_all();  // every CTA's main loop is over: its stage buffers are free
    if (warp >= 2 && ok) {
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const uint32_t dst = static_cast<uint32_t>(row / R);
        const uint32_t local = tc::smem_u32(slots + (static_cast<int>(me) * R + row % R) * kRowPad);
        const uint32_t remote = map_to_rank(local, dst);
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
            float v[32];
            tc::tmem_ld_32x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + c * 32, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_cluster_v4(remote + 4u * (c * 32 + 4 * u), v[4 * u], v[4 * u + 1],
                              v[4 * u + 2], v[4 * u + 3]);
        }
    }
    cluster_sync_all();  // every slot row has landed
    const int n4 = kBN / 4;
    for (int e = threadIdx.x; e < R_me * n4; e += blockDim.x) {
        const int rr = e / n4, c4 = e - rr * n4;
        const int64_t row = m0 + static_cast<int64_t>(me) * R + rr;
        const int64_t col = n0 + 4 * c4;
        if (row >= d_out || col >= d_in) continue;
        const float4* src = reinterpret_cast<const float4*>(slots + rr * kRowPad) + c4;
        float4 v = src[0];
        for (int z = 1; z < S; ++z) {
            const float4 w = src[z * R * (kRowPad / 4)];
            v.x += w.x;
            v.y += w.y;
            v.z += w.z;
            v.w += w.w;
        }
        float4 o = make_float4(scale * v.x, scale * v.y, scale * v.z, scale * v.w);
        float4* p = reinterpret_cast<float4*>(gW + row * d_in + col);  // d_in % 8 == 0
        if (accumulate) {
            const float4 a = *p;
            o = make_float4(a.x + o.x, a.y + o.y, a.z + o.z, a.w + o.w);
        }
        *p = o;
    }
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4f(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// The warp's TMEM lane quarter (32 accumulator rows) at taddr, columns
// [0, kBN), into shared memory at dst (this lane's row): 32 columns per load,
// or 8 in the 32-register build.
template <int FIT>
__device__ __forceinline__ void stage_rows(uint32_t taddr, uint32_t dst) {
    constexpr int W = FIT == 2 ? 8 : 32;
#pragma unroll 1
    for (int c = 0; c < kBN / W; ++c) {
        float v[W];
        if constexpr (W == 32)
            tc::tmem_ld_32x32(taddr + c * W, v);
        else
            tc::tmem_ld_32xN<W>(taddr + c * W, v);
#pragma unroll
        for (int u = 0; u < W / 4; ++u)
            st_shared_v4f(dst + 4u * (c * W + 4 * u), v[4 * u], v[4 * u + 1], v[4 * u + 2],
                          v[4 * u + 3]);
    }
}

static_assert(128 * kRowPad * 4 <= kReduceBytes &&
                  128 * kRowPad * 4 <= Cfg<2>::kStages * Cfg<2>::kStageBytes,
              "a 128-row accumulator fits in the stage buffers");

// The same reduction with each CTA's whole fp32 tile staged in its own shared
// memory (one row per lane, local stores) and the row blocks pulled: CTA d
// reads its rows from every CTA of the cluster, in slice order, with loads
// that run along the rows. A third cluster barrier keeps every tile in place
// until all its readers are done.
// One 128-row accumulator at a time: with MT = 2 the kernel calls it for the
// TMEM columns of each accumulator (tmem + 256 mt) and its rows (m0 + 128 mt).
// With FIT = 2 every warp stages its quarter, 8 columns at a time, and the
// slices' loads go one by one (the same sums in the same order).
template <int FIT>
__device__ void cluster_reduce_pull(unsigned char* smem, uint32_t tmem, bool ok, int64_t m0,
                                    int64_t n0, int64_t d_in, int64_t d_out,
                                    float* __restrict__ gW, float scale, bool accumulate) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = static_cast<int>(gridDim.z);
    const int R = (128 + S - 1) / S;  // rows summed by each CTA (the last may have fewer)
    const uint32_t me = cluster_rank();
    const int r0 = static_cast<int>(me) * R;
    const int R_me = (128 - r0 < R) ? 128 - r0 : R;
    float* tile = reinterpret_cast<float*>(smem);  // [128][kRowPad]
    cluster_sync_all();  // every CTA's main loop is over: its stage buffers are free
    if ((FIT == 2 || warp >= 2) && ok) {
        const int q = warp & 3;
        const uint32_t dst = tc::smem_u32(tile + (32 * q + lane) * kRowPad);
        stage_rows<FIT>(tmem + (static_cast<uint32_t>(32 * q) << 16), dst);
    }
    cluster_sync_all();  // every tile is in place
    const uint32_t base = tc::smem_u32(tile);
    const int n4 = kBN / 4;
    for (int e = threadIdx.x; e < R_me * n4; e += blockDim.x) {
        const int rr = e / n4, c4 = e - rr * n4;
        const int64_t row = m0 + r0 + rr;
        const int64_t col = n0 + 4 * c4;
        if (row >= d_out || col >= d_in) continue;
        const uint32_t a = base + 4u * static_cast<uint32_t>((r0 + rr) * kRowPad + 4 * c4);
        float4 v;
        if constexpr (FIT == 2) {
            v = ld_cluster_v4(map_to_rank(a, 0u));
#pragma unroll 1
            for (int z = 1; z < S; ++z) {
                const float4 w = ld_cluster_v4(map_to_rank(a, static_cast<uint32_t>(z)));
                v.x += w.x;
                v.y += w.y;
                v.z += w.z;
                v.w += w.w;
            }
        } else {
            // All S loads issued before the sums, which then run in slice order.
            float4 w[kMaxClusterSlices];
#pragma unroll
            for (int z = 0; z < kMaxClusterSlices; ++z)
                if (z < S) w[z] = ld_cluster_v4(map_to_rank(a, static_cast<uint32_t>(z)));
            v = w[0];
#pragma unroll
            for (int z = 1; z < kMaxClusterSlices; ++z) {
                if (z < S) {
                    v.x += w[z].x;
                    v.y += w[z].y;
                    v.z += w[z].z;
                    v.w += w[z].w;
                }
            }
        }
        float4 o = make_float4(scale * v.x, scale * v.y, scale * v.z, scale * v.w);
        float4* p = reinterpret_cast<float4*>(gW + row * d_in + col);  // d_in % 8 == 0
        if (accumulate) {
            const float4 a = *p;
            o = make_float4(a.x + o.x, a.y + o.y, a.z + o.z, a.w + o.w);
        }
        *p = o;
    }
    cluster_sync_all();  // no CTA leaves while another still reads its tile
}

// FIT (see threads_of): the builds that share an SM serve the multi-site
// lanes, where a contraction CTA runs beside weighting CTAs of later sites.
// Every build issues the same MMAs and sums in the same order: same results.
template <int MT, int FIT>
__global__ void __launch_bounds__(threads_of(FIT), min_ctas_of(FIT))
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              int64_t d_in, int64_t d_out, int64_t T, int64_t slice, float* __restrict__ out,
              float scale, int mode, unsigned int* __restrict__ status, int stall) {
    using C = Cfg<MT>;
    constexpr int kBM = C::kBM, kStages = C::kStages, kABytes = C::kABytes;
    constexpr int kStageBytes = C::kStageBytes;
    constexpr uint32_t kTmemCols = C::kTmemCols;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Ctl<MT>* ctl = reinterpret_cast<Ctl<MT>*>(smem + kStages * kStageBytes);

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
                for (int mt = 0; mt < MT; ++mt) {
                    const uint64_t ad =
                        tc::sdesc_sw128(a + 2 * mt * kBoxBytes + kk * 2048, kBoxBytes, 1024);
                    tc::mma_bf16(tmem + mt * kBN, ad, bd, kIdesc, (it | kk) != 0 ? 1u : 0u);
                }
            }
            tc::mma_commit(&ctl->empty[st]);
        }
        ctl->consumed = it;
        tc::mma_commit(&ctl->done);
    }
    if (FIT == 2) __syncwarp();  // warps 0 and 1 regroup after their roles
    if (FIT == 2 || warp >= 2) {
        const bool ok = tc::mbar_wait(&ctl->done, 0);
        tc::tc_fence_after();
        if (!ok) *abort_flag = 1;
        if (ok && !*abort_flag && n_k > 0 && mode < 3) {
            const int q = warp & 3;  // TMEM lane quarter this warp may access
            // The warp's 32 accumulator rows go through the idle stage buffers
            // (one row per lane in, then rows out with consecutive lanes on
            // consecutive columns), so each store instruction covers 512
            // contiguous bytes of a row: also where GW is host memory mapped
            // into the device, which takes scattered 16-byte writes slowly.
            float* rows = reinterpret_cast<float*>(smem) + q * 32 * kRowPad;
            const uint32_t rows_s = tc::smem_u32(rows) + 4u * static_cast<uint32_t>(lane * kRowPad);
#pragma unroll 1
            for (int mt = 0; mt < MT; ++mt) {
                stage_rows<FIT>(tmem + (static_cast<uint32_t>(32 * q) << 16) + mt * kBN, rows_s);
                __syncwarp();
#pragma unroll 1
                for (int rr = 0; rr < 32; ++rr) {
                    const int64_t row = m0 + 128 * mt + 32 * q + rr;
                    if (row >= d_out) break;
                    float* dst = (mode == 0)
                                     ? out + (static_cast<int64_t>(blockIdx.z) * d_out + row) * d_in
                                     : out + row * d_in;
#pragma unroll
                    for (int c4 = lane; c4 < kBN / 4; c4 += 32) {
                        const int64_t col = n0 + 4 * c4;
                        if (col >= d_in) break;  // d_in % 8 == 0: the float4 is whole
                        const float4 w4 = *reinterpret_cast<const float4*>(rows + rr * kRowPad + 4 * c4);
                        float4* p = reinterpret_cast<float4*>(dst + col);
                        if (mode == 0) {
                            *p = w4;
                        } else if (mode == 1) {
                            *p = make_float4(scale * w4.x, scale * w4.y, scale * w4.z,
                                             scale * w4.w);
                        } else {
                            const float4 o = *p;
                            *p = make_float4(o.x + scale * w4.x, o.y + scale * w4.y,
                                             o.z + scale * w4.z, o.w + scale * w4.w);
                        }
                    }
                }
                __syncwarp();  // the rows are read before the next accumulator's land
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
    if (mode >= 3) {
        __syncthreads();
        if (kPull || MT > 1 || FIT == 2) {
#pragma unroll 1
            for (int mt = 0; mt < MT; ++mt)
                cluster_reduce_pull<FIT>(smem, tmem + mt * kBN, !*abort_flag && n_k > 0, m0 + 128 * mt,
                                    n0, d_in, d_out, out, scale, mode == 4);
        } else {
            cluster_reduce(smem, tmem, !*abort_flag && n_k > 0, m0, n0, d_in, d_out, out, scale,
                           mode == 4);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}


// Token slices per output tile for tiles of `bm` channels: enough CTAs to
// give every SM one tile slice (S = 152 / tiles), each slice at least 4
// k-steps. More slices than that measured slower even where they would fill
// the GPU better (qkv 1024 x 3072, 96 tiles: 3 slices in 2 waves 131 us
// against 102 us for 1 slice): the CTAs then share one tile feed.
int64_t slices_for(int64_t T, int64_t d_in, int64_t d_out, int64_t bm) {
    const int64_t tiles = ((d_out + bm - 1) / bm) * ((d_in + kBN - 1) / kBN);
    int64_t S = 152 / tiles;
    const int64_t max_s = (T + 4 * kBK - 1) / (4 * kBK);  // at least 4 k-steps per slice
    if (S > max_s) S = max_s;
    return S < 1 ? 1 : S;
}

// Channels per tile: 256 (two accumulators) when every token slice of the
// larger tile keeps at least DUST_GEMM_MT2_MIN_SLICE tokens and there are at
// least 8 such tiles, else 128. Measured (contraction alone, us, 128 -> 256
// rows): 4096^2 over 32,768 tokens 781 -> 623; 1024 x 3072 over 16,384
// 104 -> 77; the sweep's 512 -> 2048 and 2048 -> 512 over 65,536 112 -> 101,
// 512 -> 1536 90 -> 86; but 512 -> 512 over 65,536 (4 larger tiles) 49.5 ->
// 50.5 and 512 -> 2048 over 16,384 (slices of 1,820 tokens) 42.6 -> 44:
// there the slices' partials and their reduction outweigh the faster feed.
int tile_mt(int64_t T, int64_t d_in, int64_t d_out) {
    if (DUST_GEMM_MT2_MIN_SLICE <= 0) return 1;
    const int64_t tiles2 = ((d_out + 255) / 256) * ((d_in + kBN - 1) / kBN);
    if (tiles2 < 8) return 1;
    const int64_t S = slices_for(T, d_in, d_out, 256);
    return (T / S >= DUST_GEMM_MT2_MIN_SLICE) ? 2 : 1;
}

int64_t tc_slices(int64_t T, int64_t d_in, int64_t d_out) {
    return slices_for(T, d_in, d_out, 128 * tile_mt(T, d_in, d_out));
}

}  // namespace

// The driver entry point that encodes tensor maps (nullptr if unavailable).
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


namespace {

// True when all `tiles` clusters of S CTAs can be resident at once. Clusters
// must fit inside one GPC, so a cluster size that does not divide the GPCs'
// SM counts leaves SMs unused and can push a few clusters into a second
// wave; the fp32 partials then win (measured on the 48-site sweep: 6-CTA
// clusters 5.1 ms of contraction against 4.3 ms with partials).
template <int MT, int FIT>
bool cluster_fits(int S, int64_t tiles) {
    constexpr int kMaxDev = 64;
    static int max_active[kMaxDev][kMaxClusterSlices + 1] = {};
    static std::once_flag once[kMaxDev][kMaxClusterSlices + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    std::call_once(once[dev][S], [S, dev] {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, static_cast<unsigned>(S));
        cfg.blockDim = dim3(threads_of(FIT));
        cfg.dynamicSmemBytes = Cfg<MT>::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = static_cast<unsigned>(S);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (ensure_smem_limit(reinterpret_cast<const void*>(k_gemm_tc<MT, FIT>),
                              Cfg<MT>::kSmemBytes) != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<MT, FIT>, &cfg) != cudaSuccess)
            n = 0;
        (void)cudaGetLastError();
        max_active[dev][S] = n;
    });
    return tiles <= max_active[dev][S];
}

// With `back` given, the contraction kernel ran on a stream of its own: `back`
// (the caller's stream) waits for it, and the slice reduction, if any, runs on
// `back` (at that stream's priority, not the contraction's).
cudaError_t hand_back(cudaStream_t s, cudaStream_t back, cudaEvent_t back_ev) {
    if (!back) return cudaSuccess;
    cudaError_t e = cudaEventRecord(back_ev, s);
    return e != cudaSuccess ? e : cudaStreamWaitEvent(back, back_ev, 0);
}

template <int MT, int FIT>
cudaError_t launch_mt(const CUtensorMap& ta, const CUtensorMap& tb, int64_t T, int64_t d_in,
                      int64_t d_out, float scale, bool accumulate, float* gW, float* partials,
                      cudaStream_t s, cudaStream_t back, cudaEvent_t back_ev) {
    using C = Cfg<MT>;
    const cudaError_t attr_err =
        ensure_smem_limit(reinterpret_cast<const void*>(k_gemm_tc<MT, FIT>), C::kSmemBytes);
    if (attr_err != cudaSuccess) return attr_err;
    unsigned int* st = status_word();
    if (!st) return cudaErrorUnknown;
    const int64_t S = slices_for(T, d_in, d_out, C::kBM);
    int64_t slice = (T + S - 1) / S;
    slice = (slice + kBK - 1) / kBK * kBK;
    const int64_t S_used = (T + slice - 1) / slice;
    dim3 grid(static_cast<unsigned>((d_in + kBN - 1) / kBN),
              static_cast<unsigned>((d_out + C::kBM - 1) / C::kBM), static_cast<unsigned>(S_used));
    cudaError_t e;
    const int stall = take_stall_injection() ? 1 : 0;
    if (kClusterReduce && S_used >= 2 && S_used <= kMaxClusterSlices &&
        cluster_fits<MT, FIT>(static_cast<int>(S_used),
                               static_cast<int64_t>(grid.x) * grid.y)) {
        // The slices of a tile reduce through distributed shared memory.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(threads_of(FIT));
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = static_cast<unsigned>(S_used);
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = DUST_PDL ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        {
            ProfScope ps(kStageGemmTc, s);
            e = cudaLaunchKernelEx(&cfg, k_gemm_tc<MT, FIT>, ta, tb, d_in, d_out, T, slice, gW,
                                   scale, accumulate ? 4 : 3, st, stall);
        }
        if (e == cudaSuccess) return hand_back(s, back, back_ev);
        (void)cudaGetLastError();  // clusters refused: fall back to partials + reduction
    }
    const int mode = (S_used > 1) ? 0 : (accumulate ? 2 : 1);
    {
        ProfScope ps(kStageGemmTc, s);
        e = launch_pdl(k_gemm_tc<MT, FIT>, grid, dim3(threads_of(FIT)), C::kSmemBytes, s, ta, tb,
                       d_in, d_out, T, slice, S_used > 1 ? partials : gW, scale, mode, st, stall);
    }
    if (e != cudaSuccess) return e;
    e = hand_back(s, back, back_ev);
    if (e != cudaSuccess || S_used == 1) return e;
    return launch_reduce(partials, S_used, d_out * d_in, scale, accumulate, gW, back ? back : s);
}

}  // namespace

cudaError_t launch_tc_gemm(const void* g, const void* X, int64_t T, int64_t d_in, int64_t d_out,
                           float scale, bool accumulate, float* gW, float* partials,
                           cudaStream_t s, int fit, cudaStream_t back, cudaEvent_t back_ev) {
    CUtensorMap ta, tb;
    if (!make_tmap_bf16(&ta, g, T, d_out, kBK) || !make_tmap_bf16(&tb, X, T, d_in, kBK))
        return cudaErrorInvalidValue;
    const bool mt2 = tile_mt(T, d_in, d_out) == 2;
    auto go = [&](auto k1, auto k2) {
        return mt2 ? k2(ta, tb, T, d_in, d_out, scale, accumulate, gW, partials, s, back, back_ev)
                   : k1(ta, tb, T, d_in, d_out, scale, accumulate, gW, partials, s, back, back_ev);
    };
    if (fit == 2) return go(launch_mt<1, 2>, launch_mt<2, 2>);
    if (fit == 1) return go(launch_mt<1, 1>, launch_mt<2, 1>);
    return go(launch_mt<1, 0>, launch_mt<2, 0>);
}

}  // namespace dust
