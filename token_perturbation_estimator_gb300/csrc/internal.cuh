// Internal launch interfaces shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

#include "dust.h"

namespace dust {

// Device address of the status word that kernels with bounded waits set when
// a wait runs out (0 = ok, otherwise a dust_status value). Looked up once per
// device; read and cleared by dust_last_error. nullptr if the lookup failed.
unsigned int* status_word();

// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` on the
// current device. The attribute belongs to the device, so it is set once
// per (kernel, device), under a lock, for processes that use several GPUs.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

// Asks for the largest shared-memory carveout for `kernel` on the current
// device (set once per (kernel, device)). The estimator's small-footprint
// kernels (scan, weighting, slice reduction) then leave SMs configured so
// that a contraction CTA (about 193 KB of shared memory) can become resident
// beside them: under the default preference an SM running them keeps most of
// its unified memory as L1, and the contraction waits for the SM to drain.
cudaError_t ensure_shared_carveout(const void* kernel);

// Kernel families timed by dust_profile_read.
enum Stage {
    kStageScanLocal, kStageScanCarry, kStageScanFixup, kStageWeight, kStageGemmSimt,
    kStageReduce, kStageGemmTc, kStageFused, kStageNoise, kStageJitter, kStageZero, kStageScore,
    kStageScatter, kStageForward, kStageCount
};

// Brackets the launches issued during its lifetime with profiling events
// (no-op unless profiling is enabled).
struct ProfScope {
    ProfScope(int stage, cudaStream_t s);
    ~ProfScope();
    ProfScope(const ProfScope&) = delete;
    ProfScope& operator=(const ProfScope&) = delete;
    int stage;
    cudaStream_t s;
    int slot;
};

// Test hook: true once after dust_debug_inject_timeout(1); the next
// tensor-core contraction then makes its bounded wait run out.
bool take_stall_injection();
bool stall_injection_pending();
// True while dust_profile_enable(1) is in effect.
bool profiling_on();

// Runs `enqueue` on `stream`, or replays it as a CUDA graph: the second call
// with byte-identical `key` (every argument of the call, pointers included)
// captures what `enqueue` issues into a graph on an internal stream, and
// later calls with that key launch the graph on `stream`. Graphs read and
// write the same addresses, so they see the current contents of every
// buffer. Bypassed while profiling or a test stall is pending; a call that
// cannot be captured falls back to direct launches for that key. With
// `node_priority` the graph keeps the priority of the stream each kernel was
// captured from (for work that spans internal streams of different
// priority); otherwise every kernel runs at the priority of `stream`.
dust_status graph_call(const void* key, size_t key_len, cudaStream_t stream,
                       dust_status (*enqueue)(const void* ctx, cudaStream_t s), const void* ctx,
                       bool node_priority = false);

// ---- Programmatic dependent launch. The estimator's kernels are launched so
// that the next kernel on the stream may be scheduled while the previous one
// drains (its prologue then overlaps the tail). Each such kernel calls
// pdl_wait() before its first global memory access: griddepcontrol.wait
// returns once every prerequisite grid has completed and its writes are
// visible (at once when there is none), so stream order holds for all data.
// pdl_trigger(), called right after the wait, lets the next kernel be
// scheduled once every CTA of this one is past its own wait.
#ifndef DUST_PDL
#define DUST_PDL 1
#endif

__device__ __forceinline__ void pdl_wait() {
#if DUST_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

__device__ __forceinline__ void pdl_trigger() {
#if DUST_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = DUST_PDL ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_pdl for the estimator's small-footprint kernels: with the largest
// shared-memory carveout (ensure_shared_carveout).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_shared(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
    const cudaError_t e = ensure_shared_carveout(reinterpret_cast<const void*>(kernel));
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, grid, block, smem, s, static_cast<Args&&>(args)...);
}

// Token chunk of the credit scan (one CTA, 32 lanes x 8 tokens).
constexpr int kScanChunk = 256;


// Workspace of the credit scan. All pointers are device memory.
struct ScanBuffers {
    float* r;       // [T][K] local (chunk) scan, or final after fix-up
    float* P;       // [T] product of the decay from t to its chunk's end
    float* A;       // [n_chunks][K] chunk summary: local r at the chunk start
    float* B;       // [n_chunks][2] chunk summary: decay product over the chunk, hi + lo
    float* carry;   // [n_chunks][K] true r at the first token after the chunk
    int64_t n_chunks;
};

size_t scan_workspace_bytes(int64_t K, int64_t T);
ScanBuffers scan_carve(void* ws, int64_t K, int64_t T);

cudaError_t launch_noise(void* out, int out_kind /*0 f32, 1 bf16, 2 u32*/, uint64_t seed,
                         int kind, int64_t draw_begin, int64_t n_draws, int64_t T,
                         int64_t d_out, uint32_t flags, cudaStream_t s);
cudaError_t launch_jitter(void* y, int y_bf16, int64_t ld_y, int64_t T, int64_t d_out,
                          uint64_t seed, int kind, int64_t draw, float sigma, uint32_t flags,
                          cudaStream_t s);
// Jittered forward (k_forward.cu): Y[s] = X W^T (s < clean) and
// X W^T + sigma a^(draw_begin + s - clean); bf16 X [T][d_in], W [d_out][d_in],
// Y [clean + n_draws][T][d_out]; d_in, d_out multiples of 8, 16-byte aligned.
cudaError_t launch_forward(const void* X, const void* W, int64_t T, int64_t d_in, int64_t d_out,
                           uint64_t seed, int kind, int64_t draw_begin, int64_t n_draws,
                           float sigma, bool anti, int clean, void* Y, cudaStream_t s);

// Centring + chunk-local scan + chunk carries. After it, r holds chunk-local
// values; the true r is r[t][i] + P[t] * carry[t / kScanChunk][i].
// With `ticket` (a zeroed device word) the carry pass runs in the scan
// kernel's last CTA when the summaries fit; otherwise as a second kernel.
cudaError_t launch_scan(const float* delta, int64_t K, int64_t T, const int32_t* seq_offsets,
                        int64_t n_seq, float gamma, bool center, const ScanBuffers& b,
                        cudaStream_t s, unsigned int* ticket = nullptr);
cudaError_t launch_scan_fixup(const ScanBuffers& b, int64_t K, int64_t T, cudaStream_t s);

// g[t][c] = coef * sum_i r[t][i] a_t^(draw_begin+i)[c]; with `fix` the scan
// fix-up is applied while staging r.
// Rewards from the scan buffers (b.r, plus P and carry when fix), or, when
// delta is given, straight from the loss changes Delta [K][T] (gamma = 0, where
// the scan is the identity), centred over the draws when center.
cudaError_t launch_weight(const ScanBuffers& b, bool fix, int64_t K, int64_t T, int64_t d_out,
                          uint64_t seed, int kind, int64_t draw_begin, float coef,
                          bool anti, void* g, int g_bf16, cudaStream_t s,
                          const float* delta = nullptr, bool center = false);

// CUDA-core contraction: partial[s][c][j] = sum_{t in slice s} g[t][c] x[t][j]
// followed by gW = scale * sum_s partial (+ gW).
size_t simt_gemm_workspace_bytes(int64_t T, int64_t d_in, int64_t d_out);
cudaError_t launch_simt_gemm(const void* g, int g_bf16, const void* X, int x_bf16, int64_t T,
                             int64_t d_in, int64_t d_out, float scale, bool accumulate,
                             float* gW, float* partials, cudaStream_t s);

// gW[q] = scale * sum_{s<S} partials[s][q] (+ gW[q] when accumulating), in
// slice order (deterministic).
cudaError_t launch_reduce(const float* partials, int64_t S, int64_t n, float scale,
                          bool accumulate, float* gW, cudaStream_t s);

// Tensor-core contraction (tcgen05, bf16 g and X, fp32 accumulate). `fit`
// picks the build by what shares its SMs: 0 alone (192 threads), 1 beside
// four weighting CTAs (192 threads, at most 80 registers), 2 beside five
// (128 threads, at most 32 registers); for sites that run concurrently.
// With `back` given, the kernel runs on `s` (a stream of high priority) and
// `back` then waits for it (through `back_ev`) and runs the slice reduction.
bool tc_gemm_supported(const void* g, const void* X, int64_t d_in, int64_t d_out);
size_t tc_gemm_workspace_bytes(int64_t T, int64_t d_in, int64_t d_out);
cudaError_t launch_tc_gemm(const void* g, const void* X, int64_t T, int64_t d_in, int64_t d_out,
                           float scale, bool accumulate, float* gW, float* partials,
                           cudaStream_t s, int fit = 0, cudaStream_t back = nullptr,
                           cudaEvent_t back_ev = nullptr);

// Bytes of per-call synchronisation words (the scan's ticket) at the head of
// a workspace; zeroed by one cudaMemsetAsync per call.
constexpr size_t kSyncBytes = 4096;

// Fused weighting + tensor-core contraction (d_in <= 512): g tiles are made
// in shared memory and never written to HBM.
bool fused_supported(int64_t d_in, int64_t d_out, int64_t K);
size_t fused_workspace_bytes(int64_t T, int64_t d_in, int64_t d_out);
cudaError_t launch_fused(const ScanBuffers& b, const void* X, int64_t K, int64_t T, int64_t d_in,
                         int64_t d_out, uint64_t seed, int kind, int64_t draw_begin, float coef,
                         bool anti, float scale, bool accumulate, float* gW, float* partials,
                         cudaStream_t s);

// delta[k][t] = <g[t], dO[k][t]> (local scores as loss changes), rows of d.
cudaError_t launch_local_score(const void* g, int g_bf16, const void* dO, int o_bf16, int64_t K,
                               int64_t T, int64_t d, float* out, cudaStream_t s);

// Embedding reassembly gE[v] = scale * sum over tokens with id v of g[t]
// (deterministic 64-bit fixed-point accumulation, k_scatter.cu); the
// workspace (256-byte aligned, scatter_workspace_bytes) is cleared here.
size_t scatter_workspace_bytes(int64_t T, int64_t V, int64_t d);
cudaError_t launch_scatter_gE(const void* g, int g_bf16, const int32_t* ids, int64_t T,
                              int64_t d, int64_t V, float scale, bool accumulate, float* gE,
                              void* workspace, cudaStream_t s);

// Fill gW with zeros (T == 0) unless accumulating.
cudaError_t launch_zero(float* p, int64_t n, cudaStream_t s);

}  // namespace dust
