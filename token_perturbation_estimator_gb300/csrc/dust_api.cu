// C ABI (include/dust.h): argument validation, workspace layout and dispatch.
// Everything is enqueued on the caller's stream (dust_estimate_gW_host also
// copies X on an internal stream and joins back); nothing here allocates
// device memory or synchronises, except dust_last_error.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "dust.h"
#include "internal.cuh"

using namespace dust;

namespace {

constexpr uint32_t kKnownFlags = DUST_CENTER | DUST_ANTITHETIC | DUST_ACCUMULATE |
                                 DUST_FORCE_UNFUSED | DUST_FORCE_FUSED | DUST_WORD_STREAM1 |
                                 DUST_FORCE_SIMT;

size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// With gamma = 0 and at most this many draws the weighting kernel reads the
// loss changes itself (one staging group) and no scan kernel runs.
constexpr int64_t kDirectMaxDraws = 32;

bool finite(float x) { return std::isfinite(x); }

int popcount3(uint32_t f) {
    return ((f & DUST_FORCE_UNFUSED) ? 1 : 0) + ((f & DUST_FORCE_FUSED) ? 1 : 0) +
           ((f & DUST_FORCE_SIMT) ? 1 : 0);
}

dust_status counter_ok(int64_t T, int64_t d_out) {
    if (T < 0 || d_out < 0) return DUST_ERR_INVALID_ARG;
    if (d_out > 0 && T > DUST_MAX_COUNTER / d_out) return DUST_ERR_RANGE;
    return DUST_OK;
}

dust_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DUST_OK : DUST_ERR_CUDA; }

// Noise kinds that give jitter values (all but the raw words).
bool value_kind(int kind) {
    return kind == DUST_NOISE_RADEMACHER || kind == DUST_NOISE_GAUSSIAN ||
           kind == DUST_NOISE_RADEMACHER_PACKED;
}

// Shape/flag validation shared by the estimator entry points.
dust_status check_estimate(int64_t T, int64_t d_in, int64_t d_out, int64_t K, dust_dtype x_dtype,
                           uint32_t flags) {
    if (T < 0 || d_in < 0 || d_out < 0) return DUST_ERR_INVALID_ARG;
    if (K < 1) return DUST_ERR_INVALID_ARG;
    if (K > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (flags & ~kKnownFlags) return DUST_ERR_INVALID_ARG;
    if (flags & DUST_WORD_STREAM1) return DUST_ERR_INVALID_ARG;
    if (popcount3(flags) > 1) return DUST_ERR_INVALID_ARG;
    if ((flags & DUST_ANTITHETIC) && (K & 1)) return DUST_ERR_INVALID_ARG;
    dust_status st = counter_ok(T, d_out);
    if (st != DUST_OK) return st;
    if (T > 0 && d_in > 0 && T > (int64_t(1) << 40) / d_in) return DUST_ERR_RANGE;
    return DUST_OK;
}

int choose_path(int64_t T, int64_t d_in, int64_t d_out, int64_t K, dust_dtype x_dtype,
                uint32_t flags) {
    (void)T;
    (void)K;
    const bool forced_tc = (flags & (DUST_FORCE_UNFUSED | DUST_FORCE_FUSED)) != 0;
    if (x_dtype != DUST_BF16) return forced_tc ? -DUST_ERR_UNSUPPORTED : DUST_PATH_SIMT;
    if (flags & DUST_FORCE_SIMT) return DUST_PATH_SIMT;
    const bool tc_shape = (d_in % 8 == 0) && (d_out % 8 == 0) && d_in > 0 && d_out > 0;
    if (!tc_shape) return forced_tc ? -DUST_ERR_UNSUPPORTED : DUST_PATH_SIMT;
    // The fused kernel is opt-in: on GB300 it is limited to one 1024-thread
    // CTA per SM (its TMEM accumulator spans the SM), too few warps to hide
    // the producers' latencies, and measures slower than the weighting
    // kernel followed by the tensor-core GEMM.
    if (flags & DUST_FORCE_FUSED)
        return fused_supported(d_in, d_out, K) ? DUST_PATH_FUSED_TC : -DUST_ERR_UNSUPPORTED;
    return DUST_PATH_UNFUSED_TC;
}

struct Layout {
    size_t sync = kSyncBytes, scan = 0, g = 0, gemm = 0, total = 0;
    int path = DUST_PATH_SIMT;
    int g_bf16 = 0;
};

// Workspace: scan buffers, then g [T][d_out] (bf16 when X is bf16, else
// fp32), then the contraction's split-token partials. Sized for the chosen
// path (the fused path needs no g buffer).
Layout layout(int64_t T, int64_t d_in, int64_t d_out, int64_t K, dust_dtype x_dtype,
              uint32_t flags) {
    Layout L;
    L.path = choose_path(T, d_in, d_out, K, x_dtype, flags);
    L.scan = a256(scan_workspace_bytes(K, T));
    L.g_bf16 = (x_dtype == DUST_BF16) ? 1 : 0;
    if (L.path == DUST_PATH_FUSED_TC) {
        L.g = 0;
        L.gemm = a256(fused_workspace_bytes(T, d_in, d_out));
        L.total = L.sync + L.scan + L.gemm;
        return L;
    }
    L.g = a256(static_cast<size_t>(T) * static_cast<size_t>(d_out) * (L.g_bf16 ? 2 : 4));
    size_t gemm = simt_gemm_workspace_bytes(T, d_in, d_out);
    if (L.path == DUST_PATH_UNFUSED_TC) {
        const size_t tcb = tc_gemm_workspace_bytes(T, d_in, d_out);
        if (tcb > gemm) gemm = tcb;
    }
    L.gemm = a256(gemm);
    L.total = L.sync + L.scan + L.g + L.gemm;
    return L;
}

}  // namespace

extern "C" {

const char* dust_status_string(dust_status s) {
    switch (s) {
        case DUST_OK: return "DUST_OK";
        case DUST_ERR_INVALID_ARG: return "DUST_ERR_INVALID_ARG: invalid argument";
        case DUST_ERR_RANGE: return "DUST_ERR_RANGE: size beyond a documented limit";
        case DUST_ERR_UNSUPPORTED: return "DUST_ERR_UNSUPPORTED: not supported by this build";
        case DUST_ERR_CUDA: return "DUST_ERR_CUDA: a CUDA call or launch failed";
        case DUST_ERR_TIMEOUT: return "DUST_ERR_TIMEOUT: a device-side bounded wait ran out";
        case DUST_ERR_WORKSPACE: return "DUST_ERR_WORKSPACE: workspace missing, small or misaligned";
    }
    return "unknown dust_status";
}

int32_t dust_version(void) { return 100; }

dust_status dust_noise(void* out, dust_dtype out_dtype, uint64_t seed, dust_noise_kind kind,
                       int64_t draw_begin, int64_t n_draws, int64_t T, int64_t d_out,
                       uint32_t flags, void* stream) {
    if (draw_begin < 0 || n_draws < 0) return DUST_ERR_INVALID_ARG;
    if (n_draws > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    dust_status st = counter_ok(T, d_out);
    if (st != DUST_OK) return st;
    if (flags & ~(DUST_ANTITHETIC | DUST_WORD_STREAM1)) return DUST_ERR_INVALID_ARG;
    int out_kind;
    if (kind == DUST_NOISE_RAW_WORDS) {
        if (out_dtype != DUST_U32) return DUST_ERR_INVALID_ARG;
        out_kind = 2;
    } else if (value_kind(kind)) {
        if (out_dtype == DUST_F32) out_kind = 0;
        else if (out_dtype == DUST_BF16) out_kind = 1;
        else return DUST_ERR_INVALID_ARG;
        if (flags & DUST_WORD_STREAM1) return DUST_ERR_INVALID_ARG;
    } else {
        return DUST_ERR_INVALID_ARG;
    }
    if (draw_begin > (int64_t(1) << 31) - n_draws) return DUST_ERR_RANGE;
    if (n_draws * T * d_out == 0) return DUST_OK;
    if (!out) return DUST_ERR_INVALID_ARG;
    return cuda_status(launch_noise(out, out_kind, seed, static_cast<int>(kind), draw_begin,
                                    n_draws, T, d_out, flags,
                                    static_cast<cudaStream_t>(stream)));
}

dust_status dust_jitter_apply(void* y, dust_dtype y_dtype, int64_t ld_y, int64_t T,
                              int64_t d_out, uint64_t seed, dust_noise_kind kind, int64_t draw,
                              float sigma, uint32_t flags, void* stream) {
    dust_status st = counter_ok(T, d_out);
    if (st != DUST_OK) return st;
    if (ld_y < d_out || draw < 0) return DUST_ERR_INVALID_ARG;
    if (draw >= (int64_t(1) << 31)) return DUST_ERR_RANGE;
    if (!value_kind(kind)) return DUST_ERR_INVALID_ARG;
    if (y_dtype != DUST_F32 && y_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (flags & ~DUST_ANTITHETIC) return DUST_ERR_INVALID_ARG;
    if (!finite(sigma)) return DUST_ERR_INVALID_ARG;
    if (T * d_out == 0) return DUST_OK;
    if (!y) return DUST_ERR_INVALID_ARG;
    return cuda_status(launch_jitter(y, y_dtype == DUST_BF16, ld_y, T, d_out, seed,
                                     static_cast<int>(kind), draw, sigma, flags,
                                     static_cast<cudaStream_t>(stream)));
}

dust_status dust_forward_jitter(const void* X, const void* W, int64_t T, int64_t d_in,
                                int64_t d_out, uint64_t seed, dust_noise_kind kind,
                                int64_t draw_begin, int64_t n_draws, float sigma,
                                uint32_t flags, int32_t clean, void* Y, void* stream) {
    if (T < 0 || d_in < 0 || d_out < 0 || draw_begin < 0 || n_draws < 0) return DUST_ERR_INVALID_ARG;
    if (clean != 0 && clean != 1) return DUST_ERR_INVALID_ARG;
    if (!value_kind(kind)) return DUST_ERR_INVALID_ARG;
    if (flags & ~DUST_ANTITHETIC) return DUST_ERR_INVALID_ARG;
    if (!finite(sigma)) return DUST_ERR_INVALID_ARG;
    if (n_draws > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    if (draw_begin > (int64_t(1) << 31) - n_draws) return DUST_ERR_RANGE;
    dust_status st = counter_ok(T, d_out);
    if (st != DUST_OK) return st;
    if (d_in == 0 || d_in % 8 != 0 || d_out % 8 != 0) return DUST_ERR_UNSUPPORTED;
    if (T * d_out * (clean + n_draws) == 0) return DUST_OK;
    if (!X || !W || !Y) return DUST_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W) |
         reinterpret_cast<uintptr_t>(Y)) % 16 != 0)
        return DUST_ERR_UNSUPPORTED;
    return cuda_status(launch_forward(X, W, T, d_in, d_out, seed, static_cast<int>(kind),
                                      draw_begin, n_draws, sigma, (flags & DUST_ANTITHETIC) != 0,
                                      clean, Y, static_cast<cudaStream_t>(stream)));
}

dust_status dust_local_score(const void* g, dust_dtype g_dtype, const void* delta_o,
                             dust_dtype o_dtype, int64_t K, int64_t T, int64_t d,
                             float* delta, void* stream) {
    if (K < 0 || T < 0 || d < 0) return DUST_ERR_INVALID_ARG;
    if ((g_dtype != DUST_F32 && g_dtype != DUST_BF16) ||
        (o_dtype != DUST_F32 && o_dtype != DUST_BF16))
        return DUST_ERR_INVALID_ARG;
    if (K * T == 0) return DUST_OK;
    if (!delta || (d > 0 && (!g || !delta_o))) return DUST_ERR_INVALID_ARG;
    return cuda_status(launch_local_score(g, g_dtype == DUST_BF16, delta_o, o_dtype == DUST_BF16,
                                          K, T, d, delta, static_cast<cudaStream_t>(stream)));
}

dust_status dust_scatter_gE_workspace(size_t* bytes, int64_t T, int64_t V, int64_t d) {
    if (!bytes || T < 0 || V < 0 || d < 0) return DUST_ERR_INVALID_ARG;
    *bytes = a256(scatter_workspace_bytes(T, V, d));
    return DUST_OK;
}

dust_status dust_scatter_gE(const void* g, dust_dtype g_dtype, const int32_t* ids, int64_t T,
                            int64_t d, int64_t V, float scale, uint32_t flags, float* gE,
                            void* workspace, size_t ws_bytes, void* stream) {
    if (T < 0 || d < 0 || V < 0) return DUST_ERR_INVALID_ARG;
    if (g_dtype != DUST_F32 && g_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (flags & ~DUST_ACCUMULATE) return DUST_ERR_INVALID_ARG;
    if (!finite(scale)) return DUST_ERR_INVALID_ARG;
    if (T > 0 && (T > (int64_t(1) << 31) - 1 || (d > 0 && T > (int64_t(1) << 40) / d)))
        return DUST_ERR_RANGE;
    if (V * d == 0) return DUST_OK;
    if (!gE) return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool acc = (flags & DUST_ACCUMULATE) != 0;
    if (T == 0) return acc ? DUST_OK : cuda_status(launch_zero(gE, V * d, s));
    if (!g || !ids) return DUST_ERR_INVALID_ARG;
    size_t need = 0;
    dust_scatter_gE_workspace(&need, T, V, d);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return DUST_ERR_WORKSPACE;
    return cuda_status(launch_scatter_gE(g, g_dtype == DUST_BF16, ids, T, d, V, scale, acc, gE,
                                         workspace, s));
}

dust_status dust_estimate_gE_workspace(size_t* bytes, int64_t T, int64_t d, int64_t V,
                                       int64_t K) {
    if (!bytes || T < 0 || d < 0 || V < 0 || K < 1) return DUST_ERR_INVALID_ARG;
    if (K > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    *bytes = kSyncBytes + a256(scan_workspace_bytes(K, T)) +
             a256(sizeof(float) * static_cast<size_t>(T) * static_cast<size_t>(d)) +
             a256(scatter_workspace_bytes(T, V, d));
    return DUST_OK;
}

dust_status dust_estimate_gE(const int32_t* ids, int64_t T, int64_t V, const float* delta,
                             int64_t K, int64_t d, const int32_t* seq_offsets, int64_t n_seq,
                             uint64_t seed, dust_noise_kind kind, int64_t draw_begin,
                             float sigma, float gamma, float scale, uint32_t flags, float* gE,
                             void* workspace, size_t ws_bytes, void* stream) {
    if (T < 0 || V < 0 || d < 0 || K < 1) return DUST_ERR_INVALID_ARG;
    if (K > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    if (flags & ~(DUST_CENTER | DUST_ANTITHETIC | DUST_ACCUMULATE)) return DUST_ERR_INVALID_ARG;
    if (!value_kind(kind)) return DUST_ERR_INVALID_ARG;
    if (draw_begin < 0) return DUST_ERR_INVALID_ARG;
    if (draw_begin > (int64_t(1) << 31) - K) return DUST_ERR_RANGE;
    if ((flags & DUST_ANTITHETIC) && ((K & 1) || (draw_begin & 1))) return DUST_ERR_INVALID_ARG;
    if (!finite(sigma) || sigma == 0.0f) return DUST_ERR_INVALID_ARG;
    if (!finite(gamma) || std::fabs(gamma) > 1.0f || !finite(scale)) return DUST_ERR_INVALID_ARG;
    dust_status st = counter_ok(T, d);
    if (st != DUST_OK) return st;
    if (T > 0 && (n_seq < 1 || n_seq > T)) return DUST_ERR_INVALID_ARG;
    if (V * d == 0) return DUST_OK;
    if (!gE) return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool acc = (flags & DUST_ACCUMULATE) != 0;
    if (T == 0) return acc ? DUST_OK : cuda_status(launch_zero(gE, V * d, s));
    if (!ids || !delta || !seq_offsets) return DUST_ERR_INVALID_ARG;
    size_t need = 0;
    dust_estimate_gE_workspace(&need, T, d, V, K);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return DUST_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    unsigned int* sync = reinterpret_cast<unsigned int*>(ws);
    ws += kSyncBytes;
    ScanBuffers b = scan_carve(ws, K, T);
    ws += a256(scan_workspace_bytes(K, T));
    float* g = reinterpret_cast<float*>(ws);
    ws += a256(sizeof(float) * static_cast<size_t>(T) * static_cast<size_t>(d));
    const float coef = static_cast<float>(-1.0 / (static_cast<double>(K) * sigma));
    const bool direct = gamma == 0.0f && K <= kDirectMaxDraws;  // scan = identity
    const bool center = (flags & DUST_CENTER) != 0;
    cudaError_t e = cudaSuccess;
    if (!direct) {
        if (cudaMemsetAsync(sync, 0, kSyncBytes, s) != cudaSuccess) return DUST_ERR_CUDA;
        e = launch_scan(delta, K, T, seq_offsets, n_seq, gamma, center, b, s, sync);
    }
    if (e == cudaSuccess)
        e = launch_weight(b, true, K, T, d, seed, static_cast<int>(kind), draw_begin, coef,
                          (flags & DUST_ANTITHETIC) != 0, g, 0, s, direct ? delta : nullptr,
                          center);
    if (e == cudaSuccess) e = launch_scatter_gE(g, 0, ids, T, d, V, scale, acc, gE, ws, s);
    return cuda_status(e);
}

dust_status dust_credit_scan_workspace(size_t* bytes, int64_t K, int64_t T) {
    if (!bytes || K < 1 || T < 0) return DUST_ERR_INVALID_ARG;
    if (K > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    // r lives in the caller's output; the rest in the workspace.
    *bytes = a256(scan_workspace_bytes(K, T)) + 256;
    return DUST_OK;
}

dust_status dust_credit_scan(const float* delta, int64_t K, int64_t T,
                             const int32_t* seq_offsets, int64_t n_seq, float gamma,
                             uint32_t flags, float* r, void* workspace, size_t ws_bytes,
                             void* stream) {
    if (K < 1 || T < 0 || n_seq < 0) return DUST_ERR_INVALID_ARG;
    if (K > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    if (flags & ~DUST_CENTER) return DUST_ERR_INVALID_ARG;
    if (!finite(gamma) || std::fabs(gamma) > 1.0f) return DUST_ERR_INVALID_ARG;
    if (T > 0 && (n_seq < 1 || n_seq > T)) return DUST_ERR_INVALID_ARG;
    if (T == 0) return DUST_OK;
    if (!delta || !seq_offsets || !r) return DUST_ERR_INVALID_ARG;
    size_t need = 0;
    dust_credit_scan_workspace(&need, K, T);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return DUST_ERR_WORKSPACE;
    ScanBuffers b = scan_carve(workspace, K, T);
    b.r = r;  // scan straight into the caller's output
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_scan(delta, K, T, seq_offsets, n_seq, gamma,
                                (flags & DUST_CENTER) != 0, b, s);
    if (e == cudaSuccess) e = launch_scan_fixup(b, K, T, s);
    return cuda_status(e);
}

dust_status dust_error_estimate(const float* r, int64_t K, int64_t T, int64_t d_out,
                                uint64_t seed, dust_noise_kind kind, int64_t draw_begin,
                                float sigma, uint32_t flags, void* g, dust_dtype g_dtype,
                                void* stream) {
    if (K < 1 || draw_begin < 0) return DUST_ERR_INVALID_ARG;
    if (K > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    dust_status st = counter_ok(T, d_out);
    if (st != DUST_OK) return st;
    if (!value_kind(kind)) return DUST_ERR_INVALID_ARG;
    if (g_dtype != DUST_F32 && g_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (flags & ~(DUST_CENTER | DUST_ANTITHETIC)) return DUST_ERR_INVALID_ARG;
    if ((flags & DUST_ANTITHETIC) && ((K & 1) || (draw_begin & 1))) return DUST_ERR_INVALID_ARG;
    if (!finite(sigma) || sigma == 0.0f) return DUST_ERR_INVALID_ARG;
    if (draw_begin > (int64_t(1) << 31) - K) return DUST_ERR_RANGE;
    if (T * d_out == 0) return DUST_OK;
    if (!r || !g) return DUST_ERR_INVALID_ARG;
    ScanBuffers b{};
    b.r = const_cast<float*>(r);
    const float coef = static_cast<float>(-1.0 / (static_cast<double>(K) * sigma));
    return cuda_status(launch_weight(b, false, K, T, d_out, seed, static_cast<int>(kind),
                                     draw_begin, coef, (flags & DUST_ANTITHETIC) != 0, g,
                                     g_dtype == DUST_BF16, static_cast<cudaStream_t>(stream)));
}

dust_status dust_contract_workspace(size_t* bytes, int64_t T, int64_t d_in, int64_t d_out,
                                    dust_dtype dtype, uint32_t flags) {
    if (!bytes || T < 0 || d_in < 0 || d_out < 0) return DUST_ERR_INVALID_ARG;
    if (dtype != DUST_F32 && dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (flags & ~(DUST_ACCUMULATE | DUST_FORCE_SIMT)) return DUST_ERR_INVALID_ARG;
    size_t b = simt_gemm_workspace_bytes(T, d_in, d_out);
    const size_t tcb = tc_gemm_workspace_bytes(T, d_in, d_out);
    if (tcb > b) b = tcb;
    *bytes = kSyncBytes + a256(b) + 256;
    return DUST_OK;
}

dust_status dust_contract(const void* g, const void* X, dust_dtype dtype, int64_t T, int64_t d_in,
                          int64_t d_out, float scale, uint32_t flags, float* gW, void* workspace,
                          size_t ws_bytes, void* stream) {
    size_t need = 0;
    dust_status st = dust_contract_workspace(&need, T, d_in, d_out, dtype, flags);
    if (st != DUST_OK) return st;
    if (!finite(scale)) return DUST_ERR_INVALID_ARG;
    if (d_in * d_out == 0) return DUST_OK;
    if (!gW || (reinterpret_cast<uintptr_t>(gW) % 16)) return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool acc = (flags & DUST_ACCUMULATE) != 0;
    if (T == 0) return acc ? DUST_OK : cuda_status(launch_zero(gW, d_out * d_in, s));
    if (!g || !X) return DUST_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return DUST_ERR_WORKSPACE;
    float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + kSyncBytes);
    const bool bf16 = dtype == DUST_BF16;
    cudaError_t e;
    const bool tc = bf16 && !(flags & DUST_FORCE_SIMT) && tc_gemm_supported(g, X, d_in, d_out);
    if (tc)
        e = launch_tc_gemm(g, X, T, d_in, d_out, scale, acc, gW, part, s);
    else
        e = launch_simt_gemm(g, bf16, X, bf16, T, d_in, d_out, scale, acc, gW, part, s);
    return cuda_status(e);
}

dust_status dust_estimate_gW_workspace(size_t* bytes, int64_t T, int64_t d_in, int64_t d_out,
                                       int64_t K, dust_dtype x_dtype, uint32_t flags) {
    if (!bytes) return DUST_ERR_INVALID_ARG;
    dust_status st = check_estimate(T, d_in, d_out, K, x_dtype, flags);
    if (st != DUST_OK) return st;
    const Layout L = layout(T, d_in, d_out, K, x_dtype, flags);
    if (L.path < 0) return static_cast<dust_status>(-L.path);
    *bytes = L.total;
    return DUST_OK;
}

int32_t dust_estimate_gW_path(int64_t T, int64_t d_in, int64_t d_out, int64_t K,
                              dust_dtype x_dtype, uint32_t flags) {
    dust_status st = check_estimate(T, d_in, d_out, K, x_dtype, flags);
    if (st != DUST_OK) return -static_cast<int32_t>(st);
    return choose_path(T, d_in, d_out, K, x_dtype, flags);
}

}  // extern "C"

namespace {

// Every argument check of the estimator, with nothing enqueued: DUST_OK when
// `estimate` would enqueue its work (or has nothing to do).
dust_status estimate_check(const void* X, dust_dtype x_dtype, int64_t T, int64_t d_in,
                           const float* delta, int64_t K, int64_t d_out,
                           const int32_t* seq_offsets, int64_t n_seq, dust_noise_kind kind,
                           int64_t draw_begin, float sigma, float gamma, float scale,
                           uint32_t flags, const float* gW, const void* workspace,
                           size_t ws_bytes) {
    dust_status st = check_estimate(T, d_in, d_out, K, x_dtype, flags);
    if (st != DUST_OK) return st;
    if (!value_kind(kind)) return DUST_ERR_INVALID_ARG;
    if (draw_begin < 0) return DUST_ERR_INVALID_ARG;
    if (draw_begin > (int64_t(1) << 31) - K) return DUST_ERR_RANGE;
    if ((flags & DUST_ANTITHETIC) && (draw_begin & 1)) return DUST_ERR_INVALID_ARG;
    if (!finite(sigma) || sigma == 0.0f) return DUST_ERR_INVALID_ARG;
    if (!finite(gamma) || std::fabs(gamma) > 1.0f) return DUST_ERR_INVALID_ARG;
    if (!finite(scale)) return DUST_ERR_INVALID_ARG;
    if (T > 0 && (n_seq < 1 || n_seq > T)) return DUST_ERR_INVALID_ARG;
    if (n_seq < 0) return DUST_ERR_INVALID_ARG;
    if (d_out * d_in == 0) return DUST_OK;
    if (!gW || (reinterpret_cast<uintptr_t>(gW) % 16)) return DUST_ERR_INVALID_ARG;
    if (T == 0) return DUST_OK;
    if (!X || !delta || !seq_offsets) return DUST_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(X) % 16) return DUST_ERR_INVALID_ARG;
    const Layout L = layout(T, d_in, d_out, K, x_dtype, flags);
    if (L.path < 0) return static_cast<dust_status>(-L.path);
    // The fused kernel evaluates Gaussian or per-channel Rademacher noise only.
    if (L.path == DUST_PATH_FUSED_TC && kind == DUST_NOISE_RADEMACHER_PACKED)
        return DUST_ERR_UNSUPPORTED;
    if (!workspace || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return DUST_ERR_WORKSPACE;
    return DUST_OK;
}

// The whole estimator on `stream`. When x_ready is given, X is still being
// copied on another stream: the stream waits for that event just before the
// first kernel that reads X (the contraction), so the scan and the weighting
// overlap the copy. `fit`: the contraction build (launch_tc_gemm), by what
// shares its SMs (sites running concurrently on the compute lanes). With `cs`
// given (a lane's contraction stream), the contraction kernel runs there
// after the weighting (event `cs_in`), and `stream` waits for it (event
// `cs_out`) before the slice reduction and anything later.
dust_status estimate(const void* X, dust_dtype x_dtype, int64_t T, int64_t d_in,
                     const float* delta, int64_t K, int64_t d_out, const int32_t* seq_offsets,
                     int64_t n_seq, uint64_t seed, dust_noise_kind kind, int64_t draw_begin,
                     float sigma, float gamma, float scale, uint32_t flags, float* gW,
                     void* workspace, size_t ws_bytes, void* stream, cudaEvent_t x_ready,
                     int fit = 0, cudaStream_t cs = nullptr, cudaEvent_t cs_in = nullptr,
                     cudaEvent_t cs_out = nullptr) {
    const dust_status st =
        estimate_check(X, x_dtype, T, d_in, delta, K, d_out, seq_offsets, n_seq, kind,
                       draw_begin, sigma, gamma, scale, flags, gW, workspace, ws_bytes);
    if (st != DUST_OK) return st;
    if (d_out * d_in == 0) return DUST_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool acc = (flags & DUST_ACCUMULATE) != 0;
    if (T == 0) return acc ? DUST_OK : cuda_status(launch_zero(gW, d_out * d_in, s));
    const Layout L = layout(T, d_in, d_out, K, x_dtype, flags);

    char* ws = static_cast<char*>(workspace);
    unsigned int* sync = reinterpret_cast<unsigned int*>(ws);  // [0]: the scan's ticket
    ws += L.sync;
    ScanBuffers b = scan_carve(ws, K, T);
    void* g = ws + L.scan;
    float* part = reinterpret_cast<float*>(ws + L.scan + L.g);
    const float coef = static_cast<float>(-1.0 / (static_cast<double>(K) * sigma));
    const bool anti = (flags & DUST_ANTITHETIC) != 0;

    // With gamma = 0 the credit scan is the identity (r_t = c_t): the
    // weighting kernel then centres the loss changes itself and no scan runs.
    const bool direct = gamma == 0.0f && K <= kDirectMaxDraws && L.path != DUST_PATH_FUSED_TC;
    const bool center = (flags & DUST_CENTER) != 0;
    if (!direct) {
        if (cudaMemsetAsync(sync, 0, kSyncBytes, s) != cudaSuccess) return DUST_ERR_CUDA;
        if (launch_scan(delta, K, T, seq_offsets, n_seq, gamma, center, b, s, sync) != cudaSuccess)
            return DUST_ERR_CUDA;
    }
    cudaError_t e = cudaSuccess;
    if (L.path == DUST_PATH_FUSED_TC) {
        float* fpart = reinterpret_cast<float*>(ws + L.scan);
        if (x_ready && cudaStreamWaitEvent(s, x_ready, 0) != cudaSuccess) return DUST_ERR_CUDA;
        return cuda_status(launch_fused(b, X, K, T, d_in, d_out, seed, static_cast<int>(kind),
                                        draw_begin, coef, anti, scale, acc, gW, fpart, s));
    }
    e = launch_weight(b, true, K, T, d_out, seed, static_cast<int>(kind), draw_begin, coef, anti,
                      g, L.g_bf16, s, direct ? delta : nullptr, center);
    if (e != cudaSuccess) return DUST_ERR_CUDA;
    if (x_ready && cudaStreamWaitEvent(s, x_ready, 0) != cudaSuccess) return DUST_ERR_CUDA;
    if (cs && L.path == DUST_PATH_UNFUSED_TC && tc_gemm_supported(g, X, d_in, d_out)) {
        if (cudaEventRecord(cs_in, s) != cudaSuccess || cudaStreamWaitEvent(cs, cs_in, 0) != cudaSuccess)
            return DUST_ERR_CUDA;
        return cuda_status(
            launch_tc_gemm(g, X, T, d_in, d_out, scale, acc, gW, part, cs, fit, s, cs_out));
    }
    if (L.path == DUST_PATH_UNFUSED_TC && tc_gemm_supported(g, X, d_in, d_out))
        e = launch_tc_gemm(g, X, T, d_in, d_out, scale, acc, gW, part, s, fit);
    else
        e = launch_simt_gemm(g, L.g_bf16, X, x_dtype == DUST_BF16, T, d_in, d_out, scale, acc,
                             gW, part, s);
    return cuda_status(e);
}

// A copy stream and per-site events per device for the host-buffer entry points, created
// on first use and kept for the life of the process. The mutex covers one
// call's whole enqueue sequence, so the events are re-recorded only after
// every wait on them has been enqueued.
struct CopyLane {
    std::mutex mu;
    bool ready = false;
    cudaError_t err = cudaSuccess;
    cudaStream_t copy = nullptr;  // host -> device inputs
    cudaStream_t ret = nullptr;   // device -> host results of all but the last site
    cudaEvent_t fork = nullptr, ret_done = nullptr;
    std::vector<cudaEvent_t> ev;  // per site: loss changes copied, X copied, ĜW ready
};
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxSites = 4096;
CopyLane g_lanes[kMaxDevices];

// Compute lanes of the multi-site entry points: streams of one device on
// which whole sites run, site i on lane i mod kSiteLanes, each lane with a
// contraction stream of the device's highest priority on which its sites'
// contraction kernels run. The hardware dispatches the CTAs of concurrent
// grids of equal priority in launch order, so a contraction launched behind
// another site's weighting would wait for that whole grid to be placed; at
// the higher priority its CTAs take the room the weighting CTAs leave (the
// 32-register build: one beside five weighting CTAs) and run beside them.
// The slice reductions stay on the lanes: at high priority their many
// short CTAs would take the weighting's places instead. Created on first use
// and kept for the life of the process; the lock covers a call's whole
// enqueue sequence, so the events are re-recorded only after every wait on
// them has been enqueued. Measured on the 48-site sweep (a GB300): 55.9 ms
// per pass on one stream; 54.2 on three lanes without the contraction
// streams; 52.9 with them (2 lanes 52.9, 4 lanes 53.2, 1 lane 56.2).
#ifndef DUST_SITE_LANES
#define DUST_SITE_LANES 3
#endif
constexpr int kSiteLanes = DUST_SITE_LANES;
static_assert(kSiteLanes >= 1, "at least one lane");
// The contraction build the lanes use (launch_tc_gemm's `fit`).
#ifndef DUST_SITE_FIT
#define DUST_SITE_FIT 2
#endif
constexpr int kSiteFit = DUST_SITE_FIT;

struct SiteLanes {
    std::mutex mu;
    bool ready = false;
    cudaError_t err = cudaSuccess;
    cudaStream_t lane[kSiteLanes] = {};
    cudaStream_t gemm[kSiteLanes] = {};  // the lanes' contraction streams
    cudaEvent_t fork = nullptr;
    cudaEvent_t join[kSiteLanes] = {}, gemm_join[kSiteLanes] = {};
    cudaEvent_t gemm_in[kSiteLanes] = {}, gemm_out[kSiteLanes] = {};
};
SiteLanes g_site_lanes[kMaxDevices];

// The current device's lanes, locked into `lock` (created on first use);
// nullptr if they could not be made.
SiteLanes* site_lanes(std::unique_lock<std::mutex>& lock) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    SiteLanes* L = &g_site_lanes[dev];
    lock = std::unique_lock<std::mutex>(L->mu);
    if (!L->ready) {
        int least = 0, greatest = 0;
        L->err = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        for (int l = 0; l < kSiteLanes && L->err == cudaSuccess; ++l) {
            L->err = cudaStreamCreateWithFlags(&L->lane[l], cudaStreamNonBlocking);
            if (L->err == cudaSuccess)
                L->err = cudaStreamCreateWithPriority(&L->gemm[l], cudaStreamNonBlocking, greatest);
            cudaEvent_t* evs[4] = {&L->join[l], &L->gemm_join[l], &L->gemm_in[l], &L->gemm_out[l]};
            for (cudaEvent_t* e : evs)
                if (L->err == cudaSuccess)
                    L->err = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
        }
        if (L->err == cudaSuccess)
            L->err = cudaEventCreateWithFlags(&L->fork, cudaEventDisableTiming);
        L->ready = true;
    }
    return L->err == cudaSuccess ? L : nullptr;
}

// Lanes 0 .. used-1 and their contraction streams start after the work
// enqueued on `s` so far.
bool fork_lanes(SiteLanes* L, int used, cudaStream_t s) {
    if (cudaEventRecord(L->fork, s) != cudaSuccess) return false;
    for (int l = 0; l < used; ++l)
        if (cudaStreamWaitEvent(L->lane[l], L->fork, 0) != cudaSuccess ||
            cudaStreamWaitEvent(L->gemm[l], L->fork, 0) != cudaSuccess)
            return false;
    return true;
}

// `s` waits for everything enqueued on lanes 0 .. used-1 and their
// contraction streams.
bool join_lanes(SiteLanes* L, int used, cudaStream_t s) {
    for (int l = 0; l < used; ++l)
        if (cudaEventRecord(L->join[l], L->lane[l]) != cudaSuccess ||
            cudaStreamWaitEvent(s, L->join[l], 0) != cudaSuccess ||
            cudaEventRecord(L->gemm_join[l], L->gemm[l]) != cudaSuccess ||
            cudaStreamWaitEvent(s, L->gemm_join[l], 0) != cudaSuccess)
            return false;
    return true;
}

// One device buffer of a multi-site call.
struct SiteRange {
    uintptr_t lo, hi;
    int64_t site;
    bool written;
};

// The two largest range ends seen so far that belong to two different sites.
struct EndsBySite {
    uintptr_t hi1 = 0, hi2 = 0;
    int64_t site1 = -1, site2 = -1;
    void add(uintptr_t hi, int64_t site) {
        if (site == site1) {
            if (hi > hi1) hi1 = hi;
        } else if (hi > hi1) {
            hi2 = hi1;
            site2 = site1;
            hi1 = hi;
            site1 = site;
        } else if (hi > hi2) {
            hi2 = hi;
            site2 = site;
        }
    }
    // the largest end among sites other than `site`
    uintptr_t other(int64_t site) const { return site == site1 ? hi2 : hi1; }
};

// True when no written range overlaps a range of another site. Sorted by
// start, a range overlaps an earlier one exactly when it starts before that
// one's end; it conflicts with one of another site when either is written.
bool sites_disjoint(std::vector<SiteRange>& rs) {
    std::sort(rs.begin(), rs.end(),
              [](const SiteRange& a, const SiteRange& b) { return a.lo < b.lo; });
    EndsBySite all, written;
    for (const SiteRange& r : rs) {
        if (r.lo < (r.written ? all : written).other(r.site)) return false;
        all.add(r.hi, r.site);
        if (r.written) written.add(r.hi, r.site);
    }
    return true;
}

#ifndef DUST_HOST_DIRECT_GW
#define DUST_HOST_DIRECT_GW 1
#endif

// Every argument of an estimator call, zero-padded: the key of its graph.
struct CallArgs {
    int32_t entry;  // 0: dust_estimate_gW, 1: dust_estimate_gW_host
    int32_t x_dtype, kind;
    uint32_t flags;
    int64_t T, d_in, K, d_out, n_seq, draw_begin;
    uint64_t seed;
    float sigma, gamma, scale, pad;
    const void *X, *X_host;
    const float *delta, *delta_host;
    const int32_t *seq, *seq_host;
    float *gW, *gW_host;
    void* workspace;
    size_t ws_bytes;
};

dust_status estimate_host(const void* X_host, void* X_dev, dust_dtype x_dtype, int64_t T,
                          int64_t d_in, const float* delta_host, float* delta_dev, int64_t K,
                          int64_t d_out, const int32_t* seq_offsets_host, int32_t* seq_dev,
                          int64_t n_seq, uint64_t seed, dust_noise_kind kind,
                          int64_t draw_begin, float sigma, float gamma, float scale,
                          uint32_t flags, float* gW_host, float* gW_dev, void* workspace,
                          size_t ws_bytes, void* stream);
dust_status estimate_host_sites(const dust_host_site* sites, int64_t n, dust_dtype x_dtype,
                                dust_noise_kind kind, int64_t draw_begin, float scale,
                                uint32_t flags, void* stream);

dust_status enqueue_device(const void* ctx, cudaStream_t s) {
    const CallArgs& a = *static_cast<const CallArgs*>(ctx);
    return estimate(a.X, static_cast<dust_dtype>(a.x_dtype), a.T, a.d_in, a.delta, a.K,
                    a.d_out, a.seq, a.n_seq, a.seed, static_cast<dust_noise_kind>(a.kind),
                    a.draw_begin, a.sigma, a.gamma, a.scale, a.flags, a.gW, a.workspace,
                    a.ws_bytes, s, nullptr);
}

dust_status enqueue_host(const void* ctx, cudaStream_t s) {
    const CallArgs& a = *static_cast<const CallArgs*>(ctx);
    return estimate_host(a.X_host, const_cast<void*>(a.X), static_cast<dust_dtype>(a.x_dtype),
                         a.T, a.d_in, a.delta_host, const_cast<float*>(a.delta), a.K, a.d_out,
                         a.seq_host, const_cast<int32_t*>(a.seq), a.n_seq, a.seed,
                         static_cast<dust_noise_kind>(a.kind), a.draw_begin, a.sigma, a.gamma,
                         a.scale, a.flags, a.gW_host, a.gW, a.workspace, a.ws_bytes, s);
}

static_assert(sizeof(dust_site) == 13 * 8, "dust_site has no padding (its bytes key graphs)");

// Several sites on the compute lanes (see dust.h): every check first, then
// site i on lane i mod kSiteLanes between a fork from and a join into `s`.
dust_status estimate_sites(const dust_site* sites, int64_t n, dust_dtype x_dtype,
                           dust_noise_kind kind, int64_t draw_begin, float scale, uint32_t flags,
                           cudaStream_t s) {
    if (n < 0 || (n > 0 && !sites)) return DUST_ERR_INVALID_ARG;
    if (n > kMaxSites) return DUST_ERR_RANGE;
    for (int64_t i = 0; i < n; ++i) {
        const dust_site& q = sites[i];
        const dust_status st =
            estimate_check(q.X, x_dtype, q.T, q.d_in, q.delta, q.K, q.d_out, q.seq_offsets,
                           q.n_seq, kind, draw_begin, q.sigma, q.gamma, scale, flags, q.gW,
                           q.workspace, q.ws_bytes);
        if (st != DUST_OK) return st;
    }
    if (n > 1) {
        const size_t esz = (x_dtype == DUST_BF16) ? 2 : 4;
        std::vector<SiteRange> rs;
        rs.reserve(static_cast<size_t>(5 * n));
        auto add = [&](const void* p, size_t bytes, int64_t site, bool written) {
            if (p && bytes) {
                const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
                rs.push_back(SiteRange{lo, lo + bytes, site, written});
            }
        };
        for (int64_t i = 0; i < n; ++i) {
            const dust_site& q = sites[i];
            if (q.d_out * q.d_in == 0) continue;  // nothing read or written
            add(q.gW, sizeof(float) * static_cast<size_t>(q.d_out * q.d_in), i, true);
            if (q.T == 0) continue;  // gW zeroed (or left), nothing else touched
            add(q.X, esz * static_cast<size_t>(q.T * q.d_in), i, false);
            add(q.delta, sizeof(float) * static_cast<size_t>(q.K * q.T), i, false);
            add(q.seq_offsets, sizeof(int32_t) * static_cast<size_t>(q.n_seq + 1), i, false);
            add(q.workspace, q.ws_bytes, i, true);
        }
        if (!sites_disjoint(rs)) return DUST_ERR_INVALID_ARG;
    }
    if (n == 0) return DUST_OK;
    if (n == 1) {
        const dust_site& q = sites[0];
        return estimate(q.X, x_dtype, q.T, q.d_in, q.delta, q.K, q.d_out, q.seq_offsets,
                        q.n_seq, q.seed, kind, draw_begin, q.sigma, q.gamma, scale, flags, q.gW,
                        q.workspace, q.ws_bytes, s, nullptr);
    }
    std::unique_lock<std::mutex> lock;
    SiteLanes* L = site_lanes(lock);
    if (!L) return DUST_ERR_CUDA;
    const int used = n < kSiteLanes ? static_cast<int>(n) : kSiteLanes;
    if (!fork_lanes(L, used, s)) return DUST_ERR_CUDA;
    dust_status result = DUST_OK;
    for (int64_t i = 0; i < n && result == DUST_OK; ++i) {
        const dust_site& q = sites[i];
        const int l = static_cast<int>(i % kSiteLanes);
        result = estimate(q.X, x_dtype, q.T, q.d_in, q.delta, q.K, q.d_out, q.seq_offsets,
                          q.n_seq, q.seed, kind, draw_begin, q.sigma, q.gamma, scale, flags,
                          q.gW, q.workspace, q.ws_bytes, L->lane[l], nullptr, kSiteFit,
                          L->gemm[l], L->gemm_in[l], L->gemm_out[l]);
    }
    // However the sequence ended, `s` waits for what the lanes were given.
    if (!join_lanes(L, used, s)) return DUST_ERR_CUDA;
    return result;
}

// A multi-site call: its shared arguments and its site array (the graph key
// is both, byte for byte).
struct SitesCall {
    const dust_site* sites;
    int64_t n;
    int32_t x_dtype, kind;
    int64_t draw_begin;
    float scale;
    uint32_t flags;
};

dust_status enqueue_sites(const void* ctx, cudaStream_t s) {
    const SitesCall& c = *static_cast<const SitesCall*>(ctx);
    return estimate_sites(c.sites, c.n, static_cast<dust_dtype>(c.x_dtype),
                          static_cast<dust_noise_kind>(c.kind), c.draw_begin, c.scale, c.flags,
                          s);
}

}  // namespace

extern "C" {

dust_status dust_estimate_gW_sites(const dust_site* sites, int64_t n_sites, dust_dtype x_dtype,
                                   dust_noise_kind kind, int64_t draw_begin, float scale,
                                   uint32_t flags, void* stream) {
    SitesCall c;
    c.sites = sites;
    c.n = n_sites;
    c.x_dtype = x_dtype;
    c.kind = kind;
    c.draw_begin = draw_begin;
    c.scale = scale;
    c.flags = flags;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n_sites < 2 || n_sites > kMaxSites || !sites) return enqueue_sites(&c, s);
    // key: entry tag and shared arguments, then the site array
    struct Head {
        int32_t entry, x_dtype, kind;
        uint32_t flags;
        int64_t n, draw_begin;
        float scale, pad;
    } h;
    std::memset(&h, 0, sizeof(h));
    h.entry = 2;
    h.x_dtype = x_dtype;
    h.kind = kind;
    h.flags = flags;
    h.n = n_sites;
    h.draw_begin = draw_begin;
    h.scale = scale;
    std::vector<unsigned char> key(sizeof(h) + sizeof(dust_site) * static_cast<size_t>(n_sites));
    std::memcpy(key.data(), &h, sizeof(h));
    std::memcpy(key.data() + sizeof(h), sites, sizeof(dust_site) * static_cast<size_t>(n_sites));
    // The graph keeps each kernel's stream priority: the contraction streams'
    // high priority is what lets their CTAs run beside the weighting (replayed
    // at one priority, the pass measured 53.7 ms on average against 52.9).
    return graph_call(key.data(), key.size(), s, enqueue_sites, &c, true);
}

int32_t dust_estimate_gW_sites_lanes(void) { return kSiteLanes; }

dust_status dust_estimate_gW(const void* X, dust_dtype x_dtype, int64_t T, int64_t d_in,
                             const float* delta, int64_t K, int64_t d_out,
                             const int32_t* seq_offsets, int64_t n_seq, uint64_t seed,
                             dust_noise_kind kind, int64_t draw_begin, float sigma, float gamma,
                             float scale, uint32_t flags, float* gW, void* workspace,
                             size_t ws_bytes, void* stream) {
    CallArgs a;
    std::memset(&a, 0, sizeof(a));
    a.entry = 0;
    a.x_dtype = x_dtype;
    a.kind = kind;
    a.flags = flags;
    a.T = T;
    a.d_in = d_in;
    a.K = K;
    a.d_out = d_out;
    a.n_seq = n_seq;
    a.draw_begin = draw_begin;
    a.seed = seed;
    a.sigma = sigma;
    a.gamma = gamma;
    a.scale = scale;
    a.X = X;
    a.delta = delta;
    a.seq = seq_offsets;
    a.gW = gW;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    return graph_call(&a, sizeof(a), static_cast<cudaStream_t>(stream), enqueue_device, &a);
}

dust_status dust_estimate_gW_host(const void* X_host, void* X_dev, dust_dtype x_dtype, int64_t T,
                                  int64_t d_in, const float* delta_host, float* delta_dev,
                                  int64_t K, int64_t d_out, const int32_t* seq_offsets_host,
                                  int32_t* seq_dev, int64_t n_seq, uint64_t seed,
                                  dust_noise_kind kind, int64_t draw_begin, float sigma,
                                  float gamma, float scale, uint32_t flags, float* gW_host,
                                  float* gW_dev, void* workspace, size_t ws_bytes,
                                  void* stream) {
    CallArgs a;
    std::memset(&a, 0, sizeof(a));
    a.entry = 1;
    a.x_dtype = x_dtype;
    a.kind = kind;
    a.flags = flags;
    a.T = T;
    a.d_in = d_in;
    a.K = K;
    a.d_out = d_out;
    a.n_seq = n_seq;
    a.draw_begin = draw_begin;
    a.seed = seed;
    a.sigma = sigma;
    a.gamma = gamma;
    a.scale = scale;
    a.X = X_dev;
    a.X_host = X_host;
    a.delta = delta_dev;
    a.delta_host = delta_host;
    a.seq = seq_dev;
    a.seq_host = seq_offsets_host;
    a.gW = gW_dev;
    a.gW_host = gW_host;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    // Direct launches: replayed as a graph this path measured 6 us slower per
    // call (229 against 223 us on the 512 x 2048 layer), the copy branch and
    // the kernels overlapping less well than when issued one by one.
    return enqueue_host(&a, static_cast<cudaStream_t>(stream));
}

dust_status dust_estimate_gW_host_sites(const dust_host_site* sites, int64_t n_sites,
                                        dust_dtype x_dtype, dust_noise_kind kind,
                                        int64_t draw_begin, float scale, uint32_t flags,
                                        void* stream) {
    return estimate_host_sites(sites, n_sites, x_dtype, kind, draw_begin, scale, flags, stream);
}

}  // extern "C"

namespace {

// Device byte range [lo, hi) of one buffer of a multi-site call.
struct Range {
    uintptr_t lo, hi;
    int64_t site;
    bool async;  // written by the copy stream, out of `stream`'s order
};


// The estimator for several sites from host buffers (see dust.h). Inputs go
// host -> device over an internal copy stream that runs ahead of the compute
// on `stream`: site 0's loss changes and offsets are copied on `stream` first
// (the scan needs them at once); then the copy stream, after everything
// enqueued on `stream` before this call, copies X of site 0 and, for every
// later site i, its loss changes, offsets and X, recording an event after
// each. Site i's kernels wait for its loss changes before its first kernel
// and for its X only before its contraction, so every copy after the first
// overlaps the compute of earlier sites.
dust_status estimate_host_sites(const dust_host_site* sites, int64_t n, dust_dtype x_dtype,
                                dust_noise_kind kind, int64_t draw_begin, float scale,
                                uint32_t flags, void* stream) {
    if (n < 0 || (n > 0 && !sites)) return DUST_ERR_INVALID_ARG;
    if (n > kMaxSites) return DUST_ERR_RANGE;
    const size_t esz = (x_dtype == DUST_BF16) ? 2 : 4;
    // Every check before anything is enqueued.
    for (int64_t i = 0; i < n; ++i) {
        const dust_host_site& q = sites[i];
        dust_status st = check_estimate(q.T, q.d_in, q.d_out, q.K, x_dtype, flags);
        if (st != DUST_OK) return st;
        if (q.n_seq < 0 || (q.T > 0 && q.n_seq < 1)) return DUST_ERR_INVALID_ARG;
        if (q.d_out * q.d_in > 0 && (!q.gW_host || !q.gW_dev)) return DUST_ERR_INVALID_ARG;
        if (q.T > 0 && (!q.X_host || !q.X_dev || !q.delta_host || !q.delta_dev ||
                        !q.seq_offsets_host || !q.seq_dev))
            return DUST_ERR_INVALID_ARG;
        st = estimate_check(q.X_dev, x_dtype, q.T, q.d_in, q.delta_dev, q.K, q.d_out, q.seq_dev,
                            q.n_seq, kind, draw_begin, q.sigma, q.gamma, scale, flags, q.gW_dev,
                            q.workspace, q.ws_bytes);
        if (st != DUST_OK) return st;
    }
    // Buffers that the copy stream writes while the sites compute must not
    // overlap any other device buffer of the call; what a site's kernels
    // write (its workspace and gW_dev) must not overlap a buffer of another
    // site, whose kernels run on another lane.
    if (n > 1) {
        std::vector<Range> rs;
        std::vector<SiteRange> sr;
        rs.reserve(static_cast<size_t>(5 * n));
        sr.reserve(static_cast<size_t>(5 * n));
        auto add = [&](const void* p, size_t bytes, int64_t site, bool async, bool written) {
            if (p && bytes) {
                const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
                rs.push_back(Range{lo, lo + bytes, site, async});
                sr.push_back(SiteRange{lo, lo + bytes, site, written});
            }
        };
        for (int64_t i = 0; i < n; ++i) {
            const dust_host_site& q = sites[i];
            if (q.d_out * q.d_in == 0) continue;
            // read by the return stream while later sites compute
            add(q.gW_dev, sizeof(float) * static_cast<size_t>(q.d_out * q.d_in), i, i < n - 1,
                true);
            if (q.T == 0) continue;
            add(q.X_dev, esz * static_cast<size_t>(q.T * q.d_in), i, true, false);
            add(q.delta_dev, sizeof(float) * static_cast<size_t>(q.K * q.T), i, i > 0, false);
            add(q.seq_dev, sizeof(int32_t) * static_cast<size_t>(q.n_seq + 1), i, i > 0, false);
            add(q.workspace, q.ws_bytes, i, false, true);
        }
        if (!sites_disjoint(sr)) return DUST_ERR_INVALID_ARG;
        // Sorted by start, a range overlaps an earlier one exactly when it
        // starts before the largest end seen so far; an asynchronous range
        // may overlap nothing, any other range no asynchronous one.
        std::sort(rs.begin(), rs.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
        uintptr_t end_all = 0, end_async = 0;
        for (const Range& r : rs) {
            if (r.lo < (r.async ? end_all : end_async)) return DUST_ERR_INVALID_ARG;
            end_all = r.hi > end_all ? r.hi : end_all;
            if (r.async) end_async = r.hi > end_async ? r.hi : end_async;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // Per site: the device address ĜW goes to. For the last site (the only
    // one of a single-site call) a page-locked, device-mapped gW_host is
    // written (and, accumulating, read) by the kernels in place, over the host
    // link, instead of through gW_dev and a copy back. Earlier sites write
    // gW_dev, which a return stream copies back while later sites compute
    // (in place, each site's writes would hold its contraction, and with it
    // every later kernel on `stream`, until they crossed the link).
    std::vector<float*> target(static_cast<size_t>(n));
    std::vector<char> direct(static_cast<size_t>(n), 0);
    for (int64_t i = 0; i < n; ++i) {
        const dust_host_site& q = sites[i];
        target[i] = q.gW_dev;
#if DUST_HOST_DIRECT_GW
        if (i == n - 1 && q.d_out * q.d_in > 0) {
            cudaPointerAttributes pa;
            if (cudaPointerGetAttributes(&pa, q.gW_host) == cudaSuccess &&
                pa.type == cudaMemoryTypeHost && pa.devicePointer &&
                reinterpret_cast<uintptr_t>(pa.devicePointer) % 16 == 0) {
                target[i] = static_cast<float*>(pa.devicePointer);
                direct[i] = 1;
            }
            (void)cudaGetLastError();
        }
#endif
    }

    auto small_copies = [&](const dust_host_site& q, cudaStream_t cs) {
        if (q.T == 0) return true;
        return cudaMemcpyAsync(q.delta_dev, q.delta_host,
                               sizeof(float) * static_cast<size_t>(q.K * q.T),
                               cudaMemcpyHostToDevice, cs) == cudaSuccess &&
               cudaMemcpyAsync(q.seq_dev, q.seq_offsets_host,
                               sizeof(int32_t) * static_cast<size_t>(q.n_seq + 1),
                               cudaMemcpyHostToDevice, cs) == cudaSuccess;
    };
    auto gw_in = [&](int64_t i, cudaStream_t cs) {
        const dust_host_site& q = sites[i];
        const size_t gw_bytes = sizeof(float) * static_cast<size_t>(q.d_out * q.d_in);
        if (!(flags & DUST_ACCUMULATE) || !gw_bytes || direct[i]) return true;
        return cudaMemcpyAsync(q.gW_dev, q.gW_host, gw_bytes, cudaMemcpyHostToDevice, cs) ==
               cudaSuccess;
    };
    if (n > 0 && (!small_copies(sites[0], s) || !gw_in(0, s))) return DUST_ERR_CUDA;

    // The copy lane: its input and return streams and three events per site,
    // created on first use and kept for the life of the process. The lock
    // covers the whole enqueue sequence, so the events are re-recorded only
    // after every wait on them has been enqueued. Per site i: ev[3i] its loss
    // changes and offsets copied, ev[3i+1] its X copied, ev[3i+2] its ĜW
    // computed into gW_dev (sites before the last).
    bool any_x = false;
    for (int64_t i = 0; i < n; ++i)
        if (sites[i].T * sites[i].d_in > 0 && sites[i].d_out * sites[i].d_in > 0) any_x = true;
    CopyLane* lane = nullptr;
    std::unique_lock<std::mutex> lock;
    // With several sites the compute runs on the compute lanes (as for
    // dust_estimate_gW_sites), site i on lane i mod kSiteLanes.
    SiteLanes* lanes = nullptr;
    std::unique_lock<std::mutex> lanes_lock;
    int used = 0;
    if (any_x || n > 1) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
            return DUST_ERR_CUDA;
        lane = &g_lanes[dev];
        lock = std::unique_lock<std::mutex>(lane->mu);
        if (!lane->ready) {
            lane->err = cudaStreamCreateWithFlags(&lane->copy, cudaStreamNonBlocking);
            if (lane->err == cudaSuccess)
                lane->err = cudaStreamCreateWithFlags(&lane->ret, cudaStreamNonBlocking);
            if (lane->err == cudaSuccess)
                lane->err = cudaEventCreateWithFlags(&lane->fork, cudaEventDisableTiming);
            if (lane->err == cudaSuccess)
                lane->err = cudaEventCreateWithFlags(&lane->ret_done, cudaEventDisableTiming);
            lane->ready = true;
        }
        if (lane->err != cudaSuccess) return DUST_ERR_CUDA;
        while (lane->ev.size() < static_cast<size_t>(3 * n)) {
            cudaEvent_t e = nullptr;
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                return DUST_ERR_CUDA;
            lane->ev.push_back(e);
        }
        if (n > 1) {
            lanes = site_lanes(lanes_lock);
            if (!lanes) return DUST_ERR_CUDA;
            used = n < kSiteLanes ? static_cast<int>(n) : kSiteLanes;
        }
        if (cudaEventRecord(lane->fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(lane->copy, lane->fork, 0) != cudaSuccess ||
            cudaStreamWaitEvent(lane->ret, lane->fork, 0) != cudaSuccess)
            return DUST_ERR_CUDA;
        if (lanes && !fork_lanes(lanes, used, s)) return DUST_ERR_CUDA;
        for (int64_t i = 0; i < n; ++i) {
            const dust_host_site& q = sites[i];
            if (i > 0 && (!small_copies(q, lane->copy) ||
                          cudaEventRecord(lane->ev[3 * i], lane->copy) != cudaSuccess))
                return DUST_ERR_CUDA;
            const size_t x_bytes = esz * static_cast<size_t>(q.T * q.d_in);
            if (x_bytes && q.d_out * q.d_in > 0 &&
                cudaMemcpyAsync(q.X_dev, q.X_host, x_bytes, cudaMemcpyHostToDevice,
                                lane->copy) != cudaSuccess)
                return DUST_ERR_CUDA;
            if (cudaEventRecord(lane->ev[3 * i + 1], lane->copy) != cudaSuccess)
                return DUST_ERR_CUDA;
        }
    }
    dust_status result = DUST_OK;
    for (int64_t i = 0; i < n && result == DUST_OK; ++i) {
        const dust_host_site& q = sites[i];
        cudaStream_t cs = lanes ? lanes->lane[i % kSiteLanes] : s;
        if (i > 0) {
            // the inputs came over the copy stream (or, with no lane, go now)
            const bool ok = lane ? cudaStreamWaitEvent(cs, lane->ev[3 * i], 0) == cudaSuccess
                                 : small_copies(q, cs);
            if (!ok || !gw_in(i, cs)) {
                result = DUST_ERR_CUDA;
                break;
            }
        }
        const int l = static_cast<int>(i % kSiteLanes);
        result = estimate(q.X_dev, x_dtype, q.T, q.d_in, q.delta_dev, q.K, q.d_out, q.seq_dev,
                          q.n_seq, q.seed, kind, draw_begin, q.sigma, q.gamma, scale, flags,
                          target[i], q.workspace, q.ws_bytes, cs,
                          lane ? lane->ev[3 * i + 1] : nullptr, lanes ? kSiteFit : 0,
                          lanes ? lanes->gemm[l] : nullptr, lanes ? lanes->gemm_in[l] : nullptr,
                          lanes ? lanes->gemm_out[l] : nullptr);
        const size_t gw_bytes = sizeof(float) * static_cast<size_t>(q.d_out * q.d_in);
        if (result != DUST_OK || !gw_bytes || direct[i]) continue;
        if (i < n - 1) {
            // copied back on the return stream while later sites compute
            if (cudaEventRecord(lane->ev[3 * i + 2], cs) != cudaSuccess ||
                cudaStreamWaitEvent(lane->ret, lane->ev[3 * i + 2], 0) != cudaSuccess ||
                cudaMemcpyAsync(q.gW_host, q.gW_dev, gw_bytes, cudaMemcpyDeviceToHost,
                                lane->ret) != cudaSuccess)
                result = DUST_ERR_CUDA;
        } else if (cudaMemcpyAsync(q.gW_host, q.gW_dev, gw_bytes, cudaMemcpyDeviceToHost, cs) !=
                   cudaSuccess) {
            result = DUST_ERR_CUDA;
        }
    }
    // However the sequence ended, `stream` waits for the compute lanes and
    // for every copy of the call.
    if (lanes && !join_lanes(lanes, used, s)) return DUST_ERR_CUDA;
    if (lane && n > 0) {
        if (cudaStreamWaitEvent(s, lane->ev[3 * n - 2], 0) != cudaSuccess ||
            cudaEventRecord(lane->ret_done, lane->ret) != cudaSuccess ||
            cudaStreamWaitEvent(s, lane->ret_done, 0) != cudaSuccess)
            return DUST_ERR_CUDA;
    }
    return result;
}

dust_status estimate_host(const void* X_host, void* X_dev, dust_dtype x_dtype, int64_t T,
                          int64_t d_in, const float* delta_host, float* delta_dev, int64_t K,
                          int64_t d_out, const int32_t* seq_offsets_host, int32_t* seq_dev,
                          int64_t n_seq, uint64_t seed, dust_noise_kind kind,
                          int64_t draw_begin, float sigma, float gamma, float scale,
                          uint32_t flags, float* gW_host, float* gW_dev, void* workspace,
                          size_t ws_bytes, void* stream) {
    dust_host_site q;
    q.X_host = X_host;
    q.X_dev = X_dev;
    q.T = T;
    q.d_in = d_in;
    q.d_out = d_out;
    q.delta_host = delta_host;
    q.delta_dev = delta_dev;
    q.K = K;
    q.seq_offsets_host = seq_offsets_host;
    q.seq_dev = seq_dev;
    q.n_seq = n_seq;
    q.seed = seed;
    q.sigma = sigma;
    q.gamma = gamma;
    q.gW_host = gW_host;
    q.gW_dev = gW_dev;
    q.workspace = workspace;
    q.ws_bytes = ws_bytes;
    return estimate_host_sites(&q, 1, x_dtype, kind, draw_begin, scale, flags, stream);
}

}  // namespace

extern "C" {

dust_status dust_last_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DUST_ERR_CUDA;
    unsigned int* w = status_word();
    if (!w) return DUST_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DUST_ERR_CUDA;
    if (v != 0) {
        const unsigned int z = 0;
        if (cudaMemcpy(w, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess)
            return DUST_ERR_CUDA;
    }
    return static_cast<dust_status>(v);
}

}  // extern "C"
