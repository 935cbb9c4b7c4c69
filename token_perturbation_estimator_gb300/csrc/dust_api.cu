// C ABI (include/dust.h): argument validation, workspace layout and dispatch.
// Everything is enqueued on the caller's stream (dust_estimate_gW_host also
// copies X on an internal stream and joins back); nothing here allocates
// device memory or synchronises, except dust_last_error.
#include <cmath>
#include <cstring>
#include <mutex>

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

// The whole estimator on `stream`. When x_ready is given, X is still being
// copied on another stream: the stream waits for that event just before the
// first kernel that reads X (the contraction), so the scan and the weighting
// overlap the copy.
dust_status estimate(const void* X, dust_dtype x_dtype, int64_t T, int64_t d_in,
                     const float* delta, int64_t K, int64_t d_out, const int32_t* seq_offsets,
                     int64_t n_seq, uint64_t seed, dust_noise_kind kind, int64_t draw_begin,
                     float sigma, float gamma, float scale, uint32_t flags, float* gW,
                     void* workspace, size_t ws_bytes, void* stream, cudaEvent_t x_ready) {
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool acc = (flags & DUST_ACCUMULATE) != 0;
    if (T == 0) return acc ? DUST_OK : cuda_status(launch_zero(gW, d_out * d_in, s));
    if (!X || !delta || !seq_offsets) return DUST_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(X) % 16) return DUST_ERR_INVALID_ARG;
    const Layout L = layout(T, d_in, d_out, K, x_dtype, flags);
    if (L.path < 0) return static_cast<dust_status>(-L.path);
    // The fused kernel evaluates Gaussian or per-channel Rademacher noise only.
    if (L.path == DUST_PATH_FUSED_TC && kind == DUST_NOISE_RADEMACHER_PACKED)
        return DUST_ERR_UNSUPPORTED;
    if (!workspace || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return DUST_ERR_WORKSPACE;

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
    if (L.path == DUST_PATH_UNFUSED_TC && tc_gemm_supported(g, X, d_in, d_out))
        e = launch_tc_gemm(g, X, T, d_in, d_out, scale, acc, gW, part, s);
    else
        e = launch_simt_gemm(g, L.g_bf16, X, x_dtype == DUST_BF16, T, d_in, d_out, scale, acc,
                             gW, part, s);
    return cuda_status(e);
}

// A copy stream and two events per device for dust_estimate_gW_host, created
// on first use and kept for the life of the process. The mutex covers one
// call's whole enqueue sequence, so the events are re-recorded only after
// every wait on them has been enqueued.
struct CopyLane {
    std::mutex mu;
    bool ready = false;
    cudaError_t err = cudaSuccess;
    cudaStream_t copy = nullptr;
    cudaEvent_t fork = nullptr, x_done = nullptr;
};
constexpr int kMaxDevices = 64;
CopyLane g_lanes[kMaxDevices];

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

}  // namespace

extern "C" {

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

}  // extern "C"

namespace {

dust_status estimate_host(const void* X_host, void* X_dev, dust_dtype x_dtype, int64_t T,
                          int64_t d_in, const float* delta_host, float* delta_dev, int64_t K,
                          int64_t d_out, const int32_t* seq_offsets_host, int32_t* seq_dev,
                          int64_t n_seq, uint64_t seed, dust_noise_kind kind,
                          int64_t draw_begin, float sigma, float gamma, float scale,
                          uint32_t flags, float* gW_host, float* gW_dev, void* workspace,
                          size_t ws_bytes, void* stream) {
    dust_status st = check_estimate(T, d_in, d_out, K, x_dtype, flags);
    if (st != DUST_OK) return st;
    if (n_seq < 0 || (T > 0 && n_seq < 1)) return DUST_ERR_INVALID_ARG;
    if (d_out * d_in > 0 && (!gW_host || !gW_dev)) return DUST_ERR_INVALID_ARG;
    if (T > 0 && (!X_host || !X_dev || !delta_host || !delta_dev || !seq_offsets_host ||
                  !seq_dev))
        return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t esz = (x_dtype == DUST_BF16) ? 2 : 4;
    const size_t gw_bytes = sizeof(float) * static_cast<size_t>(d_out * d_in);
    const size_t x_bytes = esz * static_cast<size_t>(T * d_in);
    // The small inputs first, on `stream`: the scan needs them at once.
    if (T > 0) {
        if (cudaMemcpyAsync(delta_dev, delta_host, sizeof(float) * static_cast<size_t>(K * T),
                            cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(seq_dev, seq_offsets_host, sizeof(int32_t) * (n_seq + 1),
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return DUST_ERR_CUDA;
    }
    // A page-locked, device-mapped gW_host is written (and, accumulating, read)
    // by the kernels in place, over the host link, instead of through gW_dev
    // and a copy back.
    float* gw_target = gW_dev;
    bool direct = false;
#if DUST_HOST_DIRECT_GW
    if (gw_bytes) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, gW_host) == cudaSuccess &&
            pa.type == cudaMemoryTypeHost && pa.devicePointer &&
            reinterpret_cast<uintptr_t>(pa.devicePointer) % 16 == 0) {
            gw_target = static_cast<float*>(pa.devicePointer);
            direct = true;
        }
        (void)cudaGetLastError();
    }
#endif
    if ((flags & DUST_ACCUMULATE) && gw_bytes && !direct &&
        cudaMemcpyAsync(gW_dev, gW_host, gw_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DUST_ERR_CUDA;
    // X, the large input, then goes over a second copy stream while delta is
    // scanned and weighted; `stream` waits for it before the contraction and,
    // in every case, before this call's work on `stream` ends. The copy starts
    // after everything enqueued on `stream` so far: earlier work that may
    // still read X_dev, and the small copies above (host-to-device copies
    // share an engine, so an earlier X copy would hold the scan's inputs up).
    CopyLane* lane = nullptr;
    std::unique_lock<std::mutex> lock;
    if (x_bytes > 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
            return DUST_ERR_CUDA;
        lane = &g_lanes[dev];
        lock = std::unique_lock<std::mutex>(lane->mu);
        if (!lane->ready) {
            lane->err = cudaStreamCreateWithFlags(&lane->copy, cudaStreamNonBlocking);
            if (lane->err == cudaSuccess)
                lane->err = cudaEventCreateWithFlags(&lane->fork, cudaEventDisableTiming);
            if (lane->err == cudaSuccess)
                lane->err = cudaEventCreateWithFlags(&lane->x_done, cudaEventDisableTiming);

            lane->ready = true;
        }
        if (lane->err != cudaSuccess) return DUST_ERR_CUDA;
        if (cudaEventRecord(lane->fork, s) != cudaSuccess ||
            cudaStreamWaitEvent(lane->copy, lane->fork, 0) != cudaSuccess ||
            cudaMemcpyAsync(X_dev, X_host, x_bytes, cudaMemcpyHostToDevice, lane->copy) !=
                cudaSuccess ||
            cudaEventRecord(lane->x_done, lane->copy) != cudaSuccess)
            return DUST_ERR_CUDA;
    }
    auto join = [&]() {
        return !lane || cudaStreamWaitEvent(s, lane->x_done, 0) == cudaSuccess;
    };
    st = estimate(X_dev, x_dtype, T, d_in, delta_dev, K, d_out, seq_dev, n_seq, seed, kind,
                  draw_begin, sigma, gamma, scale, flags, gw_target, workspace, ws_bytes, stream,
                  lane ? lane->x_done : nullptr);
    if (!join()) return DUST_ERR_CUDA;
    if (st != DUST_OK) return st;
    if (gw_bytes && !direct &&
        cudaMemcpyAsync(gW_host, gW_dev, gw_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DUST_ERR_CUDA;
    return DUST_OK;
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
