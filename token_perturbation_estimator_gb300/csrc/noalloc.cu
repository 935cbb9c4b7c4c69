// dust_credit_scan_noalloc: the centring + credit scan with its scratch in a
// fixed device array that ships inside this library, for callers that cannot
// allocate device memory themselves.
//
// Who needs it: code that runs where it is not allowed to own device
// memory, such as a plugin inside a host framework whose pooling allocator
// reserves the whole device up front (a raw cudaMalloc there bypasses the
// pool's accounting and can fail or fragment), or a latency-critical loop in
// which cudaMalloc/cudaFree may synchronise the device. Such a caller still
// provides delta, seq_offsets and r; the scan's chunk summaries live here.
//
// The array (kNoAllocScratchBytes, below) is a static __device__ variable:
// every GPU that loads this part of the library keeps it until the process
// exits. Its device address is looked up once per device, on that device's
// first call, with that device current; make that first call before any
// stream capture. Every call shares the array, so calls whose GPU work
// overlaps (different streams, or different host threads on one device) race
// on it. Each call writes every scratch word it reads, so nothing needs to be
// cleared between calls.
#include <cmath>
#include <mutex>

#include "dust.h"
#include "internal.cuh"

namespace dust {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Bytes of scratch one scan of K draws over T tokens needs: P [T],
// A [n_chunks][K], carry [n_chunks][K], B [n_chunks][2].
size_t noalloc_need(int64_t K, int64_t T) {
    const int64_t nc = (T + kScanChunk - 1) / kScanChunk;
    return round256(sizeof(float) * T) + 2 * round256(sizeof(float) * nc * K) +
           round256(sizeof(float) * 2 * nc);
}

// Device address of g_noalloc_scratch on the current device (nullptr on
// failure), looked up on the first call per device.
unsigned char* noalloc_base() {
    constexpr int kMaxDev = 64;
    static unsigned char* cache[kMaxDev] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        cache[dev] = static_cast<unsigned char*>(p);
    }
    return cache[dev];
}

}  // namespace

}  // namespace dust

using namespace dust;

extern "C" {

size_t dust_credit_scan_noalloc_capacity(void) { return kNoAllocScratchBytes; }

dust_status dust_credit_scan_noalloc(const float* delta, int64_t K, int64_t T,
                                     const int32_t* seq_offsets, int64_t n_seq, float gamma,
                                     uint32_t flags, float* r, void* stream) {
    if (K < 1 || T < 0 || n_seq < 0) return DUST_ERR_INVALID_ARG;
    if (K > DUST_MAX_DRAWS) return DUST_ERR_RANGE;
    if (flags & ~DUST_CENTER) return DUST_ERR_INVALID_ARG;
    if (!std::isfinite(gamma) || std::fabs(gamma) > 1.0f) return DUST_ERR_INVALID_ARG;
    if (T > 0 && (n_seq < 1 || n_seq > T)) return DUST_ERR_INVALID_ARG;
    if (T == 0) return DUST_OK;
    if (!delta || !seq_offsets || !r) return DUST_ERR_INVALID_ARG;
    if (noalloc_need(K, T) > kNoAllocScratchBytes) return DUST_ERR_RANGE;
    unsigned char* base = noalloc_base();
    if (!base) return DUST_ERR_CUDA;

    const int64_t nc = (T + kScanChunk - 1) / kScanChunk;
    ScanBuffers b;
    b.n_chunks = nc;
    b.r = r;
    unsigned char* p = base;
    b.P = reinterpret_cast<float*>(p);
    p += round256(sizeof(float) * T);
    b.A = reinterpret_cast<float*>(p);
    p += round256(sizeof(float) * nc * K);
    b.carry = reinterpret_cast<float*>(p);
    p += round256(sizeof(float) * nc * K);
    b.B = reinterpret_cast<float*>(p);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_scan(delta, K, T, seq_offsets, n_seq, gamma,
                                (flags & DUST_CENTER) != 0, b, s);
    if (e == cudaSuccess) e = launch_scan_fixup(b, K, T, s);
    return e == cudaSuccess ? DUST_OK : DUST_ERR_CUDA;
}

}  // extern "C"
