// Replay of repeated identical estimator calls as CUDA graphs.
//
// One estimator call issues a memset and three to five kernels; on the host
// that is about 20 microseconds, and small layers are launch-bound (64 x 64,
// 256 tokens: 35.8 -> 32.6 us per synchronised call with graphs). A call
// whose every argument matches an earlier one is captured once into a graph
// and afterwards launched with a single cudaGraphLaunch. The
// graph holds the same pointers and scalars, so it reads the buffers' current
// contents and is exactly the work the direct launches would do.
#include <cstddef>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.cuh"

#ifndef DUST_GRAPHS
#define DUST_GRAPHS 1
#endif

namespace dust {

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kMaxEntries = 16;

struct Entry {
    std::vector<unsigned char> key;
    bool captured = false;  // exec is valid
    bool refused = false;   // capture failed once: always launch directly
    cudaGraphExec_t exec = nullptr;
    uint64_t used = 0;
};

struct Cache {
    std::mutex mu;
    bool ready = false;
    cudaError_t err = cudaSuccess;
    cudaStream_t capture = nullptr;
    std::vector<Entry> entries;
    uint64_t tick = 0;
};

Cache g_cache[kMaxDevices];

Entry* find(Cache& c, const void* key, size_t len) {
    for (auto& e : c.entries)
        if (e.key.size() == len && std::memcmp(e.key.data(), key, len) == 0) return &e;
    return nullptr;
}

Entry* insert(Cache& c, const void* key, size_t len) {
    if (c.entries.size() >= kMaxEntries) {
        size_t lru = 0;
        for (size_t i = 1; i < c.entries.size(); ++i)
            if (c.entries[i].used < c.entries[lru].used) lru = i;
        if (c.entries[lru].exec) cudaGraphExecDestroy(c.entries[lru].exec);
        c.entries.erase(c.entries.begin() + static_cast<std::ptrdiff_t>(lru));
    }
    Entry e;
    e.key.assign(static_cast<const unsigned char*>(key),
                 static_cast<const unsigned char*>(key) + len);
    e.used = ++c.tick;
    c.entries.push_back(std::move(e));
    return &c.entries.back();
}

}  // namespace

dust_status graph_call(const void* key, size_t key_len, cudaStream_t stream,
                       dust_status (*enqueue)(const void* ctx, cudaStream_t s), const void* ctx,
                       bool node_priority) {
    if (!DUST_GRAPHS || profiling_on() || stall_injection_pending()) return enqueue(ctx, stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return enqueue(ctx, stream);
    Cache& c = g_cache[dev];
    std::unique_lock<std::mutex> lock(c.mu);
    Entry* e = find(c, key, key_len);
    if (!e) {  // first sight of these arguments: direct launches
        insert(c, key, key_len);
        lock.unlock();
        return enqueue(ctx, stream);
    }
    e->used = ++c.tick;
    if (e->refused) {
        lock.unlock();
        return enqueue(ctx, stream);
    }
    if (!e->captured) {
        if (!c.ready) {
            c.err = cudaStreamCreateWithFlags(&c.capture, cudaStreamNonBlocking);
            c.ready = true;
        }
        cudaGraph_t graph = nullptr;
        cudaGraphExec_t exec = nullptr;
        bool ok = c.err == cudaSuccess &&
                  cudaStreamBeginCapture(c.capture, cudaStreamCaptureModeThreadLocal) ==
                      cudaSuccess;
        if (ok) {
            const dust_status st = enqueue(ctx, c.capture);
            // End the capture whatever happened, so the stream leaves capture mode.
            const cudaError_t end = cudaStreamEndCapture(c.capture, &graph);
            ok = st == DUST_OK && end == cudaSuccess && graph != nullptr &&
                 cudaGraphInstantiateWithFlags(
                     &exec, graph,
                     node_priority ? cudaGraphInstantiateFlagUseNodePriority : 0) == cudaSuccess;
        }
        if (graph) cudaGraphDestroy(graph);
        if (!ok) {
            (void)cudaGetLastError();
            if (exec) cudaGraphExecDestroy(exec);
            e->refused = true;
            lock.unlock();
            return enqueue(ctx, stream);
        }
        e->exec = exec;
        e->captured = true;
    }
    return cudaGraphLaunch(e->exec, stream) == cudaSuccess ? DUST_OK : DUST_ERR_CUDA;
}

}  // namespace dust
