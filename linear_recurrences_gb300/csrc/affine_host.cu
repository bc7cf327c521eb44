// Affine scan of host arrays, pipelined through device slots.
//
// "Selective-scan CUDA kernels" (opening paragraphs): the recurrence
// h[t] = a[t] h[t-1] + b[t] may be cut anywhere; the second part is the
// same recurrence started from the first part's last state. Chunks of the
// host input are copied into one of kSlots device slots (a, b, h each),
// scanned there from the previous chunk's last output and copied back. The
// copies towards the device run on one stream, the scans on the caller's
// stream and the copies back on a third, so both directions of the host
// link and the GPU are busy at once; events order the reuse of each slot.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr int kSlots = 3;
constexpr int64_t kChunk = 1LL << 23;  // elements per chunk (32 MB per array)
constexpr int kMaxDevices = 64;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Copy streams and events of one device, created on first use and kept for
// the life of the process.
struct Pipe {
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t loaded[kSlots] = {}, scanned[kSlots] = {}, drained[kSlots] = {};
};
std::mutex g_mu;
Pipe g_pipes[kMaxDevices];

// Releases whatever a failed make_pipe created, leaving p as it started.
void drop_pipe(Pipe &p) {
    cudaEvent_t *evs[] = {&p.start, &p.done};
    for (cudaEvent_t *e : evs)
        if (*e) cudaEventDestroy(*e);
    for (int s = 0; s < kSlots; ++s) {
        if (p.loaded[s]) cudaEventDestroy(p.loaded[s]);
        if (p.scanned[s]) cudaEventDestroy(p.scanned[s]);
        if (p.drained[s]) cudaEventDestroy(p.drained[s]);
    }
    if (p.up) cudaStreamDestroy(p.up);
    if (p.down) cudaStreamDestroy(p.down);
    cudaGetLastError();
    p = Pipe{};
}

bool make_pipe(Pipe &p) {
    const unsigned ev = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.done, ev) == cudaSuccess;
    for (int s = 0; ok && s < kSlots; ++s)
        ok = cudaEventCreateWithFlags(&p.loaded[s], ev) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.scanned[s], ev) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.drained[s], ev) == cudaSuccess;
    if (!ok) {
        drop_pipe(p);
        return false;
    }
    p.ready = true;
    return true;
}

struct HostPlan {
    int64_t chunk;   // elements per chunk (the last may be shorter)
    size_t scan_ws;  // bytes of the scan's workspace (first in the workspace)
    size_t slot;     // bytes of one array of one slot
    size_t total;
};

HostPlan host_plan(int64_t n) {
    HostPlan pl{};
    pl.chunk = std::min<int64_t>(n, kChunk);
    pl.scan_ws = align256(affine_workspace_bytes(pl.chunk));
    pl.slot = align256((size_t)pl.chunk * sizeof(float));
    pl.total = pl.scan_ws + (size_t)3 * kSlots * pl.slot;
    return pl;
}

}  // namespace

size_t affine_host_workspace_bytes(int64_t n) {
    if (n <= 0) return 0;
    return host_plan(n).total;
}

ss_status affine_host_launch(const float *a, const float *b, float *h, int64_t n, void *workspace,
                             size_t ws_bytes, cudaStream_t stream, unsigned long long timeout_ns) {
    const HostPlan pl = host_plan(n);
    if (workspace == nullptr || ws_bytes < pl.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SS_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    Pipe &p = g_pipes[dev];
    if (!p.ready && !make_pipe(p)) return SS_ERR_CUDA;

    char *ws = static_cast<char *>(workspace);
    float *sa[kSlots], *sb[kSlots], *sh[kSlots];
    for (int s = 0; s < kSlots; ++s) {
        char *base = ws + pl.scan_ws + (size_t)3 * s * pl.slot;
        sa[s] = reinterpret_cast<float *>(base);
        sb[s] = reinterpret_cast<float *>(base + pl.slot);
        sh[s] = reinterpret_cast<float *>(base + 2 * pl.slot);
    }
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // everything starts after the work already queued on the caller's stream
    if (!ok(cudaEventRecord(p.start, stream)) || !ok(cudaStreamWaitEvent(p.up, p.start, 0)) ||
        !ok(cudaStreamWaitEvent(p.down, p.start, 0)))
        return SS_ERR_CUDA;
    const int64_t chunks = (n + pl.chunk - 1) / pl.chunk;
    for (int64_t k = 0; k < chunks; ++k) {
        const int s = (int)(k % kSlots);
        const int64_t off = k * pl.chunk;
        const int64_t len = std::min<int64_t>(pl.chunk, n - off);
        const size_t bytes = (size_t)len * sizeof(float);
        // slot s's inputs were last read by the scan of chunk k - kSlots
        if (k >= kSlots && !ok(cudaStreamWaitEvent(p.up, p.scanned[s], 0))) return SS_ERR_CUDA;
        if (!ok(cudaMemcpyAsync(sa[s], a + off, bytes, cudaMemcpyDefault, p.up)) ||
            !ok(cudaMemcpyAsync(sb[s], b + off, bytes, cudaMemcpyDefault, p.up)) ||
            !ok(cudaEventRecord(p.loaded[s], p.up)))
            return SS_ERR_CUDA;
        // its output was last read by the copy back of chunk k - kSlots
        if (!ok(cudaStreamWaitEvent(stream, p.loaded[s], 0)) ||
            (k >= kSlots && !ok(cudaStreamWaitEvent(stream, p.drained[s], 0))))
            return SS_ERR_CUDA;
        // chunk k starts from chunk k - 1's last state, still in its slot
        // (the scan that overwrites that slot comes later on this stream)
        const float *h0 = k > 0 ? sh[(k - 1) % kSlots] + (pl.chunk - 1) : nullptr;
        const ss_status st =
            affine_launch(sa[s], sb[s], sh[s], len, ws, stream, timeout_ns, -1, false, h0);
        if (st != SS_OK) return st;
        if (!ok(cudaEventRecord(p.scanned[s], stream)) ||
            !ok(cudaStreamWaitEvent(p.down, p.scanned[s], 0)) ||
            !ok(cudaMemcpyAsync(h + off, sh[s], bytes, cudaMemcpyDefault, p.down)) ||
            !ok(cudaEventRecord(p.drained[s], p.down)))
            return SS_ERR_CUDA;
    }
    // the caller's stream completes after the last copy back
    if (!ok(cudaEventRecord(p.done, p.down)) || !ok(cudaStreamWaitEvent(stream, p.done, 0)))
        return SS_ERR_CUDA;
    return SS_OK;
}

}  // namespace ss
