// ss_affine_scan_noalloc: the affine scan with its scratch memory in a static
// device array, for callers that cannot allocate device memory.
//
// The regular entry point takes a caller-provided workspace (descriptor
// words the look-back kernel publishes and polls). Some callers have no way
// to provide one: code running where cudaMalloc is forbidden or unsafe (for
// example inside an allocator, a plugin that must not touch the device heap,
// or a real-time path that may not allocate after start-up). This variant
// uses a fixed array instead, allocated by the CUDA module loader when the
// library is loaded and held by every GPU that loads it until the process
// exits.
//
// The array is shared by every call: it keeps the last call's descriptors,
// whose launch tags make them harmless to the next call. Only the error word
// must start each call at zero (a set word makes the look-back waits give
// up), so each call clears it on its stream; ss_affine_scan_noalloc_status()
// reads the last call's device-detected error from it. Two calls that
// can overlap on the GPU (different streams, or different host threads
// without ordering) race on the array and must not be issued.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "ss.h"
#include "ss_common.cuh"
#include "ss_internal.h"

namespace {

// Header plus one 32-byte descriptor per 4096-element tile, for up to
// SS_AFFINE_NOALLOC_MAX_N elements (zero-filled at module load). Every call
// also checks the scan's own workspace size against it, so a change of the
// tile or descriptor size cannot make a call write past the array.
constexpr size_t kScratchBytes = ss::kWsHeaderBytes + (size_t)(SS_AFFINE_NOALLOC_MAX_N / 4096) * 32;
static __device__ __align__(256) unsigned char g_affine_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};  // device address of g_affine_scratch, per device

// Device address of the scratch array on the current device. The first call
// for a device looks it up (host code cannot use the symbol directly).
ss_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_affine_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return SS_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return SS_OK;
}

}  // namespace

extern "C" ss_status ss_affine_scan_noalloc(const float *a, const float *b, float *h, int64_t n,
                                            void *stream) {
    if (n < 0) return SS_ERR_INVALID;
    if (n == 0) return SS_OK;
    if (n > SS_AFFINE_NOALLOC_MAX_N || ss::affine_workspace_bytes(n) > kScratchBytes)
        return SS_ERR_UNSUPPORTED;
    if (!a || !b || !h) return SS_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
         reinterpret_cast<uintptr_t>(h)) & 3u)
        return SS_ERR_INVALID;
    void *ws = nullptr;
    const ss_status st = scratch_for_current_device(&ws);
    if (st != SS_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // a previous call's error word must not make this call's waits give up
    if (cudaMemsetAsync(&static_cast<ss::WsHeader *>(ws)->error, 0, sizeof(unsigned), s) != cudaSuccess)
        return SS_ERR_CUDA;
    return ss::affine_launch(a, b, h, n, ws, s, ss::spin_timeout_ns(), ss::take_skip_unit());
}

extern "C" ss_status ss_affine_scan_noalloc_status(void *stream) {
    void *ws = nullptr;
    const ss_status st = scratch_for_current_device(&ws);
    if (st != SS_OK) return st;
    return ss_get_device_status(ws, stream);
}
