// Device primitives shared by the selective-scan kernels (sm_103a).
//
// Workspace header, bounded waits, relaxed/acquire/release global accesses,
// shared-memory barriers (mbarrier) and bulk async copies, all as inline PTX.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ss.h"

namespace ss {

// ------------------------------------------------------------------ workspace
// First 256 bytes of every workspace. Zero-filled by the caller before the
// first launch; every launch leaves it ready for the next one.
struct WsHeader {
    unsigned int epoch;       // tag of the last finished launch (0 = none yet)
    unsigned int ticket;      // next work-unit ticket of the running launch
    unsigned int done;        // CTAs of the running launch that finished
    unsigned int error;       // first device-detected error (ss_status), 0 = none
    unsigned int error_info[4];
    unsigned int pad[56];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kWsHeaderBytes = 256;

// ------------------------------------------------------------------ timing
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ memory order
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// One 32-byte load (4 relaxed 64-bit words, each single-copy atomic on its
// own); p 32-byte aligned.
__device__ __forceinline__ void ld_relaxed_u64x4(const unsigned long long *p, unsigned long long &a,
                                                 unsigned long long &b, unsigned long long &c,
                                                 unsigned long long &d) {
    asm volatile("ld.relaxed.gpu.global.v4.u64 {%0, %1, %2, %3}, [%4];"
                 : "=l"(a), "=l"(b), "=l"(c), "=l"(d) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// L2-coherent load of payload written by another CTA (bypasses L1).
__device__ __forceinline__ float ld_cg_f32(const float *p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_cg_f32x4(const float4 *p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p) : "memory");
    return v;
}

// Tagged 64-bit word: high 32 bits = launch tag, low 32 bits = float payload.
// One aligned 64-bit access is single-copy atomic, so a reader that sees the
// current tag also sees the payload written with it.
__device__ __forceinline__ unsigned long long pack_tagged(unsigned tag, float v) {
    return ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
}
__device__ __forceinline__ unsigned tag_of(unsigned long long w) { return (unsigned)(w >> 32); }
__device__ __forceinline__ float val_of(unsigned long long w) { return __uint_as_float((unsigned)w); }

// ------------------------------------------------------------------ errors
// Keeps the first error of a launch; later ones are dropped.
__device__ __forceinline__ void record_error(WsHeader *ws, unsigned code, unsigned a,
                                             unsigned b, unsigned c) {
    if (atomicCAS(&ws->error, 0u, code) == 0u) {
        ws->error_info[0] = a;
        ws->error_info[1] = b;
        ws->error_info[2] = c;
    }
}

// ------------------------------------------------------------------ end of launch
// Every CTA calls this once, after its last global access of the launch.
// The last CTA to arrive resets the ticket and done counters and publishes
// `tag` as the finished launch's epoch, so the next launch (stream-ordered
// after this one) uses tag + 1 and never confuses old descriptors with new.
__device__ __forceinline__ void finish_launch(WsHeader *ws, unsigned tag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned total = gridDim.x * gridDim.y * gridDim.z;
        const unsigned prev = atomicAdd(&ws->done, 1u);
        if (prev == total - 1u) {
            ws->ticket = 0u;
            ws->done = 0u;
            __threadfence();
            atomicExch(&ws->epoch, tag);
        }
    }
}

// Takes the CTA's work-unit ticket and the launch tag (thread 0), and
// broadcasts both. Tickets are handed out in the order CTAs start, so every
// lower ticket belongs to a CTA that is running or finished. The modulo keeps
// the ticket inside the grid even if the workspace was not zero-filled as
// required (results are then undefined, but every access stays in bounds and
// every wait is bounded).
__device__ __forceinline__ void take_ticket(WsHeader *ws, unsigned &ticket, unsigned &tag) {
    __shared__ unsigned s_ticket, s_tag;
    if (threadIdx.x == 0) {
        s_ticket = atomicAdd(&ws->ticket, 1u) % (gridDim.x * gridDim.y * gridDim.z);
        s_tag = ld_relaxed_u32(&ws->epoch) + 1u;
    }
    __syncthreads();
    ticket = s_ticket;
    tag = s_tag;
}

// ------------------------------------------------------------------ mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// Plain arrival (release at CTA scope: this thread's earlier writes are
// visible to threads that observe the phase completing).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Bulk (non-tensor) async copy global -> shared, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// 2D tile copy global -> shared through a tensor map, completing on `bar`.
// x (innermost coordinate) times the element size must be a multiple of 16
// bytes; dst 128-byte aligned.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y),
          "r"(smem_addr(bar)) : "memory");
}

// Waits for phase `parity` of `bar` for at most `timeout_ns`. Returns false
// on timeout (the copies it tracks may still be in flight).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
    return true;
}

// 3D tile copy global -> shared through a tensor map, completing on `bar`.
// Coordinates (x, y, z) innermost first; boxes reaching past the tensor's
// extent arrive zero-filled. dst 128-byte aligned.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z),
          "r"(smem_addr(bar)) : "memory");
}
// 3D tile copy shared -> global through a tensor map (bulk async-group);
// elements of the box outside the tensor's extent are not written. Writers
// of the tile must have executed fence_proxy_async_smem() and synchronised
// with the issuing thread first.
__device__ __forceinline__ void tma_store_3d(const void *tmap, const void *src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N bulk groups of this thread are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ dependent launches
// Lets the next kernel of the stream, if launched as a programmatic dependent,
// start its prologue while this one runs.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the grids this one depends on have finished and their memory
// is visible (returns at once for an ordinary launch).
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ cp.async (LDGSTS)
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, unsigned src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_4(void *dst, const void *src, unsigned src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ MUFU
// 2^x on the special-function unit (flush-to-zero for subnormal results).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace ss
