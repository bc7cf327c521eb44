// Projection GEMM of the selective-scan layer on the 5th-generation tensor
// cores: P = x W^T, plus a bias on the first n_bias columns, bf16 inputs,
// fp32 accumulation in tensor memory, one rounding to bf16 at the end.
//
// "POPCORNBENCH FW-GLM-5-1 l2_p30", the model's parameters and forward pass:
// proj_delta is a linear projection with a bias, proj_B and proj_C are
// projections without one, and the page asks for the three to be computed
// together. Stacking their weights (D + 2N rows of D) makes them one GEMM
// whose output row m is (pre-activation, B_t, C_t) of step m. A bf16 Linear
// layer adds its bias to the fp32 accumulator and rounds once; the epilogue
// here does the same.
//
// Kernel (persistent, one CTA per SM, warp-specialised, 6 warps):
//   warp 0    TMA producer: the A tile (128 rows of x) and the B tile (BN
//             rows of W, or half of them in a pair) of each 128-column
//             K-block, as two 64-column boxes each, into a ring of
//             shared-memory stages, both K-major with the 128-byte swizzle
//             (one 128-byte row per box row, 8-row atoms of 1 KB);
//   warp 1    allocates 512 columns of tensor memory (two fp32 accumulators
//             of 128 lanes x 256 columns) and, from one thread, issues
//             tcgen05.mma (M = 128, or 256 in a pair; N = BN, K = 16 per
//             instruction, eight per K-block); tcgen05.commit frees each
//             stage when its MMAs have
//             read it and hands a finished accumulator to the epilogue;
//   warps 2-5 epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
//             (tile rows), 32 columns per tcgen05.ld, adds the bias, rounds
//             to bf16 and writes the 32 x 32 chunk to shared memory, from
//             where one TMA tile store sends it to global memory.
// With two accumulators the epilogue of one tile runs under the main loop
// of the next. When there are two M-blocks or more, CTAs run in clusters of
// two on neighbouring SMs and share one MMA of M = 256 (cta_group::2): the
// pair takes two M-blocks of the same N-block at a time, each CTA loads its
// own x tile and its half of the W tile (so a stage is A + BN/2 rows and
// each W byte leaves L2 once per pair), and the leader's one thread issues
// MMAs that read both CTAs' shared memory and accumulate into both CTAs'
// tensor memory (each its 128 rows, all BN columns). Both CTAs' tile copies
// complete on the leader's stage barrier (which the leader arms for the
// pair's bytes); the leader's commits arrive on both CTAs' barriers (stage
// free, accumulator full) and the epilogue warps of both release an
// accumulator on the leader's barrier. Halving the W rows each SM stages and reads
// halves the shared-memory traffic of W, which with M = 128 MMAs per SM
// competes with the operand reads of the tensor cores. Pairs take
// (M-block pair, N-block) tiles round-robin, so the pairs working at one
// time share their x tiles through L2; W stays in L2 throughout.
//
// Every wait is bounded: on timeout the CTA records SS_ERR_TIMEOUT in the
// workspace header, every role leaves its loop, the producer waits (bounded)
// for the copies it issued, the MMA thread waits (bounded) for its MMAs, and
// tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr int kBM = 128;          // tile rows (UMMA M)
constexpr int kBK = 64;           // K-box: 64 bf16 = one 128-byte swizzled row
constexpr int kSub = 2;           // K-boxes per stage: 128 K-columns per barrier round trip
constexpr int kUmmaK = 16;        // K per tcgen05.mma with 16-bit inputs
constexpr int kMaxBN = 256;       // UMMA N limit for M = 128
constexpr int kAccCols = 256;     // tensor-memory columns per accumulator
constexpr int kAccs = 2;          // accumulators (the epilogue of one tile under the next's MMAs)
constexpr int kTmemCols = kAccs * kAccCols;
constexpr int kThreads = 192;     // producer warp, MMA warp, 4 epilogue warps
constexpr int kMaxStages = 8;
constexpr size_t kATileBytes = (size_t)kBM * kBK * 2;  // 16 KB
constexpr size_t kSmemBudget = 224 * 1024;             // dynamic, incl. 1 KB alignment slack
constexpr size_t kStagingBytes = 4 * 2 * 32 * 32 * 2;  // epilogue: 2 buffers of 32 x 32 bf16 per warp
constexpr int64_t kMaxExtent = 0x7fffff00LL;  // M, K, Nout: int32 tile coordinates stay in range

struct GemmParams {
    CUtensorMap tm_a;    // x as (K, M) bf16, box (64, 128), 128-byte swizzle
    CUtensorMap tm_b;    // W as (K, Nout) bf16, box (64, BN), 128-byte swizzle
    CUtensorMap tm_out;  // out as (Nout, M) bf16, row stride ld_out, box (32, 32), 64-byte swizzle
    __nv_bfloat16 *out;  // (M, ld_out) row-major
    const float *bias;   // (n_bias,) or null
    long long M;
    long long ld_out;
    long long num_tiles;
    WsHeader *ws;
    unsigned long long timeout_ns;
    int Nout, K, BN, n_bias;
    int stages, k_blocks, n_tiles_n;
    unsigned idesc;      // tcgen05 instruction descriptor (kind::f16)
};

struct GemmShared {
    uint64_t full[kMaxStages];   // stage s holds its K-block (TMA complete_tx)
    uint64_t empty[kMaxStages];  // stage s was read by its MMAs (tcgen05.commit)
    uint64_t acc_full[2];        // accumulator a holds a finished tile
    uint64_t acc_empty[2];       // accumulator a was read by the epilogue (4 warps, 8 in a pair)
    uint64_t drain;              // the MMA thread's last MMAs completed
    uint32_t tmem_base;
    int abort;
};

// ---------------------------------------------------------------- tcgen05 / TMA wrappers
// Shared-memory matrix descriptor of a K-major bf16 tile with the 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte
// offset), leading byte offset unused for this layout, descriptor version 1
// (bits 46-48), swizzle mode 2 (bits 61-63). The tile must start on a
// 1024-byte boundary; the K-step inside a row is taken by advancing the start
// address by 32 bytes (16 elements).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar)) : "memory");
}

// The CTA-pair forms (cta_group::2, one MMA of M = 256 over two SMs). Every
// tcgen05 instruction of a kernel names the same group, so the pair kernel
// uses these for its allocation, MMAs, commits and release throughout.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrives once on `bar`, at the same offset in both CTAs of the pair, when
// every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_addr(bar)), "h"((uint16_t)0x3) : "memory");
}

template <bool TWO> __device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t cols) {
    if constexpr (TWO) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr(dst)), "r"(cols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr(dst)), "r"(cols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
}

template <bool TWO> __device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    if constexpr (TWO)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                     : "memory");
}

// Address of `p` (a shared variable of this CTA) in the CTA of cluster rank
// `rank`, at the same offset.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, unsigned rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t caddr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
    return v;
}

// 2D tile copy into this CTA's `dst`, completing on the barrier at cluster
// address `bar_cluster`, which may be in the other CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const void *tmap, int x, int y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2 [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y),
          "r"(bar_cluster) : "memory");
}

// Arrival on a barrier of either CTA of the cluster, releasing at cluster
// scope (this thread's earlier accesses are ordered before it for threads of
// the other CTA that observe the phase complete).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 2D tile copy shared -> global through a tensor map (clipped at the
// tensor's extent), in this thread's current bulk group.
__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_addr(src)), "r"(x), "r"(y)
                 : "memory");
}

// Waits for phase `parity` of `bar`; false once the CTA is aborting or the
// wait outlived the launch's timeout (which starts the abort).
// `cluster`: the phase is completed by arrivals from the other CTA of the
// pair, whose earlier accesses the waiter must see (acquire at cluster scope).
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, unsigned parity, const GemmParams &p,
                                              GemmShared &sh, unsigned where, bool cluster = false) {
    auto try_wait = [&] {
        return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (try_wait()) return true;
    const uint64_t t0 = globaltimer_ns();
    for (unsigned it = 1;; ++it) {
        if (try_wait()) return true;
        if ((it & 255u) == 0u) {
            if (*reinterpret_cast<volatile int *>(&sh.abort)) return false;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                *reinterpret_cast<volatile int *>(&sh.abort) = 1;
                record_error(p.ws, SS_ERR_TIMEOUT, 5u, where, blockIdx.x);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- kernel
// TWO: clusters of two CTAs running one M = 256 MMA per K-step between them
// (see the top of the file); otherwise every CTA runs its own M = 128 MMAs.
template <bool TWO>
__global__ void __launch_bounds__(kThreads, 1) proj_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ GemmShared sh;
    // stages start on 1024-byte boundaries (the swizzle atom), at the same
    // offsets in both CTAs of a pair (the pair's MMAs address both by the
    // leader's offsets)
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int b_rows = TWO ? p.BN / 2 : p.BN;  // W rows of a stage held by this CTA
    const size_t b_box = (size_t)b_rows * kBK * 2;  // one K-box of this CTA's W rows
    const size_t stage_bytes = kSub * (kATileBytes + b_box);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // work units: (M-block, N-block) tiles, or (M-block pair, N-block) per cluster
    const unsigned rank = TWO ? cluster_rank() : 0u;
    const long long unit0 = TWO ? blockIdx.x / 2 : blockIdx.x;
    const long long unit_step = TWO ? gridDim.x / 2 : gridDim.x;
    auto m_block = [&](long long u) { return TWO ? 2 * (u / p.n_tiles_n) + rank : u / p.n_tiles_n; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sh.acc_full[a], 1);
            mbar_init(&sh.acc_empty[a], TWO ? 8 : 4);  // the epilogue warps (of both CTAs)
        }
        mbar_init(&sh.drain, 1);
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        // a pair allocates collectively: the same columns in both CTAs
        tmem_alloc<TWO>(&sh.tmem_base, kTmemCols);
        tc_fence_before();
    }
    if (TWO)
        cluster_sync();  // both CTAs' barriers initialised, both allocations made
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    bool run = true;
    if (TWO) {
        // the pair's MMAs write both CTAs' tensor memory at the leader's
        // address: a pair whose columns differ does no work (both CTAs see
        // the same two addresses, so both decide alike)
        const uint32_t other = ld_cluster_u32(cluster_addr(&sh.tmem_base, rank ^ 1u));
        if (other != tmem) {
            run = false;
            if (threadIdx.x == 0) record_error(p.ws, SS_ERR_CUDA, 5u, 6u, blockIdx.x);
        }
    }

    if (!run) {
    } else if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            unsigned phase = 0;
            long long issued = 0;
            bool ok = true;
            for (long long u = unit0; ok && u < p.num_tiles; u += unit_step) {
                const int m0 = (int)m_block(u) * kBM;
                const int n0 = (int)(u % p.n_tiles_n) * p.BN;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!wait_or_abort(&sh.empty[stage], phase ^ 1u, p, sh, 1u)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + stage * stage_bytes;
                    if constexpr (TWO) {
                        // both CTAs' copies complete on the leader's barrier,
                        // which the leader arms for the pair's bytes
                        const uint32_t fb = cluster_addr(&sh.full[stage], 0);
                        if (rank == 0)
                            mbar_arrive_expect_tx(&sh.full[stage], 2u * (unsigned)stage_bytes);
#pragma unroll
                        for (int j = 0; j < kSub; ++j) {
                            const int x = (kb * kSub + j) * kBK;
                            tma_load_2d_pair(sa + j * kATileBytes, &p.tm_a, x, m0, fb);
                            tma_load_2d_pair(sa + kSub * kATileBytes + j * b_box, &p.tm_b, x,
                                             n0 + (int)rank * b_rows, fb);
                        }
                    } else {
                        mbar_arrive_expect_tx(&sh.full[stage], (unsigned)stage_bytes);
#pragma unroll
                        for (int j = 0; j < kSub; ++j) {
                            const int x = (kb * kSub + j) * kBK;
                            tma_load_2d(sa + j * kATileBytes, &p.tm_a, x, m0, &sh.full[stage]);
                            tma_load_2d(sa + kSub * kATileBytes + j * b_box, &p.tm_b, x, n0,
                                        &sh.full[stage]);
                        }
                    }
                    ++issued;
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the last copy into each stage has landed before the CTA leaves
            // (immediate unless the CTA is aborting); a pair's copies all
            // complete on the leader's barriers, and the other CTA does not
            // leave before the leader (the cluster barrier at the end)
            const long long first = issued > p.stages ? issued - p.stages : 0;
            if (!TWO || rank == 0)
                for (long long i = first; i < issued; ++i)
                    mbar_wait_bounded(&sh.full[i % p.stages], (unsigned)((i / p.stages) & 1),
                                      p.timeout_ns);
        }
    } else if (warp == 1) {
        if (lane == 0 && (!TWO || rank == 0)) {
            // -------------------------------------------- MMA issuer
            int stage = 0;
            unsigned phase = 0;
            int acc = 0;
            unsigned acc_phase = 0;
            bool ok = true;
            const uint32_t smem0 = smem_addr(smem);
            for (long long u = unit0; ok && u < p.num_tiles; u += unit_step) {
                if (!wait_or_abort(&sh.acc_empty[acc], acc_phase ^ 1u, p, sh, 2u, TWO)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * kAccCols);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    // the stage landed (in a pair: in both CTAs; the copies'
                    // completion on this barrier is what orders their data
                    // before the MMAs, as for a single CTA, so a CTA-scope
                    // wait suffices and measured 1% faster than cluster scope)
                    if (!wait_or_abort(&sh.full[stage], phase, p, sh, 3u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem0 + (uint32_t)(stage * stage_bytes);
                    const uint32_t sb = sa + (uint32_t)(kSub * kATileBytes);
#pragma unroll
                    for (int j = 0; j < kSub; ++j)
#pragma unroll
                        for (int k = 0; k < kBK / kUmmaK; ++k) {
                            const uint64_t ad =
                                sw128_desc(sa + (uint32_t)(j * kATileBytes) + k * kUmmaK * 2);
                            const uint64_t bd =
                                sw128_desc(sb + (uint32_t)(j * b_box) + k * kUmmaK * 2);
                            const uint32_t accum = (kb | j | k) != 0;
                            if constexpr (TWO)
                                umma_bf16_pair(d_tmem, ad, bd, p.idesc, accum);
                            else
                                umma_bf16(d_tmem, ad, bd, p.idesc, accum);
                        }
                    // stage free once these MMAs read it (in both CTAs of a pair)
                    if constexpr (TWO)
                        umma_commit_pair(&sh.empty[stage]);
                    else
                        umma_commit(&sh.empty[stage]);
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // tile done: hand it to the epilogue (of both CTAs)
                if constexpr (TWO)
                    umma_commit_pair(&sh.acc_full[acc]);
                else
                    umma_commit(&sh.acc_full[acc]);
                if (++acc == kAccs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if constexpr (TWO)
                umma_commit_pair(&sh.drain);
            else
                umma_commit(&sh.drain);
            mbar_wait_bounded(&sh.drain, 0u, p.timeout_ns);
        } else if (TWO && lane == 0) {
            // the other CTA of a pair: the leader's MMAs write this CTA's
            // tensor memory, and have completed before it is released
            mbar_wait_bounded(&sh.drain, 0u, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------ epilogue
        // Lane = tile row. Each 32-column chunk is written to one of the
        // warp's two 2 KB staging buffers in shared memory (its 32 rows x 64
        // bytes) and leaves as one TMA tile store, clipped at M and Nout, so
        // whole row segments reach L2 and the lanes move on while the copy
        // runs. The buffer holds the chunk in the store's 64-byte swizzle
        // (16-byte piece q of row r at position q ^ ((r >> 1) & 3)), so the
        // 8 rows of each 16-byte store phase fall in distinct banks.
        const int quarter = warp & 3;  // tensor-memory lanes 32 quarter .. + 31
        uint4 *stg = reinterpret_cast<uint4 *>(smem + (size_t)p.stages * stage_bytes) +
                     (size_t)(warp - 2) * 2 * 128;
        // the accumulator's release goes to the MMA thread's CTA
        const uint32_t acc_empty0 = TWO ? cluster_addr(&sh.acc_empty[0], 0) : 0u;
        unsigned chunk_no = 0;
        int acc = 0;
        unsigned acc_phase = 0;
        for (long long u = unit0; u < p.num_tiles; u += unit_step) {
            // warp-uniform outcome: tcgen05.ld below is warp-collective
            if (!__all_sync(0xffffffffu, wait_or_abort(&sh.acc_full[acc], acc_phase, p, sh, 4u)))
                break;
            tc_fence_after();
            const long long row0 = m_block(u) * kBM + quarter * 32;
            const int n0 = (int)(u % p.n_tiles_n) * p.BN;
            for (int c = 0; c < p.BN; c += 32, ++chunk_no) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kAccCols + c), r);
                const int col0 = n0 + c;
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                if (p.bias && col0 < p.n_bias) {
                    // lane j fetches the bias of column col0 + j (one coalesced
                    // load), every lane takes the 32 values by shuffle
                    const float bj = col0 + lane < p.n_bias ? __ldg(p.bias + col0 + lane) : 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xffffffffu, bj, j);
                }
                uint4 *buf = stg + (chunk_no & 1u) * 128;
                if (lane == 0) bulk_wait_read<1>();  // this buffer's last store has read it
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 w;
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
                    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
                    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
                    w.x = *reinterpret_cast<uint32_t *>(&h0);
                    w.y = *reinterpret_cast<uint32_t *>(&h1);
                    w.z = *reinterpret_cast<uint32_t *>(&h2);
                    w.w = *reinterpret_cast<uint32_t *>(&h3);
                    buf[lane * 4 + (q ^ ((lane >> 1) & 3))] = w;
                }
                fence_proxy_async_smem();  // visible to the tensor copy
                __syncwarp();
                if (lane == 0 && row0 < p.M && col0 < p.Nout) {
                    tma_store_2d(&p.tm_out, buf, col0, (int)row0);
                    bulk_commit();
                }
            }
            // the accumulator is free once every lane's loads have completed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (TWO)
                    mbar_arrive_cluster(acc_empty0 + (uint32_t)(acc * sizeof(uint64_t)));
                else
                    mbar_arrive(&sh.acc_empty[acc]);
            }
            if (++acc == kAccs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait<0>();  // every store has left shared memory
    }
    __syncthreads();
    // neither CTA of a pair releases its tensor memory or leaves while the
    // other may still arrive on its barriers
    if (TWO) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<TWO>(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- planning
struct GemmPlan {
    int BN, n_tiles_n, stages, k_blocks;
    long long num_tiles;  // work units: tiles, or tile pairs when pair
    bool pair;
    size_t smem;
};

GemmPlan plan_gemm(int64_t M, int64_t K, int64_t Nout) {
    GemmPlan g{};
    g.n_tiles_n = (int)((Nout + kMaxBN - 1) / kMaxBN);
    const int64_t per = (Nout + g.n_tiles_n - 1) / g.n_tiles_n;
    g.BN = (int)((per + 31) / 32 * 32);
    g.k_blocks = (int)((K + kSub * kBK - 1) / (kSub * kBK));
    const int64_t m_tiles = (M + kBM - 1) / kBM;
    // pairs need two M-blocks and W half-tiles of whole 8-row swizzle atoms
    g.pair = m_tiles >= 2 && (g.BN / 2) % 8 == 0;
    g.num_tiles = (g.pair ? (m_tiles + 1) / 2 : m_tiles) * g.n_tiles_n;
    // a pair's CTAs each hold half of the W tile
    const size_t stage_bytes = kSub * (kATileBytes + (size_t)(g.pair ? g.BN / 2 : g.BN) * kBK * 2);
    g.stages = (int)std::min<size_t>(kMaxStages, (kSmemBudget - 1024 - kStagingBytes) / stage_bytes);
    g.smem = 1024 + (size_t)g.stages * stage_bytes + kStagingBytes;
    return g;
}

// Per device: the SM count and the pairs that fit at once for the last
// shared-memory size asked for, and the kernels' dynamic shared-memory limit
// (a per-device attribute, only ever raised, so a launch sized under an
// earlier query stays valid). Filled on first use and when the size
// changes, under a lock.
struct LaunchInfo {
    int smem = -1, sms = 0, clusters = 0, smem_limit = 0;
};
constexpr int kMaxDevices = 64;
std::mutex g_info_mutex;
LaunchInfo g_info[kMaxDevices];

ss_status launch_info(size_t smem, LaunchInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_info_mutex);
    LaunchInfo &li = g_info[dev];
    if (li.smem != (int)smem) {
        int sms = 0, clusters = 0;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const int limit = std::max(li.smem_limit, (int)smem);
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms < 2 ||
            cudaFuncSetAttribute(proj_gemm_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, limit) !=
                cudaSuccess ||
            cudaFuncSetAttribute(proj_gemm_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, limit) !=
                cudaSuccess) {
            cudaGetLastError();
            return SS_ERR_CUDA;
        }
        li.smem_limit = limit;
        cfg.gridDim = dim3(2 * (unsigned)(sms / 2), 1, 1);
        if (cudaOccupancyMaxActiveClusters(&clusters, proj_gemm_kernel<true>, &cfg) !=
                cudaSuccess ||
            clusters < 1) {
            cudaGetLastError();
            return SS_ERR_CUDA;
        }
        li.smem = (int)smem;
        li.sms = sms;
        li.clusters = clusters;
    }
    *out = li;
    return SS_OK;
}

}  // namespace

int proj_gemm_describe_plan(int64_t M, int64_t K, int64_t Nout, int64_t *out) {
    if (!out || M <= 0 || K <= 0 || Nout <= 0 || M > kMaxExtent || K > kMaxExtent ||
        Nout > kMaxExtent)
        return -1;
    const GemmPlan g = plan_gemm(M, K, Nout);
    out[0] = g.BN;
    out[1] = g.n_tiles_n;
    out[2] = (int64_t)kSub * kBK;  // K-columns per stage
    out[3] = g.k_blocks;
    out[4] = g.stages;
    out[5] = g.pair ? 1 : 0;
    out[6] = g.num_tiles;
    out[7] = (int64_t)g.smem;
    return 0;
}

bool proj_gemm_supported(const void *x, const void *W, const void *out, int64_t M, int64_t K,
                         int64_t Nout, int64_t ld_out) {
    auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    // tile coordinates are 32-bit and run up to a tile past each extent
    return M > 0 && K > 0 && Nout > 0 && K % 8 == 0 && ld_out % 8 == 0 && ld_out >= Nout &&
           M <= kMaxExtent && K <= kMaxExtent && Nout <= kMaxExtent && al16(x) && al16(W) &&
           al16(out);
}

ss_status proj_gemm_launch(const void *x, const void *W, void *out, const float *bias,
                           int64_t n_bias, int64_t M, int64_t K, int64_t Nout, int64_t ld_out,
                           void *workspace, cudaStream_t stream, unsigned long long timeout_ns) {
    if (!proj_gemm_supported(x, W, out, M, K, Nout, ld_out)) return SS_ERR_UNSUPPORTED;
    const GemmPlan g = plan_gemm(M, K, Nout);
    if (g.stages < 2) return SS_ERR_UNSUPPORTED;
    GemmParams prm;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {(uint32_t)kBK, (uint32_t)kBM};
        if (!encode_tiled_map(&prm.tm_a, x, true, 2, dims, strides, box, 128))
            return SS_ERR_UNSUPPORTED;
    }
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)Nout};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {(uint32_t)kBK, (uint32_t)(g.pair ? g.BN / 2 : g.BN)};
        if (!encode_tiled_map(&prm.tm_b, W, true, 2, dims, strides, box, 128))
            return SS_ERR_UNSUPPORTED;
    }
    {
        const uint64_t dims[2] = {(uint64_t)Nout, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)ld_out * 2};
        const uint32_t box[2] = {32u, 32u};
        if (!encode_tiled_map(&prm.tm_out, out, true, 2, dims, strides, box, 64))
            return SS_ERR_UNSUPPORTED;
    }
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.bias = bias;
    prm.M = M;
    prm.ld_out = ld_out;
    prm.num_tiles = g.num_tiles;
    prm.ws = static_cast<WsHeader *>(workspace);
    prm.timeout_ns = timeout_ns;
    prm.Nout = (int)Nout;
    prm.K = (int)K;
    prm.BN = g.BN;
    prm.n_bias = bias ? (int)std::min<int64_t>(n_bias, Nout) : 0;
    prm.stages = g.stages;
    prm.k_blocks = g.k_blocks;
    prm.n_tiles_n = g.n_tiles_n;
    // kind::f16 descriptor: fp32 accumulator (bits 4-5 = 1), bf16 A and B
    // (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits
    // 17-22, M >> 4 in bits 24-28 (M = 256 for a pair's MMA)
    const unsigned mma_m = g.pair ? 2 * kBM : kBM;
    prm.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((unsigned)(g.BN >> 3) << 17) |
                ((mma_m >> 4) << 24);
    LaunchInfo li;
    const ss_status st = launch_info(g.smem, &li);
    if (st != SS_OK) return st;
    if (!g.pair) {
        const long long grid = std::min<long long>(g.num_tiles, li.sms);
        proj_gemm_kernel<false><<<(unsigned)grid, kThreads, g.smem, stream>>>(prm);
        return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many pairs as can be resident at once, capped by the work
    cfg.gridDim = dim3(2 * (unsigned)std::min<long long>(g.num_tiles, li.clusters), 1, 1);
    if (cudaLaunchKernelEx(&cfg, proj_gemm_kernel<true>, prm) != cudaSuccess) return SS_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace ss
