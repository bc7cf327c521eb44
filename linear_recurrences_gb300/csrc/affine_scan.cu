// Single-pass affine scan h[t] = a[t] * h[t-1] + b[t] with decoupled look-back.
//
// "Selective-scan CUDA kernels" (persus.netlify.app): the recurrence is a
// prefix scan over affine pairs, associative but not commutative; the fastest
// of its designs is a decoupled look-back with a warp-parallel predecessor
// walk and several items per thread scanned in registers. This is a new
// sm_103a kernel built on that idea:
//
//  * one CTA per 4096-element tile; tile ids come from a ticket counter in
//    CTA start order, so every lower tile is running or done;
//  * the tile's a and b are staged into shared memory by two bulk async
//    copies (cp.async.bulk) completing on an mbarrier;
//  * each warp owns 512 consecutive elements as four 128-element stripes;
//    a lane scans its four-element slice of each stripe in registers, then
//    four interleaved warp-shuffle scans and a fold over the 8 warps give
//    the tile aggregate;
//  * the aggregate is published as two tagged 64-bit words; warp 0 walks
//    back 32 predecessors at a time to the nearest tile that has published
//    its inclusive state, and lane 0 applies the aggregates after it to that
//    state one by one, in sequence order;
//  * the tile's inclusive state is published, and each lane re-sweeps its
//    elements from shared memory starting at its carry-in, storing h with
//    coalesced 128-bit stores.
//
// Determinism: a tile publishes I_k = a_k * e_k + b_k (one fma) where e_k is
// the state entering the tile. Applying predecessor aggregates to a state
// with the same fma in sequence order reproduces I_{k-1} bit for bit, no
// matter which earlier tile the walk started from, so e_k == I_{k-1} always
// and every output is independent of scheduling.
#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 16;                 // elements per thread
constexpr int kTile = kThreads * kItems;   // 4096 elements per tile
constexpr int kStripes = kItems / 4;       // float4 slices per thread
constexpr int kWarpElems = 32 * kItems;    // 512 elements per warp
constexpr int kMaxWindows = 8;             // look-back holds up to 256 predecessors
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kCopyTimeoutNs = 2000000000ull;  // bulk-copy completion bound

struct TileDesc {
    unsigned long long agg_a;  // tag | a-part of the tile aggregate
    unsigned long long agg_b;  // tag | b-part of the tile aggregate
    unsigned long long inc;    // tag | state h at the end of the tile
    unsigned long long pad;
};
static_assert(sizeof(TileDesc) == 32, "descriptor is 32 bytes");

struct Pair {
    float a, b;
};

// p then q: x -> q.a * (p.a * x + p.b) + q.b  ==  (p.a*q.a, q.a*p.b + q.b).
__device__ __forceinline__ Pair compose(Pair p, Pair q) {
    return {p.a * q.a, fmaf(q.a, p.b, q.b)};
}
__device__ __forceinline__ float apply(Pair p, float h) { return fmaf(p.a, h, p.b); }

struct AffineParams {
    const float *a;
    const float *b;
    float *h;
    long long n;
    WsHeader *ws;
    TileDesc *desc;
    unsigned long long timeout_ns;
    long long skip_unit;  // test hook: this tile publishes nothing (-1: none)
    int bulk_ok;   // a and b are 16-byte aligned
    int vec_out;   // h is 16-byte aligned
};

// Polls tile t's descriptor until it holds at least an aggregate.
// kind: 2 = inclusive state available (val), 1 = aggregate (agg), 0 = timed out.
__device__ __forceinline__ int poll_desc(const TileDesc *d, unsigned tag, WsHeader *ws,
                                         unsigned long long timeout_ns, float &val, Pair &agg) {
    uint64_t t0 = 0;
    for (unsigned it = 0;; ++it) {
        const unsigned long long inc = ld_relaxed_u64(&d->inc);
        if (tag_of(inc) == tag) {
            val = val_of(inc);
            return 2;
        }
        const unsigned long long wa = ld_relaxed_u64(&d->agg_a);
        const unsigned long long wb = ld_relaxed_u64(&d->agg_b);
        if (tag_of(wa) == tag && tag_of(wb) == tag) {
            agg = {val_of(wa), val_of(wb)};
            return 1;
        }
        if (it == 0) {
            t0 = globaltimer_ns();
        } else if ((it & 63u) == 0u) {
            if (globaltimer_ns() - t0 > timeout_ns || ld_relaxed_u32(&ws->error) != 0u)
                return 0;
        }
    }
}

__global__ void __launch_bounds__(kThreads)
affine_scan_kernel(const AffineParams p) {
    __shared__ __align__(128) float s_a[kTile];
    __shared__ __align__(128) float s_b[kTile];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ Pair s_warp[kWarps];
    __shared__ Pair s_walk[kMaxWindows * 32];
    __shared__ float s_carry;

    unsigned tile, tag;
    take_ticket(p.ws, tile, tag);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const long long base = (long long)tile * kTile;
    const long long rem = p.n - base;
    const int valid = rem >= kTile ? kTile : (int)rem;

    // ---- load: stage a and b of the tile in shared memory
    if (p.bulk_ok && valid == kTile) {
        if (tid == 0) {
            mbar_init(&s_bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            mbar_arrive_expect_tx(&s_bar, 2u * kTile * sizeof(float));
            bulk_g2s(s_a, p.a + base, kTile * sizeof(float), &s_bar);
            bulk_g2s(s_b, p.b + base, kTile * sizeof(float), &s_bar);
        }
        if (!mbar_wait_bounded(&s_bar, 0, kCopyTimeoutNs)) {
            record_error(p.ws, SS_ERR_TIMEOUT, 1u, tile, 0u);
            // wait once more so no copy is still writing when the CTA leaves
            mbar_wait_bounded(&s_bar, 0, kCopyTimeoutNs);
        }
    } else {
        // ragged last tile or unaligned inputs: plain loads, identity padding
        for (int i = tid; i < kTile; i += kThreads) {
            const bool in = i < valid;
            s_a[i] = in ? p.a[base + i] : 1.0f;
            s_b[i] = in ? p.b[base + i] : 0.0f;
        }
        __syncthreads();
    }

    // ---- thread scan: aggregate of each four-element slice
    Pair st[kStripes];
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const int off = warp * kWarpElems + j * 128 + lane * 4;
        const float4 va = *reinterpret_cast<const float4 *>(&s_a[off]);
        const float4 vb = *reinterpret_cast<const float4 *>(&s_b[off]);
        Pair q = {va.x, vb.x};
        q = compose(q, {va.y, vb.y});
        q = compose(q, {va.z, vb.z});
        q = compose(q, {va.w, vb.w});
        st[j] = q;
    }

    // ---- warp scans over lanes, one per stripe (left operand = earlier lane)
    Pair inc[kStripes];
#pragma unroll
    for (int j = 0; j < kStripes; ++j) inc[j] = st[j];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < kStripes; ++j) {
            const float pa = __shfl_up_sync(kFull, inc[j].a, off);
            const float pb = __shfl_up_sync(kFull, inc[j].b, off);
            if (lane >= off) inc[j] = compose({pa, pb}, inc[j]);
        }
    }
    Pair ex[kStripes];    // exclusive prefix of this lane within stripe j
    Pair qpre[kStripes];  // composition of the warp's earlier stripes
    Pair wagg = {1.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const float ea = __shfl_up_sync(kFull, inc[j].a, 1);
        const float eb = __shfl_up_sync(kFull, inc[j].b, 1);
        ex[j] = lane == 0 ? Pair{1.0f, 0.0f} : Pair{ea, eb};
        const Pair tot = {__shfl_sync(kFull, inc[j].a, 31), __shfl_sync(kFull, inc[j].b, 31)};
        qpre[j] = wagg;
        wagg = compose(wagg, tot);
    }
    if (lane == 0) s_warp[warp] = wagg;
    __syncthreads();

    // ---- block: this warp's exclusive prefix and the tile aggregate
    Pair rpre = {1.0f, 0.0f};
    for (int w = 0; w < warp; ++w) rpre = compose(rpre, s_warp[w]);

    Pair tagg = {1.0f, 0.0f};
    const bool publish = (long long)tile != p.skip_unit;
    if (tid == 0) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tagg = compose(tagg, s_warp[w]);
        TileDesc *d = p.desc + tile;
        if (publish) {
            st_relaxed_u64(&d->agg_a, pack_tagged(tag, tagg.a));
            st_relaxed_u64(&d->agg_b, pack_tagged(tag, tagg.b));
            if (tile == 0) st_relaxed_u64(&d->inc, pack_tagged(tag, tagg.b));
        }
    }

    // ---- look-back (warp 0)
    if (warp == 0) {
        float e = 0.0f;
        if (tile > 0) {
            int win = 0;
            int anchor_lane = -1;
            float anchor = 0.0f;
            bool timed_out = false;
            const uint64_t walk_t0 = globaltimer_ns();
            for (;;) {
                const long long t = (long long)tile - 32LL * (win + 1) + lane;
                int kind;
                float v = 0.0f;
                Pair g = {1.0f, 0.0f};
                if (t < 0) {
                    kind = 2;  // the state before tile 0 is h[-1] = 0
                } else {
                    kind = poll_desc(p.desc + t, tag, p.ws, p.timeout_ns, v, g);
                }
                s_walk[win * 32 + lane] = g;
                const unsigned bad = __ballot_sync(kFull, kind == 0);
                if (bad) {
                    timed_out = true;
                    break;
                }
                const unsigned incs = __ballot_sync(kFull, kind == 2);
                if (incs) {
                    anchor_lane = 31 - __clz(incs);
                    anchor = __shfl_sync(kFull, v, anchor_lane);
                    break;
                }
                if (win + 1 < kMaxWindows) {
                    ++win;
                } else if (globaltimer_ns() - walk_t0 > p.timeout_ns ||
                           ld_relaxed_u32(&p.ws->error) != 0u) {
                    timed_out = true;  // oldest window never showed an inclusive state
                    break;
                }  // else poll the oldest window again
            }
            __syncwarp();
            if (timed_out) {
                if (lane == 0) record_error(p.ws, SS_ERR_TIMEOUT, 2u, tile, (unsigned)win);
            } else if (lane == 0) {
                // anchor state, then the aggregates after it, oldest first
                float s = anchor;
                for (int i = win * 32 + anchor_lane + 1; i < win * 32 + 32; ++i) s = apply(s_walk[i], s);
                for (int w = win - 1; w >= 0; --w) {
                    const Pair *q = s_walk + w * 32;
#pragma unroll 8
                    for (int i = 0; i < 32; ++i) s = apply(q[i], s);
                }
                e = s;
            }
        }
        if (lane == 0) {
            s_carry = e;
            if (tile > 0 && publish)
                st_relaxed_u64(&p.desc[tile].inc, pack_tagged(tag, apply(tagg, e)));
        }
    }
    __syncthreads();

    // ---- fix-up: re-sweep each slice from its carry-in, store h
    const float ew = apply(rpre, s_carry);
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const int off = warp * kWarpElems + j * 128 + lane * 4;
        const float4 va = *reinterpret_cast<const float4 *>(&s_a[off]);
        const float4 vb = *reinterpret_cast<const float4 *>(&s_b[off]);
        float4 o;
        float s = apply(ex[j], apply(qpre[j], ew));
        o.x = s = fmaf(va.x, s, vb.x);
        o.y = s = fmaf(va.y, s, vb.y);
        o.z = s = fmaf(va.z, s, vb.z);
        o.w = fmaf(va.w, s, vb.w);
        const long long g = base + off;
        if (p.vec_out && off + 4 <= valid) {
            __stcs(reinterpret_cast<float4 *>(p.h + g), o);
        } else {
            if (off + 0 < valid) p.h[g + 0] = o.x;
            if (off + 1 < valid) p.h[g + 1] = o.y;
            if (off + 2 < valid) p.h[g + 2] = o.z;
            if (off + 3 < valid) p.h[g + 3] = o.w;
        }
    }

    finish_launch(p.ws, tag);
}

}  // namespace

size_t affine_workspace_bytes(int64_t n) {
    if (n <= 0) return 0;
    const int64_t tiles = (n + kTile - 1) / kTile;
    return kWsHeaderBytes + (size_t)tiles * sizeof(TileDesc);
}

ss_status affine_launch(const float *a, const float *b, float *h, int64_t n, void *workspace,
                        cudaStream_t stream, unsigned long long timeout_ns, long long skip_unit) {
    const int64_t tiles = (n + kTile - 1) / kTile;
    if (tiles > 0x7fffffffLL) return SS_ERR_UNSUPPORTED;
    AffineParams prm;
    prm.a = a;
    prm.b = b;
    prm.h = h;
    prm.n = n;
    prm.ws = reinterpret_cast<WsHeader *>(workspace);
    prm.desc = reinterpret_cast<TileDesc *>(reinterpret_cast<char *>(workspace) + kWsHeaderBytes);
    prm.timeout_ns = timeout_ns;
    prm.skip_unit = skip_unit;
    prm.bulk_ok = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
    prm.vec_out = (reinterpret_cast<uintptr_t>(h) & 15u) == 0;
    affine_scan_kernel<<<(unsigned)tiles, kThreads, 0, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace ss
