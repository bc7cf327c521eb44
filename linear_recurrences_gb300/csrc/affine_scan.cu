// Single-pass affine scan h[t] = a[t] * h[t-1] + b[t] with decoupled look-back.
//
// "Selective-scan CUDA kernels" (persus.netlify.app): the recurrence is a
// prefix scan over affine pairs, associative but not commutative; the fastest
// of its designs is a decoupled look-back with a warp-parallel predecessor
// walk and several items per thread scanned in registers. This is a new
// sm_103a kernel built on that idea:
//
//  * a persistent grid (as many CTAs as fit) takes 4096-element tiles from a
//    ticket counter in start order, so every lower tile is running or done;
//    a CTA asks L2 to prefetch each tile when it takes the tile's ticket, a
//    step before the tile is staged into shared memory (prefetching further
//    ahead, or holding tickets further ahead, measured slower);
//  * each CTA owns a ring of kBufs tile buffers in shared memory, filled by
//    two bulk async copies (cp.async.bulk) per tile on an mbarrier, 8 compute
//    warps and one control warp. Per step the compute warps scan the next
//    tile and publish its aggregate while the control warp looks back for the
//    current tile; the compute warps then fix up and store the current tile
//    and refill its buffer with the tile kBufs ahead, and the look-back
//    overlaps the scan;
//  * each warp owns 512 consecutive elements as four 128-element stripes;
//    a lane scans its four-element slice of each stripe in registers, then
//    four interleaved warp-shuffle scans and a fold over the 8 warps give
//    the tile aggregate;
//  * the aggregate is published as two tagged 64-bit words; the control warp
//    walks back 64 predecessors per L2 round trip (each lane reads the whole
//    32-byte descriptors of two tiles, one load each) to the nearest tile
//    that has published its inclusive state, and lane 0 applies the
//    aggregates after it to that state one by one, in sequence order;
//  * the tile's inclusive state is published, and each lane re-sweeps its
//    elements from shared memory starting at its carry-in, storing h with
//    coalesced 128-bit streaming stores.
//
// Determinism: a tile publishes I_k = a_k * e_k + b_k (one fma) where e_k is
// the state entering the tile. Applying predecessor aggregates to a state
// with the same fma in sequence order reproduces I_{k-1} bit for bit, no
// matter which earlier tile the walk started from, so e_k == I_{k-1} always
// and every output is independent of scheduling.
//
// Progress: a CTA holds at most kTicks + 1 tickets (current and the ones after
// it), scanned and published in ticket order. The lowest unfinished tile is
// always some CTA's current tile and every tile below it is finished, so its
// look-back completes.
#include <algorithm>
#include <mutex>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr int kThreads = 256;                // compute threads (8 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kCtaThreads = kThreads + 32;  // plus one control warp
constexpr int kItems = 16;                 // elements per thread
constexpr int kTile = kThreads * kItems;   // 4096 elements per tile
constexpr int kStripes = kItems / 4;       // float4 slices per thread
constexpr int kWarpElems = 32 * kItems;    // 512 elements per warp
constexpr int kMaxWindows = 8;             // look-back holds up to 256 predecessors
constexpr int kPoll = 2;                   // windows polled per round trip
static_assert(kMaxWindows % kPoll == 0, "windows are polled kPoll at a time");
constexpr unsigned kFull = 0xffffffffu;
constexpr int kBufs = 2;                                     // tile buffers per CTA
constexpr int kTicks = kBufs;  // tickets a CTA holds: one per buffer
constexpr size_t kDynSmem = 2 * kBufs * kTile * sizeof(float);  // a and b per buffer
constexpr unsigned long long kCopyTimeoutNs = 2000000000ull;  // bulk-copy completion bound

// 32 bytes, 32-byte aligned (the workspace and the header are), so a poll
// reads a whole descriptor with one load.
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

// Barrier among the 8 compute warps only (the control warp does not take part).
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

// p then q: x -> q.a * (p.a * x + p.b) + q.b  ==  (p.a*q.a, q.a*p.b + q.b).
__device__ __forceinline__ Pair compose(Pair p, Pair q) {
    return {p.a * q.a, fmaf(q.a, p.b, q.b)};
}
__device__ __forceinline__ float apply(Pair p, float h) { return fmaf(p.a, h, p.b); }

struct AffineParams {
    const float *a;
    const float *b;
    float *h;
    const float *h0;  // state before element 0 (one float), or null for 0
    long long n;
    WsHeader *ws;
    TileDesc *desc;
    unsigned long long timeout_ns;
    long long skip_unit;  // test hook: this tile publishes nothing (-1: none)
    int bulk_ok;   // a and b are 16-byte aligned
    int vec_out;   // h is 16-byte aligned
};

// Per-tile results of the in-tile scan that the fix-up needs later.
struct TileScan {
    Pair ex[kStripes];    // exclusive prefix of this lane within stripe j
    Pair qpre[kStripes];  // composition of the warp's earlier stripes
    Pair rpre;            // composition of the CTA's earlier warps
    Pair tagg;            // tile aggregate (thread 0 only)
};

// Starts staging tile `tile` into (sa, sb): two bulk copies on `bar` for a
// full tile of aligned inputs, else plain loads with identity padding
// (completed by the barrier that precedes the tile's scan).
__device__ __forceinline__ void stage_tile(const AffineParams &p, unsigned tile, float *sa,
                                           float *sb, uint64_t *bar) {
    const long long base = (long long)tile * kTile;
    const long long rem = p.n - base;
    if (p.bulk_ok && rem >= kTile) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(bar, 2u * kTile * sizeof(float));
            bulk_g2s(sa, p.a + base, kTile * sizeof(float), bar);
            bulk_g2s(sb, p.b + base, kTile * sizeof(float), bar);
        }
    } else {
        const int valid = rem >= kTile ? kTile : (int)rem;
        for (int i = threadIdx.x; i < kTile; i += kThreads) {
            const bool in = i < valid;
            sa[i] = in ? p.a[base + i] : 1.0f;
            sb[i] = in ? p.b[base + i] : 0.0f;
        }
    }
}

// Asks L2 to fetch tile `tile`'s inputs ahead of its staging (full tiles of
// aligned inputs only; the hint changes no data).
__device__ __forceinline__ void prefetch_tile_l2(const AffineParams &p, long long tile) {
    const long long base = tile * kTile;
    if (p.bulk_ok && p.n - base >= kTile) {
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     :: "l"(p.a + base), "r"((unsigned)(kTile * sizeof(float))) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     :: "l"(p.b + base), "r"((unsigned)(kTile * sizeof(float))) : "memory");
    }
}

// Waits for tile `tile`'s data (load number `use` of buffer `bar`), scans it
// and publishes its aggregate. The compute warps call it; the tile aggregate is
// left in *s_tagg for the control warp.
__device__ __forceinline__ void scan_tile(const AffineParams &p, unsigned tile, unsigned tag,
                                          const float *s_a, const float *s_b, uint64_t *bar,
                                          unsigned use, Pair *s_warp, Pair *s_tagg, TileScan &r) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long rem = p.n - (long long)tile * kTile;
    if (p.bulk_ok && rem >= kTile) {
        const unsigned parity = use & 1u;
        if (!mbar_wait_bounded(bar, parity, kCopyTimeoutNs)) {
            record_error(p.ws, SS_ERR_TIMEOUT, 1u, tile, 0u);
            // wait once more so no copy is still writing when the CTA leaves
            mbar_wait_bounded(bar, parity, kCopyTimeoutNs);
        }
    }
    compute_sync();  // plain-loaded tiles: every thread's writes are visible

    // thread scan: aggregate of each four-element slice
    Pair inc[kStripes];
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const int off = warp * kWarpElems + j * 128 + lane * 4;
        const float4 va = *reinterpret_cast<const float4 *>(&s_a[off]);
        const float4 vb = *reinterpret_cast<const float4 *>(&s_b[off]);
        Pair q = {va.x, vb.x};
        q = compose(q, {va.y, vb.y});
        q = compose(q, {va.z, vb.z});
        q = compose(q, {va.w, vb.w});
        inc[j] = q;
    }
    // warp scans over lanes, one per stripe (left operand = earlier lane)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < kStripes; ++j) {
            const float pa = __shfl_up_sync(kFull, inc[j].a, off);
            const float pb = __shfl_up_sync(kFull, inc[j].b, off);
            if (lane >= off) inc[j] = compose({pa, pb}, inc[j]);
        }
    }
    Pair wagg = {1.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const float ea = __shfl_up_sync(kFull, inc[j].a, 1);
        const float eb = __shfl_up_sync(kFull, inc[j].b, 1);
        r.ex[j] = lane == 0 ? Pair{1.0f, 0.0f} : Pair{ea, eb};
        const Pair tot = {__shfl_sync(kFull, inc[j].a, 31), __shfl_sync(kFull, inc[j].b, 31)};
        r.qpre[j] = wagg;
        wagg = compose(wagg, tot);
    }
    if (lane == 0) s_warp[warp] = wagg;
    compute_sync();
    r.rpre = {1.0f, 0.0f};
    for (int w = 0; w < warp; ++w) r.rpre = compose(r.rpre, s_warp[w]);
    r.tagg = {1.0f, 0.0f};
    if (tid == 0) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) r.tagg = compose(r.tagg, s_warp[w]);
        *s_tagg = r.tagg;
        if ((long long)tile != p.skip_unit) {
            TileDesc *d = p.desc + tile;
            st_relaxed_u64(&d->agg_a, pack_tagged(tag, r.tagg.a));
            st_relaxed_u64(&d->agg_b, pack_tagged(tag, r.tagg.b));
            // tile 0's inclusive state; from an initial state the control
            // warp publishes it with the carry instead
            if (tile == 0 && !p.h0) st_relaxed_u64(&d->inc, pack_tagged(tag, r.tagg.b));
        }
    }
    compute_sync();  // s_warp is free for the next tile
}

// ---- comparison variant: a log-step (Hillis-Steele) scan of the tile.
// "Selective-scan CUDA kernels", the predictions: the page's Hillis-Steele
// ran in PyTorch, which it notes is not a fair comparison with its
// single-pass kernel. Here the same persistent look-back kernel runs with
// the tile scanned by the log-step algorithm instead: each thread keeps its
// 16 elements in registers; in step k every element E >= 2^k is combined
// with element E - 2^k as it was after step k-1, the values passing through
// the tile's shared-memory buffer; 12 steps for 4096 elements (work
// O(n log n) instead of O(n)). The tile buffer ends up holding every
// element's inclusive pair from the tile start, and the fix-up is one fma.
__device__ __forceinline__ void scan_tile_hs(const AffineParams &p, unsigned tile, unsigned tag,
                                             float *s_a, float *s_b, uint64_t *bar, unsigned use,
                                             Pair *s_tagg) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long rem = p.n - (long long)tile * kTile;
    if (p.bulk_ok && rem >= kTile) {
        const unsigned parity = use & 1u;
        if (!mbar_wait_bounded(bar, parity, kCopyTimeoutNs)) {
            record_error(p.ws, SS_ERR_TIMEOUT, 1u, tile, 0u);
            mbar_wait_bounded(bar, parity, kCopyTimeoutNs);
        }
    }
    compute_sync();
    float a[kItems], b[kItems];
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const int off = warp * kWarpElems + j * 128 + lane * 4;
        const float4 va = *reinterpret_cast<const float4 *>(&s_a[off]);
        const float4 vb = *reinterpret_cast<const float4 *>(&s_b[off]);
        a[4 * j] = va.x; a[4 * j + 1] = va.y; a[4 * j + 2] = va.z; a[4 * j + 3] = va.w;
        b[4 * j] = vb.x; b[4 * j + 1] = vb.y; b[4 * j + 2] = vb.z; b[4 * j + 3] = vb.w;
    }
    for (int o = 1; o < kTile; o <<= 1) {
        float pa[kItems], pb[kItems];  // element E - o after the previous step
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            const int E = warp * kWarpElems + (k >> 2) * 128 + lane * 4 + (k & 3);
            pa[k] = E >= o ? s_a[E - o] : 1.0f;
            pb[k] = E >= o ? s_b[E - o] : 0.0f;
        }
        compute_sync();  // every partner is read before any is overwritten
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            const Pair c = compose({pa[k], pb[k]}, {a[k], b[k]});
            a[k] = c.a;
            b[k] = c.b;
        }
#pragma unroll
        for (int j = 0; j < kStripes; ++j) {
            const int off = warp * kWarpElems + j * 128 + lane * 4;
            *reinterpret_cast<float4 *>(&s_a[off]) = make_float4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
            *reinterpret_cast<float4 *>(&s_b[off]) = make_float4(b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
        }
        compute_sync();  // this step's values are in place
    }
    if (tid == 0) {
        const Pair tagg = {s_a[kTile - 1], s_b[kTile - 1]};
        *s_tagg = tagg;
        if ((long long)tile != p.skip_unit) {
            TileDesc *d = p.desc + tile;
            st_relaxed_u64(&d->agg_a, pack_tagged(tag, tagg.a));
            st_relaxed_u64(&d->agg_b, pack_tagged(tag, tagg.b));
            if (tile == 0 && !p.h0) st_relaxed_u64(&d->inc, pack_tagged(tag, tagg.b));
        }
    }
}

// Fix-up of the log-step variant: h = A_E * carry + B_E from the tile
// buffer's inclusive pairs.
__device__ __forceinline__ void fix_up_hs(const AffineParams &p, unsigned tile, const float *s_a,
                                          const float *s_b, float carry) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long base = (long long)tile * kTile;
    const long long rem = p.n - base;
    const int valid = rem >= kTile ? kTile : (int)rem;
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const int off = warp * kWarpElems + j * 128 + lane * 4;
        const float4 va = *reinterpret_cast<const float4 *>(&s_a[off]);
        const float4 vb = *reinterpret_cast<const float4 *>(&s_b[off]);
        const float4 o = make_float4(fmaf(va.x, carry, vb.x), fmaf(va.y, carry, vb.y),
                                     fmaf(va.z, carry, vb.z), fmaf(va.w, carry, vb.w));
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
}

// Control warp: the state entering `tile` (nearest published inclusive state,
// then the aggregates after it applied in sequence order); publishes the
// tile's inclusive state and leaves the carry in *s_carry.
// Windows of 32 predecessors are polled nearest first (lane l holds tile
// tile - 32(w+1) + l); the walk stops at the first window holding an
// inclusive state, after every tile above it has shown its aggregate.
__device__ __forceinline__ void look_back(const AffineParams &p, unsigned tile, unsigned tag,
                                          const Pair &tagg, Pair *s_walk, float *s_carry) {
    const int lane = threadIdx.x & 31;
    float e = 0.0f;
    if (tile == 0) {
        if (p.h0) e = *p.h0;
    } else {
        int win = 0;
        int anchor_lane = -1;
        float anchor = 0.0f;
        bool timed_out = false;
        const uint64_t walk_t0 = globaltimer_ns();
        for (;;) {
            // kPoll windows per round trip: lane l polls tiles
            // tile - 32(win + 1 + i) + l, i < kPoll
            int kind[kPoll];  // 0 nothing yet, 1 aggregate, 2 inclusive state
            float v[kPoll];
            Pair g[kPoll];
#pragma unroll
            for (int i = 0; i < kPoll; ++i) {
                // before tile 0: the state h[-1] counts as inclusive (0 here,
                // h0 substituted once the anchor is chosen)
                kind[i] = (long long)tile - 32LL * (win + 1 + i) + lane < 0 ? 2 : 0;
                v[i] = 0.0f;
                g[i] = {1.0f, 0.0f};
            }
            for (unsigned it = 0;; ++it) {
                unsigned long long wi[kPoll], wa[kPoll], wb[kPoll];
#pragma unroll
                for (int i = 0; i < kPoll; ++i) {  // every word in flight at once
                    if (kind[i] == 0) {
                        const TileDesc *d = p.desc + (tile - 32LL * (win + 1 + i) + lane);
                        unsigned long long pad;
                        ld_relaxed_u64x4(&d->agg_a, wa[i], wb[i], wi[i], pad);
                    }
                }
                bool pending = false;
#pragma unroll
                for (int i = 0; i < kPoll; ++i) {
                    if (kind[i] == 0) {
                        if (tag_of(wi[i]) == tag) {
                            v[i] = val_of(wi[i]);
                            kind[i] = 2;
                        } else if (tag_of(wa[i]) == tag && tag_of(wb[i]) == tag) {
                            g[i] = {val_of(wa[i]), val_of(wb[i])};
                            kind[i] = 1;
                        } else {
                            pending = true;
                        }
                    }
                }
                if (!pending) break;
                if ((it & 63u) == 63u &&
                    (globaltimer_ns() - walk_t0 > p.timeout_ns || ld_relaxed_u32(&p.ws->error) != 0u))
                    break;  // a kind stays 0: gave up
            }
            bool gave_up = false;
#pragma unroll
            for (int i = 0; i < kPoll; ++i) {
                s_walk[(win + i) * 32 + lane] = g[i];
                gave_up |= kind[i] == 0;
            }
            if (__ballot_sync(kFull, gave_up)) {
                timed_out = true;
                break;
            }
            bool found = false;
#pragma unroll
            for (int i = 0; i < kPoll; ++i) {
                const unsigned incs = __ballot_sync(kFull, kind[i] == 2);
                if (!found && incs) {  // nearest window holding an inclusive state
                    win += i;
                    anchor_lane = 31 - __clz(incs);
                    anchor = __shfl_sync(kFull, v[i], anchor_lane);
                    found = true;
                }
            }
            if (found) {
                if (p.h0 && (long long)tile - 32LL * (win + 1) + anchor_lane < 0) anchor = *p.h0;
                break;
            }
            if (win + kPoll < kMaxWindows) {
                win += kPoll;
            } else if (globaltimer_ns() - walk_t0 > p.timeout_ns ||
                       ld_relaxed_u32(&p.ws->error) != 0u) {
                timed_out = true;  // oldest windows never showed an inclusive state
                break;
            }  // else poll the oldest windows again
        }
        __syncwarp();
        if (timed_out) {
            if (lane == 0) record_error(p.ws, SS_ERR_TIMEOUT, 2u, tile, (unsigned)win);
        } else if (lane == 0) {
            // anchor state, then the aggregates after it, oldest first; one
            // fma per aggregate with operands fetched ahead
            float s = anchor;
            {
                const float4 *q = reinterpret_cast<const float4 *>(s_walk + win * 32);
                float4 v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = q[i];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (2 * i > anchor_lane) s = fmaf(v[i].x, s, v[i].y);
                    if (2 * i + 1 > anchor_lane) s = fmaf(v[i].z, s, v[i].w);
                }
            }
            for (int w = win - 1; w >= 0; --w) {
                const float4 *q = reinterpret_cast<const float4 *>(s_walk + w * 32);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float4 v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = q[4 * c + i];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        s = fmaf(v[i].x, s, v[i].y);
                        s = fmaf(v[i].z, s, v[i].w);
                    }
                }
            }
            e = s;
        }
    }
    if (lane == 0) {
        *s_carry = e;
        if ((tile > 0 || p.h0) && (long long)tile != p.skip_unit)
            st_relaxed_u64(&p.desc[tile].inc, pack_tagged(tag, apply(tagg, e)));
    }
    __syncwarp();
}

// Re-sweeps each lane's slices of `tile` from the carry-in and stores h.
__device__ __forceinline__ void fix_up(const AffineParams &p, unsigned tile, const float *s_a,
                                       const float *s_b, const TileScan &r, float carry) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long base = (long long)tile * kTile;
    const long long rem = p.n - base;
    const int valid = rem >= kTile ? kTile : (int)rem;
    const float ew = apply(r.rpre, carry);
#pragma unroll
    for (int j = 0; j < kStripes; ++j) {
        const int off = warp * kWarpElems + j * 128 + lane * 4;
        const float4 va = *reinterpret_cast<const float4 *>(&s_a[off]);
        const float4 vb = *reinterpret_cast<const float4 *>(&s_b[off]);
        float4 o;
        float s = apply(r.ex[j], apply(r.qpre[j], ew));
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
}

// Shared state of one CTA of the affine-scan kernel.
struct AffineShared {
    uint64_t bar[kBufs];       // one mbarrier per tile buffer
    Pair warp_agg[kWarps];     // per-warp aggregates of the tile being scanned
    Pair tagg[2];              // tile aggregates handed to the control warp
    unsigned tick[kTicks];     // ticket of CTA-local tile q in tick[q % kTicks]
    unsigned tag;              // this launch's descriptor tag
    float carry;               // state entering the current tile
};

// Control warp: per step, take the ticket of tile q + kTicks (and prefetch it
// to L2), look back for tile q, then meet the compute warps at the step's two
// barriers.
__device__ __forceinline__ void control_loop(const AffineParams &p, AffineShared &sh, Pair *s_walk,
                                             unsigned num_tiles) {
    const int lane = threadIdx.x & 31;
    const unsigned tag = sh.tag;
    unsigned cur = sh.tick[0], nxt = sh.tick[1];
    __syncthreads();  // the compute warps' scan of tile 0 (its aggregate) is done
    for (unsigned q = 0; cur < num_tiles; ++q) {
        // ticket first: its round trip overlaps the look-back's polls
        unsigned t = 0;
        if (lane == 0) {
            t = atomicAdd(&p.ws->ticket, 1u);
            if (t < num_tiles) prefetch_tile_l2(p, t);  // staged at the end of this step
        }
        look_back(p, cur, tag, sh.tagg[q & 1], s_walk, &sh.carry);
        if (lane == 0) sh.tick[q % kTicks] = t;  // tile q's slot is no longer read
        __syncthreads();  // carry and ticket are published
        __syncthreads();  // tile q is stored, its buffer restaged
        cur = nxt;
        nxt = sh.tick[(q + 2) % kTicks];
    }
}

// Compute warps: per step, scan tile q + 1 (publishing its aggregate), then
// fix up and store tile q and restage its buffer. Two steps per loop trip so
// the two scan results swap roles without indexing (tile q's results are in
// rc for even q, in rn for odd q).
template <bool HS>
__device__ __forceinline__ void compute_loop(const AffineParams &p, AffineShared &sh, float *s_dyn,
                                             unsigned num_tiles) {
    const unsigned tag = sh.tag;
    auto abuf = [&](unsigned q) { return s_dyn + (q % kBufs) * (2 * kTile); };
    // CTA-local tile q: staged in buffer q % kBufs, its load number q / kBufs
    auto scan = [&](unsigned tile, unsigned q, Pair *tagg, TileScan &r) {
        if constexpr (HS)
            scan_tile_hs(p, tile, tag, abuf(q), abuf(q) + kTile, &sh.bar[q % kBufs], q / kBufs, tagg);
        else
            scan_tile(p, tile, tag, abuf(q), abuf(q) + kTile, &sh.bar[q % kBufs], q / kBufs,
                      sh.warp_agg, tagg, r);
    };
    auto fix = [&](unsigned tile, unsigned q, const TileScan &r) {
        if constexpr (HS)
            fix_up_hs(p, tile, abuf(q), abuf(q) + kTile, sh.carry);
        else
            fix_up(p, tile, abuf(q), abuf(q) + kTile, r, sh.carry);
    };
    unsigned cur = sh.tick[0], nxt = sh.tick[1];
    for (int i = 0; i < kBufs; ++i) {
        const unsigned t = sh.tick[i];
        if (t < num_tiles) stage_tile(p, t, abuf(i), abuf(i) + kTile, &sh.bar[i]);
    }
    TileScan rc, rn;
    if (cur < num_tiles)
        scan(cur, 0, &sh.tagg[0], rc);
    __syncthreads();  // tile 0's aggregate is visible to the control warp
    for (unsigned q = 0; cur < num_tiles; q += 2) {
        if (nxt < num_tiles)
            scan(nxt, q + 1, &sh.tagg[1], rn);
        __syncthreads();
        unsigned after = sh.tick[(q + kBufs) % kTicks];
        fix(cur, q, rc);
        compute_sync();  // tile q's buffer is free
        if (after < num_tiles) stage_tile(p, after, abuf(q), abuf(q) + kTile, &sh.bar[q % kBufs]);
        __syncthreads();
        cur = nxt;
        nxt = sh.tick[(q + 2) % kTicks];
        if (cur >= num_tiles) break;

        const unsigned q1 = q + 1;
        if (nxt < num_tiles)
            scan(nxt, q1 + 1, &sh.tagg[0], rc);
        __syncthreads();
        after = sh.tick[(q1 + kBufs) % kTicks];
        fix(cur, q1, rn);
        compute_sync();
        if (after < num_tiles) stage_tile(p, after, abuf(q1), abuf(q1) + kTile, &sh.bar[q1 % kBufs]);
        __syncthreads();
        cur = nxt;
        nxt = sh.tick[(q1 + 2) % kTicks];
    }
}

// Persistent, software-pipelined, warp-specialised. Each CTA owns a ring of
// kBufs tile buffers, 8 compute warps and one control warp. CTA-local tile
// q (the q-th ticket this CTA took) lives in buffer q % kBufs. Per step q the
// compute warps scan tile q+1 and publish its aggregate while the control
// warp looks back for tile q and takes the ticket of tile q+kBufs; then the
// compute warps fix up and store tile q and refill its buffer with tile
// q+kBufs. A tile's aggregate never waits on another tile's look-back, and
// the look-back overlaps the scan. Both loops pass the same two barriers per
// step and stop at the same step.
template <bool HS>
__global__ void __launch_bounds__(kCtaThreads, kBufs == 2 ? 3 : 2)
affine_scan_kernel(const AffineParams p) {
    extern __shared__ __align__(128) float s_dyn[];  // [kBufs][a | b][kTile]
    __shared__ AffineShared sh;
    __shared__ __align__(16) Pair s_walk[kMaxWindows * 32];

    const unsigned num_tiles = (unsigned)((p.n + kTile - 1) / kTile);
    if (threadIdx.x == kThreads) {
        sh.tag = ld_relaxed_u32(&p.ws->epoch) + 1u;
        for (int i = 0; i < kTicks; ++i) sh.tick[i] = atomicAdd(&p.ws->ticket, 1u);
        for (int i = 0; i < kBufs; ++i) mbar_init(&sh.bar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x >= kThreads)
        control_loop(p, sh, s_walk, num_tiles);
    else
        compute_loop<HS>(p, sh, s_dyn, num_tiles);
    finish_launch(p.ws, sh.tag);
}

}  // namespace

size_t affine_workspace_bytes(int64_t n) {
    if (n <= 0) return 0;
    const int64_t tiles = (n + kTile - 1) / kTile;
    return kWsHeaderBytes + (size_t)tiles * sizeof(TileDesc);
}

namespace {

// Per device: CTAs of each kernel variant that fit on one SM, and the SM
// count. Filled on a device's first launch (which also raises the kernel's
// dynamic shared-memory limit, a per-device attribute), under a lock.
constexpr int kMaxDevices = 64;
struct DeviceLaunch {
    int sms = 0;
    int per_sm[2] = {0, 0};  // [HS]
};
std::mutex g_launch_mutex;
DeviceLaunch g_launch[kMaxDevices];

template <bool HS>
ss_status launch_variant(const AffineParams &prm, int64_t tiles, cudaStream_t stream) {
    // persistent grid: as many CTAs as fit at once, capped by the tile count
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SS_ERR_UNSUPPORTED;
    int per_sm = 0, sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_launch_mutex);
        DeviceLaunch &d = g_launch[dev];
        if (d.per_sm[HS] <= 0) {
            int n_sms = 0, n = 0;
            if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaFuncSetAttribute(affine_scan_kernel<HS>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kDynSmem) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, affine_scan_kernel<HS>,
                                                              kCtaThreads, kDynSmem) != cudaSuccess ||
                n < 1 || n_sms < 1) {
                cudaGetLastError();
                return SS_ERR_CUDA;
            }
            d.sms = n_sms;
            d.per_sm[HS] = n;
        }
        per_sm = d.per_sm[HS];
        sms = d.sms;
    }
    const long long grid = std::min<long long>(tiles, (long long)sms * per_sm);
    affine_scan_kernel<HS><<<(unsigned)grid, kCtaThreads, kDynSmem, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

ss_status affine_launch(const float *a, const float *b, float *h, int64_t n, void *workspace,
                        cudaStream_t stream, unsigned long long timeout_ns, long long skip_unit,
                        bool log_step_tiles, const float *h0) {
    const int64_t tiles = (n + kTile - 1) / kTile;
    if (tiles > 0x7fffffffLL) return SS_ERR_UNSUPPORTED;
    AffineParams prm;
    prm.a = a;
    prm.b = b;
    prm.h = h;
    prm.h0 = h0;
    prm.n = n;
    prm.ws = reinterpret_cast<WsHeader *>(workspace);
    prm.desc = reinterpret_cast<TileDesc *>(reinterpret_cast<char *>(workspace) + kWsHeaderBytes);
    prm.timeout_ns = timeout_ns;
    prm.skip_unit = skip_unit;
    prm.bulk_ok = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
    prm.vec_out = (reinterpret_cast<uintptr_t>(h) & 15u) == 0;
    return log_step_tiles ? launch_variant<true>(prm, tiles, stream)
                          : launch_variant<false>(prm, tiles, stream);
}

}  // namespace ss
