// S6 selective-scan forward and bidirectional kernels (sm_103a).
//
// "POPCORNBENCH FW-GLM-5-1 l2_p30" (arjun-banerjee.github.io), forward-pass
// derivation: dA = exp(delta*A), dBx = delta*B_t*x, h = dA*h + dBx,
// y_t = sum_n h*C_t + D*x, with x, delta, y (B,L,D), B_t, C_t (B,L,N),
// A (D,N); softplus on delta via log(1 + exp(v)). "ARM-Scan"
// (krithiksama.me), Approach: the reverse recurrence reuses the forward
// one's discretisation. The pages' kernels (one thread per (b,d) running all
// of L; a NEON/multicore CPU scan) are prior art; this file is a new design:
//
//  * lane = one channel d with NG of its N states in registers, updated
//    two at a time with packed f32x2 fma/mul; a warp is 32 consecutive
//    channels, so x, delta and y accesses are coalesced;
//  * each warp streams its timesteps through a 3-slot shared-memory ring:
//    one bulk async copy (cp.async.bulk) per x and delta row and one per
//    B_t / C_t tile land on the slot's mbarrier while the warp computes on
//    the slot two stages behind;
//  * a CTA is WT warps that split one chunk of L into WT sub-chunks; a
//    sequence (b, 32 channels) is split into K chunks, one CTA each;
//  * with K == 1 and WT == 1 a warp runs its chains over all of L (the
//    register path). Otherwise each warp first sweeps its sub-chunk from a
//    zero state to get the sub-chunk aggregate (prod dA, end state), the
//    CTA folds these in shared memory, publishes the chunk aggregate in a
//    tagged global descriptor and takes its carry from a decoupled
//    look-back over earlier chunks (a look-forward over later ones for the
//    reverse direction); each warp then re-sweeps its sub-chunk from its
//    carry and writes y;
//  * exp and log run on the MUFU unit (ex2/lg2), with A pre-scaled by
//    log2(e); state and accumulation are fp32, bf16 inputs are widened
//    exactly and y is rounded to nearest even.
//
// Determinism: every carry is produced by applying aggregates to a state
// with one fma each, in sequence order, starting from the nearest published
// inclusive state. By induction that equals the inclusive state the
// predecessor publishes, bit for bit, so results do not depend on timing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <cstdio>
#include <cstdlib>

#include "f32x2.cuh"
#include "s6_common.cuh"
#include "ss_common.cuh"
#include "ss_internal.h"
#include "s6_tp.h"
#include "s6_ws.h"

namespace ss {
namespace {

constexpr int kMaxWT = 4;       // warps per CTA along time (hard limit)
constexpr int kDefaultWT = 4;   // default: small CTAs so several fit per SM
// CTAs of kMaxWT warps that the launch bounds guarantee per SM (registers)
template <bool BIDIR> constexpr int kMinCtas = 3;
constexpr int kMaxWindows = 4;  // look-back holds up to 128 predecessor chunks
constexpr int kMaxStages = 3;   // ring slots (and mbarriers) per warp, at most
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kCopyTimeoutNs = 2000000000ull;

// Descriptor payload fields, each [32 lanes][NG] floats per (sequence, chunk).
enum { F_P = 0, F_H = 1, F_INC = 2, F_HR = 3, F_RINC = 4 };
// Descriptor flags per (sequence, chunk).
enum { FL_AGG = 0, FL_INC = 1, FL_RINC = 2, FL_PAD = 3 };

struct S6Params {
    CUtensorMap tm_x, tm_d, tm_b, tm_c;  // 2D maps: (D or N) x (B*L rows); valid if tma
    const void *x, *delta, *Bt, *Ct;
    const float *A, *Dskip;
    void *y;
    float *yscratch;   // bidirectional bf16: fp32 forward outputs (B, L, D)
    long long L, D;
    long long ldd, ldbc;  // row strides (elements) of delta and of Bt, Ct
    int N;
    int dtiles;        // ceil(D / 32)
    int K;             // chunks per sequence
    int WT;            // warps per CTA
    int Tsub;          // timesteps per warp
    int bulk;          // rows and tiles are 16-byte aligned: stage with TMA tile copies
    WsHeader *ws;
    unsigned *flags;   // [(seq*K + k)*4 + FL_*]
    float *payload;    // [((seq*K + k)*NF + field)*32*NG + lane*NG + i]
    unsigned long long timeout_ns;
    long long skip_unit;  // test hook: this unit publishes nothing (-1: none)
    const float *delta_bias;  // (D,) added to delta before softplus, or null
    const float *h0;      // (B, D, N) state before t = 0, or null (zeros); forward only
    float *h_last;        // (B, D, N) receives the state after t = L - 1, or null
};

template <int NG>
__device__ __forceinline__ float *field_ptr(const S6Params &p, int NF, long long unit, int field,
                                            int lane) {
    return p.payload + ((unit * NF + field) * 32 + lane) * NG;
}

// Publishes flag `which` of `unit` once every thread of the CTA has written
// its part of the payload (each thread fences its own writes first).
__device__ __forceinline__ void publish_cta(const S6Params &p, long long unit, int which,
                                            unsigned tag) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0 && unit != p.skip_unit) st_release_u32(p.flags + unit * 4 + which, tag);
}

// Four consecutive states (a quad) of one lane's payload field.
__device__ __forceinline__ float4 *quad_ptr(float *field, int qd) {
    return reinterpret_cast<float4 *>(field) + qd;
}
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {
    return make_float4(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y), fmaf(a.z, b.z, c.z),
                       fmaf(a.w, b.w, c.w));
}

// ------------------------------------------------------------------ staging ring
// Per-warp shared memory: kStages slots of {x rows, delta rows, Bt tile, Ct
// tile} of kTS timesteps in the storage type, then fp32 copies of the current
// Bt / Ct rows padded to 16 states (used for bf16 storage or N != NG). bf16
// stages hold twice the timesteps, so the per-stage work (copy issue, wait,
// widening) is spread over more steps in the same shared memory.
template <typename IO> struct Ring {
    static constexpr int kTS = sizeof(IO) == 2 ? 16 : 8;
    static constexpr int kXBytes = kTS * 32 * (int)sizeof(IO);
    static constexpr int kBBytes = kTS * 16 * (int)sizeof(IO);
    static constexpr int kSlot = 2 * kXBytes + 2 * kBBytes;
    static constexpr int kConv = 2 * kTS * 16 * 4;
    static constexpr int kStages = 3;
    static_assert(kStages <= kMaxStages, "one mbarrier per slot");
    static constexpr int kWarp = kStages * kSlot + kConv;
};

struct WarpCtx {
    unsigned char *ring;   // this warp's ring
    uint64_t *bars;        // this warp's mbarriers, one per ring slot
    int slot;              // next ring slot to consume (and to refill after it)
    unsigned phases;       // bit s: parity of slot s's next completion
    long long b, d0, d;
    int cw;                // valid channels in this warp's tile
    int lane;
    int ch;                // channel of this lane within the warp's tile
    int half;              // which NG-state slice of the channel this lane holds
    bool dvalid;
    float dbias;           // bias added to this channel's delta (0 if none)
    long long t0, t1;      // this warp's timesteps
};

enum { MODE_AGG = 0, MODE_OUT = 1 };

// Starts loading stage `st` (timesteps t0 + st*kTS ...) into `slot`.
template <typename IO, int MODE, int LPC>
__device__ __forceinline__ void issue_stage(const S6Params &p, WarpCtx &w, int st, int slot) {
    constexpr int CPW = 32 / LPC;  // channels per warp
    using R = Ring<IO>;
    constexpr int kTS = R::kTS;
    const long long ts = w.t0 + (long long)st * kTS;
    const int nrows = (int)min((long long)kTS, w.t1 - ts);
    unsigned char *sl = w.ring + slot * R::kSlot;
    IO *xs = reinterpret_cast<IO *>(sl);
    IO *ds = reinterpret_cast<IO *>(sl + R::kXBytes);
    IO *bs = reinterpret_cast<IO *>(sl + 2 * R::kXBytes);
    IO *cs = reinterpret_cast<IO *>(sl + 2 * R::kXBytes + R::kBBytes);
    const IO *xg = static_cast<const IO *>(p.x);
    const IO *dg = static_cast<const IO *>(p.delta);
    const IO *bg = static_cast<const IO *>(p.Bt);
    const IO *cg = static_cast<const IO *>(p.Ct);
    const long long row0 = w.b * p.L + ts;
    const int N = p.N;
    if (p.bulk) {
        // one elected lane: expect the tile bytes, then four 2D tile copies
        // (boxes past the tensor's end arrive zero-filled and are never used)
        if (w.lane == 0) {
            const unsigned xbytes = kTS * (unsigned)CPW * (unsigned)sizeof(IO);
            const unsigned bbytes = kTS * (unsigned)N * (unsigned)sizeof(IO);
            uint64_t *bar = w.bars + slot;
            mbar_arrive_expect_tx(bar, 2u * xbytes + (MODE == MODE_OUT ? 2u : 1u) * bbytes);
            const int row = (int)row0;
            tma_load_2d(xs, &p.tm_x, (int)w.d0, row, bar);
            tma_load_2d(ds, &p.tm_d, (int)w.d0, row, bar);
            tma_load_2d(bs, &p.tm_b, 0, row, bar);
            if (MODE == MODE_OUT) tma_load_2d(cs, &p.tm_c, 0, row, bar);
        }
    } else {
        // unaligned shapes: plain loads, synchronous
        if (w.half == 0) {
            for (int r = 0; r < nrows; ++r) {
                xs[r * CPW + w.ch] = w.dvalid ? xg[(row0 + r) * p.D + w.d] : IO(0.0f);
                ds[r * CPW + w.ch] = w.dvalid ? dg[(row0 + r) * p.ldd + w.d] : IO(0.0f);
            }
        }
        for (int i = w.lane; i < nrows * N; i += 32) {
            const long long gi = (row0 + i / N) * p.ldbc + i % N;
            bs[i] = bg[gi];
            if (MODE == MODE_OUT) cs[i] = cg[gi];
        }
        __syncwarp();
    }
}

template <typename IO>
__device__ __forceinline__ void wait_stage(const S6Params &p, WarpCtx &w, int slot) {
    if (!p.bulk) return;
    const unsigned parity = (w.phases >> slot) & 1u;
    w.phases ^= 1u << slot;
    if (!mbar_wait_bounded(w.bars + slot, parity, kCopyTimeoutNs)) {
        if (w.lane == 0) record_error(p.ws, SS_ERR_TIMEOUT, 5u, (unsigned)w.b, (unsigned)w.t0);
        mbar_wait_bounded(w.bars + slot, parity, kCopyTimeoutNs);
    }
}

// Output handling of a MODE_OUT sweep.
enum { OUT_Y = 0,        // store y in the storage type
       OUT_HALF = 1,     // forward half of a bidirectional output: fp32 to yf
       OUT_SUM = 2 };    // reverse half: add the fp32 forward half, store y

// One timestep of this lane's chains. xv, dv: x and delta of (t, d); brow,
// crow: Bt and Ct rows of t as fp32; yp: this lane's output element.
template <int NG, int LPC, typename IO, bool SP, bool BIDIR, int MODE, int OUT>
__device__ __forceinline__ void step(float xv, float dv, const float *brow, const float *crow,
                                     const u64 (&A2)[NG / 2], float Dd, u64 (&h)[NG / 2],
                                     u64 (&hr)[NG / 2], u64 (&Q)[NG / 2], float &sdel, IO *yp,
                                     float *yfp, float yfv, bool store) {
    const float dl = SP ? softplus_mufu(dv) : dv;
    const float u = dl * xv;
    const u64 dd = f2(dl, dl);
    const u64 uu = f2(u, u);
    if constexpr (MODE == MODE_AGG) {
#pragma unroll
        for (int q4 = 0; q4 < NG / 4; ++q4) {
            const ulonglong2 bq = *reinterpret_cast<const ulonglong2 *>(brow + 4 * q4);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q2 = 2 * q4 + e;
                const u64 dA = f2_exp2_scaled(dd, A2[q2]);
                const u64 dbx = f2mul(uu, e ? bq.y : bq.x);
                h[q2] = f2fma(dA, h[q2], dbx);
                if constexpr (BIDIR) {
                    hr[q2] = f2fma(Q[q2], dbx, hr[q2]);
                    Q[q2] = f2mul(Q[q2], dA);
                }
            }
        }
        sdel += dl;
    } else {
        u64 acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int q4 = 0; q4 < NG / 4; ++q4) {
            const ulonglong2 bq = *reinterpret_cast<const ulonglong2 *>(brow + 4 * q4);
            const ulonglong2 cq = *reinterpret_cast<const ulonglong2 *>(crow + 4 * q4);
            const u64 dA0 = f2_exp2_scaled(dd, A2[2 * q4]);
            const u64 dA1 = f2_exp2_scaled(dd, A2[2 * q4 + 1]);
            h[2 * q4] = f2fma(dA0, h[2 * q4], f2mul(uu, bq.x));
            h[2 * q4 + 1] = f2fma(dA1, h[2 * q4 + 1], f2mul(uu, bq.y));
            acc0 = f2fma(h[2 * q4], cq.x, acc0);
            acc1 = f2fma(h[2 * q4 + 1], cq.y, acc1);
        }
        const u64 acc = f2add(acc0, acc1);
        float accs = f2lo(acc) + f2hi(acc);
#pragma unroll
        for (int o = 1; o < LPC; o <<= 1)  // the channel's other state slices
            accs += __shfl_xor_sync(0xffffffffu, accs, o);
        const float yv = fmaf(Dd, xv, accs);
        if (store) {
            if constexpr (OUT == OUT_Y) store_io(yp, yv);
            else if constexpr (OUT == OUT_HALF) *yfp = yv;
            else store_io(yp, yv + yfv);
        }
    }
}

// Widens the stage's Bt (and Ct) rows to fp32 x 16 states in `bconv` /
// `cconv`. bf16 with N == 16: 16-byte chunks of 8 values spread over the
// lanes (Bt chunks first, then Ct); other shapes: element by element, padded
// with zeros.
template <typename IO, int MODE>
__device__ __forceinline__ void widen_rows(const WarpCtx &w, const IO *bs, const IO *cs, int nrows,
                                           int N, float *bconv, float *cconv) {
    constexpr int kTS = Ring<IO>::kTS;
    if (sizeof(IO) == 2 && N == 16) {
        constexpr int kChunks = kTS * 2;  // per matrix
#pragma unroll
        for (int i0 = 0; i0 < (MODE == MODE_OUT ? 2 : 1) * kChunks; i0 += 32) {
            const int i = i0 + w.lane;
            if (i < (MODE == MODE_OUT ? 2 : 1) * kChunks) {
                const bool isC = i >= kChunks;
                const int c = isC ? i - kChunks : i;
                const uint4 v = *reinterpret_cast<const uint4 *>((isC ? cs : bs) + c * 8);
                float4 *dst = reinterpret_cast<float4 *>((isC ? cconv : bconv) + c * 8);
                dst[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
                dst[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                                     __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
            }
        }
    } else {
        for (int i = w.lane; i < nrows * 16; i += 32) {
            const int r = i >> 4, n = i & 15;
            bconv[i] = n < N ? to_f32(bs[r * N + n]) : 0.0f;
            if (MODE == MODE_OUT) cconv[i] = n < N ? to_f32(cs[r * N + n]) : 0.0f;
        }
    }
    __syncwarp();
}

// Issues the first ring stages of a pass (up to kStages) starting at the
// warp's next slot, so that they can land while the warp does other work.
template <typename IO, int MODE, int LPC, bool REV>
__device__ __forceinline__ void sweep_prime(const S6Params &p, WarpCtx &w) {
    constexpr int kTS = Ring<IO>::kTS;
    constexpr int kStages = Ring<IO>::kStages;
    const long long len = w.t1 - w.t0;
    if (len <= 0) return;
    const int nst = (int)((len + kTS - 1) / kTS);
    const int pre = min(kStages, nst);
    int sl = w.slot;
    for (int q = 0; q < pre; ++q) {
        issue_stage<IO, MODE, LPC>(p, w, REV ? nst - 1 - q : q, sl);
        sl = sl == kStages - 1 ? 0 : sl + 1;
    }
}

// One pass of this lane's chains over its timesteps, streamed through the ring.
// MODE_AGG: from the state in h (zero), accumulate the sub-chunk aggregate.
// MODE_OUT: from the state in h, write outputs (OUT_* above).
// PRIMED: sweep_prime already issued the first stages.
// Every stage a pass issues is consumed by the same pass, in issue order, so
// the ring's next slot carries over from one pass to the next.
template <int NG, int LPC, typename IO, bool SP, bool BIDIR, int MODE, bool REV, int OUT,
          bool PRIMED = false>
__device__ __forceinline__ void sweep(const S6Params &p, WarpCtx &w, const u64 (&A2)[NG / 2],
                                      float Dd, u64 (&h)[NG / 2], u64 (&hr)[NG / 2],
                                      u64 (&Q)[NG / 2], float &sdel, float *yf) {
    using R = Ring<IO>;
    constexpr int kTS = R::kTS;
    constexpr int kStages = R::kStages;
    const long long len = w.t1 - w.t0;
    if (len <= 0) return;
    const int nst = (int)((len + kTS - 1) / kTS);
    constexpr int CPW = 32 / LPC;
    const int N = p.N;
    const bool conv = (sizeof(IO) == 2) || (N != NG * LPC);
    float *bconv = reinterpret_cast<float *>(w.ring + kStages * R::kSlot);
    float *cconv = bconv + kTS * 16;
    if (!PRIMED) sweep_prime<IO, MODE, LPC, REV>(p, w);
    const long long D = p.D;
    IO *ybase = static_cast<IO *>(p.y) + w.b * p.L * D + w.d;   // y[b, 0, d]
    float *yfbase = yf ? yf + w.b * p.L * D + w.d : nullptr;
    const bool store = w.dvalid && w.half == 0;
    const int bstride = conv ? 16 : N;

    int slot = w.slot;
    for (int q = 0; q < nst; ++q) {
        const int st = REV ? nst - 1 - q : q;
        wait_stage<IO>(p, w, slot);
        const unsigned char *sl = w.ring + slot * R::kSlot;
        const IO *xs = reinterpret_cast<const IO *>(sl) + w.ch;
        const IO *ds = reinterpret_cast<const IO *>(sl + R::kXBytes) + w.ch;
        const IO *bs = reinterpret_cast<const IO *>(sl + 2 * R::kXBytes);
        const IO *cs = reinterpret_cast<const IO *>(sl + 2 * R::kXBytes + R::kBBytes);
        const long long ts = w.t0 + (long long)st * kTS;
        const int nrows = (int)min((long long)kTS, w.t1 - ts);
        if (conv) widen_rows<IO, MODE>(w, bs, cs, nrows, N, bconv, cconv);
        // this lane's state slice of each Bt / Ct row
        const float *bf = (conv ? bconv : reinterpret_cast<const float *>(bs)) + w.half * NG;
        const float *cf = (conv ? cconv : reinterpret_cast<const float *>(cs)) + w.half * NG;
        IO *yp = ybase + ts * D;
        float *yfp = yfbase ? yfbase + ts * D : nullptr;
        if (nrows == kTS) {
            // unrolled 8 steps at a time: a fully unrolled 16-step body of
            // every variant does not fit the instruction cache
#pragma unroll 1
            for (int r0 = 0; r0 < kTS; r0 += 8) {
                // reverse half of a bidirectional output: the 8 forward halves
                // it adds to are loaded together, ahead of the steps
                float yfv[8];
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int r = REV ? kTS - 1 - (r0 + rr) : r0 + rr;
                    yfv[rr] = (OUT == OUT_SUM && store) ? __ldcg(yfp + r * D) : 0.0f;
                }
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int r = REV ? kTS - 1 - (r0 + rr) : r0 + rr;
                    step<NG, LPC, IO, SP, BIDIR, MODE, OUT>(
                        to_f32(xs[r * CPW]), to_f32(ds[r * CPW]) + w.dbias, bf + r * bstride,
                        cf + r * bstride, A2, Dd, h, hr, Q, sdel, yp + r * D,
                        yfp ? yfp + r * D : nullptr, yfv[rr], store);
                }
            }
        } else {
            for (int rr = 0; rr < nrows; ++rr) {
                const int r = REV ? nrows - 1 - rr : rr;
                const float yfv = (OUT == OUT_SUM && store) ? __ldcg(yfp + r * D) : 0.0f;
                step<NG, LPC, IO, SP, BIDIR, MODE, OUT>(to_f32(xs[r * CPW]), to_f32(ds[r * CPW]) + w.dbias,
                                                        bf + r * bstride, cf + r * bstride, A2, Dd,
                                                        h, hr, Q, sdel, yp + r * D,
                                                        yfp ? yfp + r * D : nullptr, yfv, store);
            }
        }
        __syncwarp();  // every lane is done with this slot (and the fp32 rows)
        if (q + kStages < nst)
            issue_stage<IO, MODE, LPC>(p, w, REV ? nst - 1 - (q + kStages) : q + kStages, slot);
        slot = slot == kStages - 1 ? 0 : slot + 1;
    }
    w.slot = slot;
}

// ------------------------------------------------------------------ look-back
// Warp-parallel walk over the nearest predecessor (FWD) or successor (!FWD)
// chunks of the same sequence. Lane l examines chunk k -/+ (1 + l + 32*win)
// and waits until it holds at least an aggregate. Returns the chunk index of
// the nearest published inclusive state (-1 or K for the sequence boundary,
// whose state is zero), or -2 if any wait ran out.
template <bool FWD>
__device__ int find_anchor(const S6Params &p, long long seq, int k, unsigned tag, int lane) {
    const uint64_t t0 = globaltimer_ns();
    int win = 0;
    for (;;) {
        const int m = FWD ? k - 1 - (lane + 32 * win) : k + 1 + (lane + 32 * win);
        bool is_inc = false, gave_up = false;
        if (FWD ? (m < 0) : (m >= p.K)) {
            is_inc = true;
        } else {
            const unsigned *fl = p.flags + (seq * p.K + m) * 4;
            const int inc_field = FWD ? FL_INC : FL_RINC;
            for (unsigned it = 0;; ++it) {
                if (ld_acquire_u32(fl + inc_field) == tag) {
                    is_inc = true;
                    break;
                }
                if (ld_acquire_u32(fl + FL_AGG) == tag) break;
                if ((it & 63u) == 63u &&
                    (globaltimer_ns() - t0 > p.timeout_ns || ld_relaxed_u32(&p.ws->error) != 0u)) {
                    gave_up = true;
                    break;
                }
            }
        }
        if (__ballot_sync(kFull, gave_up)) return -2;
        const unsigned incs = __ballot_sync(kFull, is_inc);
        if (incs) {
            const int l = __ffs(incs) - 1;  // nearest lane with an inclusive state
            const int dist = l + 32 * win;
            return FWD ? k - 1 - dist : k + 1 + dist;
        }
        if (globaltimer_ns() - t0 > p.timeout_ns || ld_relaxed_u32(&p.ws->error) != 0u) return -2;
        if (win + 1 < kMaxWindows) ++win;  // else look at the farthest window again
    }
}

// Chunk aggregate of this lane's states 4qd .. 4qd+3: the sub-chunk
// aggregates (P, H) folded in sequence order, and Hr (reverse direction)
// folded in reverse order.
template <int NG, int NSUB, bool BIDIR>
__device__ __forceinline__ void chunk_aggregate(const float *s_sub, int WT, int lane, int qd,
                                                float4 &P, float4 &H, float4 &Hr) {
    float Pv[4] = {1.0f, 1.0f, 1.0f, 1.0f}, Hv[4] = {}, Hrv[4] = {};
    for (int v = 0; v < WT; ++v) {
        const float *sv = s_sub + v * NSUB * NG * 32 + lane;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 4 * qd + e;
            Pv[e] *= sv[i * 32];
            Hv[e] = fmaf(sv[i * 32], Hv[e], sv[(NG + i) * 32]);
        }
    }
    if constexpr (BIDIR) {
        for (int v = WT - 1; v >= 0; --v) {
            const float *sv = s_sub + v * NSUB * NG * 32 + lane;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 4 * qd + e;
                Hrv[e] = fmaf(sv[i * 32], Hrv[e], sv[(2 * NG + i) * 32]);
            }
        }
    }
    P = make_float4(Pv[0], Pv[1], Pv[2], Pv[3]);
    H = make_float4(Hv[0], Hv[1], Hv[2], Hv[3]);
    Hr = make_float4(Hrv[0], Hrv[1], Hrv[2], Hrv[3]);
}

// Applies the aggregates of chunks m = from, from + dir, ... (stopping before
// `to`) to the state quad c, one fma per state each, in that order. The
// aggregates are loaded eight chunks at a time, so a walk over W chunks
// waits for about W / 8 round trips to L2.
template <int NG>
__device__ __forceinline__ float4 apply_quads(const S6Params &p, int NF, long long seq, int from,
                                              int to, int dir, int fieldH, int lane, int qd,
                                              float4 c) {
    constexpr int U = 8;
    for (int m = from; m != to;) {
        const int n = min(U, (to - m) * dir);
        float4 P[U], H[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (u < n) {
                const long long unit = seq * p.K + m + u * dir;
                P[u] = ld_cg_f32x4(quad_ptr(field_ptr<NG>(p, NF, unit, F_P, lane), qd));
                H[u] = ld_cg_f32x4(quad_ptr(field_ptr<NG>(p, NF, unit, fieldH, lane), qd));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (u < n) c = fma4(P[u], c, H[u]);
        m += n * dir;
    }
    return c;
}

// State n of this lane's channel before t = 0: h0 if given, else zero.
__device__ __forceinline__ float initial_state(const S6Params &p, const WarpCtx &w, int n) {
    return (p.h0 && w.dvalid && n < p.N) ? p.h0[(w.b * p.D + w.d) * p.N + n] : 0.0f;
}

// ------------------------------------------------------------------ kernel
template <int NG, int LPC, typename IO, bool SP, bool BIDIR>
__global__ void __launch_bounds__(kMaxWT * 32, kMinCtas<BIDIR>)
s6_kernel(const __grid_constant__ S6Params p) {
    constexpr int CPW = 32 / LPC;  // channels per warp
    constexpr int NSUB = BIDIR ? 3 : 2;  // sub-aggregate fields: P, H (, Hr)
    constexpr int NF = BIDIR ? 5 : 3;    // descriptor fields
    constexpr int NP = NG / 2;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ int s_anchor[2];  // look-back / look-forward results
    // TMA destinations need 128-byte alignment; the launch adds 128 bytes of slack
    unsigned char *s_ring = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    uint64_t *s_bars = reinterpret_cast<uint64_t *>(s_ring + p.WT * Ring<IO>::kWarp);  // [WT][kMaxStages]
    float *s_sub = reinterpret_cast<float *>(s_bars + p.WT * kMaxStages);   // [WT][NSUB][32][NG]
    float *s_car = s_sub + p.WT * NSUB * 32 * NG;  // [directions][32][NG]

    const bool chunked = p.K > 1;
    unsigned ticket, tag = 0;
    if (chunked) {
        take_ticket(p.ws, ticket, tag);
    } else {
        ticket = blockIdx.x;
    }
    const long long seq = ticket / (unsigned)p.K;
    const int k = (int)(ticket % (unsigned)p.K);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    WarpCtx w;
    w.ring = s_ring + warp * Ring<IO>::kWarp;
    w.bars = s_bars + warp * kMaxStages;
    w.slot = 0;
    w.phases = 0;
    w.lane = lane;
    w.ch = lane / LPC;
    w.half = lane % LPC;
    w.b = seq / p.dtiles;
    w.d0 = (seq % p.dtiles) * CPW;
    w.d = w.d0 + w.ch;
    w.dvalid = w.d < p.D;
    w.cw = (int)min((long long)CPW, p.D - w.d0);
    const long long tc0 = (long long)k * p.WT * p.Tsub;
    w.t0 = min(tc0 + (long long)warp * p.Tsub, p.L);
    w.t1 = min(w.t0 + (long long)p.Tsub, p.L);
    if (lane == 0 && p.bulk) {
        for (int s = 0; s < Ring<IO>::kStages; ++s) mbar_init(w.bars + s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    u64 A2[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const int n0 = w.half * NG + 2 * q;  // this lane's states n0, n0 + 1
        float lo = 0.0f, hi = 0.0f;
        if (w.dvalid && n0 < p.N) lo = p.A[w.d * p.N + n0] * kLog2e;
        if (w.dvalid && n0 + 1 < p.N) hi = p.A[w.d * p.N + n0 + 1] * kLog2e;
        A2[q] = f2(lo, hi);
    }
    const float Dd = (w.dvalid && p.Dskip) ? p.Dskip[w.d] : 0.0f;
    w.dbias = (w.dvalid && p.delta_bias) ? p.delta_bias[w.d] : 0.0f;

    u64 h[NP], hr[NP], Q[NP];
    float sdel = 0.0f;
    // state entering the sequence: h0, or zero
    float cf[NG], cr[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) {
        cf[i] = BIDIR ? 0.0f : initial_state(p, w, w.half * NG + i);
        cr[i] = 0.0f;
    }

    if (chunked || p.WT > 1) {
        // ---- sub-chunk aggregate from a zero state
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            h[q] = 0ull;
            hr[q] = 0ull;
            Q[q] = f2(1.0f, 1.0f);
        }
        sweep<NG, LPC, IO, SP, BIDIR, MODE_AGG, false, OUT_Y>(p, w, A2, Dd, h, hr, Q, sdel, nullptr);
        // s_sub[((w*NSUB + field)*NG + i)*32 + lane]: lane-fastest, conflict-free
        float *mine = s_sub + warp * NSUB * NG * 32 + lane;
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            mine[(2 * q) * 32] = ex2_approx(f2lo(A2[q]) * sdel);  // prod of dA over the sub-chunk
            mine[(2 * q + 1) * 32] = ex2_approx(f2hi(A2[q]) * sdel);
            mine[(NG + 2 * q) * 32] = f2lo(h[q]);
            mine[(NG + 2 * q + 1) * 32] = f2hi(h[q]);
            if constexpr (BIDIR) {
                mine[(2 * NG + 2 * q) * 32] = f2lo(hr[q]);
                mine[(2 * NG + 2 * q + 1) * 32] = f2hi(hr[q]);
            }
        }
        // the output pass's first stages load while the carries are found
        sweep_prime<IO, MODE_OUT, LPC, false>(p, w);
        __syncthreads();

        if (chunked) {
            const long long unit = seq * p.K + k;
            // chunk aggregate to the descriptor; the state quads of the 32
            // channels are spread over the CTA's warps
            for (int qd = warp; qd < NG / 4; qd += p.WT) {
                float4 P4, H4, Hr4;
                chunk_aggregate<NG, NSUB, BIDIR>(s_sub, p.WT, lane, qd, P4, H4, Hr4);
                __stcg(quad_ptr(field_ptr<NG>(p, NF, unit, F_P, lane), qd), P4);
                __stcg(quad_ptr(field_ptr<NG>(p, NF, unit, F_H, lane), qd), H4);
                if constexpr (BIDIR) __stcg(quad_ptr(field_ptr<NG>(p, NF, unit, F_HR, lane), qd), Hr4);
            }
            publish_cta(p, unit, FL_AGG, tag);
            // nearest published inclusive state on the left
            if (warp == 0) {
                const int j = find_anchor<true>(p, seq, k, tag, lane);
                if (lane == 0) s_anchor[0] = j;
            }
            __syncthreads();

            // forward carry: the anchor's inclusive state, then the aggregates
            // after it applied in sequence order
            const int j = s_anchor[0];
            if (j == -2 && threadIdx.x == 0) record_error(p.ws, SS_ERR_TIMEOUT, 3u, (unsigned)unit, 0u);
            for (int qd = warp; qd < NG / 4; qd += p.WT) {
                float4 c = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (j >= 0) c = ld_cg_f32x4(quad_ptr(field_ptr<NG>(p, NF, seq * p.K + j, F_INC, lane), qd));
                if (j == -1 && !BIDIR) {  // the sequence's start: h0
                    const int n0 = w.half * NG + 4 * qd;
                    c = make_float4(initial_state(p, w, n0), initial_state(p, w, n0 + 1),
                                    initial_state(p, w, n0 + 2), initial_state(p, w, n0 + 3));
                }
                if (j != -2) c = apply_quads<NG>(p, NF, seq, j + 1, k, 1, F_H, lane, qd, c);
                s_car[(4 * qd) * 32 + lane] = c.x;
                s_car[(4 * qd + 1) * 32 + lane] = c.y;
                s_car[(4 * qd + 2) * 32 + lane] = c.z;
                s_car[(4 * qd + 3) * 32 + lane] = c.w;
                float4 P4, H4, Hr4;
                chunk_aggregate<NG, NSUB, BIDIR>(s_sub, p.WT, lane, qd, P4, H4, Hr4);
                __stcg(quad_ptr(field_ptr<NG>(p, NF, unit, F_INC, lane), qd), fma4(P4, c, H4));
            }
            publish_cta(p, unit, FL_INC, tag);

            if constexpr (BIDIR) {
                // reverse carry: the same on the right, in reverse order. The
                // search starts only after this chunk's forward inclusive state
                // is out: a forward walk never waits on a reverse one, so the
                // two chains cannot wait on each other.
                if (warp == 0) {
                    const int jr0 = find_anchor<false>(p, seq, k, tag, lane);
                    if (lane == 0) s_anchor[1] = jr0;
                }
                __syncthreads();
                const int jr = s_anchor[1];
                if (jr == -2 && threadIdx.x == 0) record_error(p.ws, SS_ERR_TIMEOUT, 4u, (unsigned)unit, 0u);
                for (int qd = warp; qd < NG / 4; qd += p.WT) {
                    float4 c = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (jr >= 0 && jr < p.K)
                        c = ld_cg_f32x4(quad_ptr(field_ptr<NG>(p, NF, seq * p.K + jr, F_RINC, lane), qd));
                    if (jr != -2) c = apply_quads<NG>(p, NF, seq, jr - 1, k, -1, F_HR, lane, qd, c);
                    s_car[(NG + 4 * qd) * 32 + lane] = c.x;
                    s_car[(NG + 4 * qd + 1) * 32 + lane] = c.y;
                    s_car[(NG + 4 * qd + 2) * 32 + lane] = c.z;
                    s_car[(NG + 4 * qd + 3) * 32 + lane] = c.w;
                    float4 P4, H4, Hr4;
                    chunk_aggregate<NG, NSUB, BIDIR>(s_sub, p.WT, lane, qd, P4, H4, Hr4);
                    __stcg(quad_ptr(field_ptr<NG>(p, NF, unit, F_RINC, lane), qd), fma4(P4, c, Hr4));
                }
                publish_cta(p, unit, FL_RINC, tag);
            }
            // (the barrier in publish_cta also completes s_car)
#pragma unroll
            for (int i = 0; i < NG; ++i) {
                cf[i] = s_car[i * 32 + lane];
                if constexpr (BIDIR) cr[i] = s_car[(NG + i) * 32 + lane];
            }
        }

        // this warp's carries: the chunk carry (zero for an unsplit
        // sequence) moved across the earlier (forward) or later (reverse)
        // sub-chunks of the CTA, in order
        for (int v = 0; v < warp; ++v) {
            const float *s = s_sub + v * NSUB * NG * 32 + lane;
#pragma unroll
            for (int i = 0; i < NG; ++i) cf[i] = fmaf(s[i * 32], cf[i], s[(NG + i) * 32]);
        }
        if constexpr (BIDIR) {
            for (int v = p.WT - 1; v > warp; --v) {
                const float *s = s_sub + v * NSUB * NG * 32 + lane;
#pragma unroll
                for (int i = 0; i < NG; ++i) cr[i] = fmaf(s[i * 32], cr[i], s[(2 * NG + i) * 32]);
            }
        }
    }

    // ---- outputs: forward sweep from the carry (and the reverse sweep)
#pragma unroll
    for (int q = 0; q < NP; ++q) h[q] = f2(cf[2 * q], cf[2 * q + 1]);
    const bool primed = chunked || p.WT > 1;
    if constexpr (BIDIR) {
        float *yf = p.yscratch ? p.yscratch : static_cast<float *>(p.y);
        if (primed)
            sweep<NG, LPC, IO, SP, BIDIR, MODE_OUT, false, OUT_HALF, true>(p, w, A2, Dd, h, hr, Q, sdel, yf);
        else
            sweep<NG, LPC, IO, SP, BIDIR, MODE_OUT, false, OUT_HALF>(p, w, A2, Dd, h, hr, Q, sdel, yf);
#pragma unroll
        for (int q = 0; q < NP; ++q) h[q] = f2(cr[2 * q], cr[2 * q + 1]);
        sweep<NG, LPC, IO, SP, BIDIR, MODE_OUT, true, OUT_SUM>(p, w, A2, Dd, h, hr, Q, sdel, yf);
    } else {
        if (primed)
            sweep<NG, LPC, IO, SP, BIDIR, MODE_OUT, false, OUT_Y, true>(p, w, A2, Dd, h, hr, Q, sdel, nullptr);
        else
            sweep<NG, LPC, IO, SP, BIDIR, MODE_OUT, false, OUT_Y>(p, w, A2, Dd, h, hr, Q, sdel, nullptr);
        // the warp that ran the last step holds h[L - 1]
        if (p.h_last && w.dvalid && w.t0 < w.t1 && w.t1 == p.L) {
            float *dst = p.h_last + (w.b * p.D + w.d) * p.N;
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const int n0 = w.half * NG + 2 * q;
                if (n0 < p.N) dst[n0] = f2lo(h[q]);
                if (n0 + 1 < p.N) dst[n0 + 1] = f2hi(h[q]);
            }
        }
    }

    if (chunked) finish_launch(p.ws, tag);
}

// ------------------------------------------------------------------ planning
struct Plan {
    int NG, LPC, WT, K, Tsub, dtiles;
    long long seqs;
    size_t flag_bytes, payload_bytes, scratch_bytes, desc_bytes, total;
    size_t smem;
    bool tp;      // the time-parallel single pass (s6_tp.cu) runs this shape
    TPPlan tpp;   // its launch shape; its packed B_t / C_t follow the chunked
                  // plan's section of the workspace
    size_t tp_offset;
    bool ws;      // the wavefront single pass (s6_ws.cu) runs this shape
    WSPlan wsp;   // its launch shape (it needs the workspace header only)
};

// Plan override for tests (ss_testing_s6_plan): kind 0 = the planner's
// choice; 1 = the chunked kernel with (WT, Tsub) = (a, b) (0, 0 = the
// planner's) and c lanes per channel (0 or 1: one); 2 = the time-parallel
// single pass with (G, T, W) = (a, b, c); 3 = the wavefront single pass
// with (T, S) = (a, b).
std::atomic<int> g_ovr_kind{0}, g_ovr_a{0}, g_ovr_b{0}, g_ovr_c{0};
// The time-parallel pass is built and tested but not yet taken by default:
// measured on GB300 it does not beat the chunked kernel on the fp32 and bf16
// forward workloads (its per-pair scan costs as many instructions as the
// chunked kernel's second sweep).
constexpr bool kTPByDefault = false;

Plan make_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int bidir) {
    Plan pl{};
    const long long sms = device_sm_count();
    pl.NG = N <= 4 ? 4 : (N <= 8 ? 8 : 16);
    pl.LPC = 1;
    // Two lanes per channel (8 states each) doubles the warps but repeats the
    // per-timestep scalar work on both lanes; measured slower on every S6
    // shape tried, so it is only taken on request.
    const int ovr = g_ovr_kind.load();
    if (ovr == 1) {  // test override: 2 or 4 lanes per channel
        const int v = g_ovr_c.load();
        if ((v == 2 || v == 4) && pl.NG == 16) {
            pl.NG = 16 / v;
            pl.LPC = v;
        }
    }
    const int cpw = 32 / pl.LPC;
    pl.dtiles = (int)((D + cpw - 1) / cpw);
    pl.seqs = B * pl.dtiles;
    const long long target_warps = sms * 16;
    long long S = (target_warps + pl.seqs - 1) / std::max<long long>(pl.seqs, 1);
    S = std::max<long long>(1, std::min<long long>(S, (L + 31) / 32));
    int WT = (int)std::min<long long>(S, kDefaultWT);
    long long K = (S + WT - 1) / WT;
    long long Tsub = (L + K * WT - 1) / (K * WT);
    const int kTS = io_bf16 ? Ring<__nv_bfloat16>::kTS : Ring<float>::kTS;
    Tsub = (Tsub + kTS - 1) / kTS * kTS;
    // once L is split at all (two sweeps), at most 128 steps per warp: shorter
    // chunks keep a chunk's inputs in L2 between its two sweeps and give the
    // look-back more chunks to overlap
    if (K * WT > 1) Tsub = std::min<long long>(Tsub, 128);
    // a bidirectional sequence needs all of its chunks resident at once:
    // keep K within one chunk per SM
    if (bidir) Tsub = std::max<long long>(Tsub, (L + (long long)WT * sms - 1) / ((long long)WT * sms));
    // whole waves: a CTA count just above a multiple of what fits at once
    // leaves most SMs idle in the last wave. For plans of more than one
    // wave, among sub-chunk lengths from half of the above (up to one and a
    // half times it for bidirectional plans, whose residency bound already
    // lengthens them and whose working set stays well inside L2), take the
    // one minimising waves x (steps per warp + 16, the per-chunk fold and
    // look-back in steps); 4-warp CTAs fit kMinCtas per SM by their launch
    // bounds, fewer if shared memory runs out first.
    if (WT == kMaxWT && (long long)WT * Tsub < L) {
        const size_t ring = io_bf16 ? Ring<__nv_bfloat16>::kWarp : Ring<float>::kWarp;
        const size_t smem = 128 + (size_t)WT * (ring + kMaxStages * sizeof(uint64_t)) +
                            (size_t)(WT * (bidir ? 3 : 2) + (bidir ? 2 : 1)) * 32 * pl.NG *
                                sizeof(float);
        const long long per_sm =
            std::max<long long>(1, std::min<long long>(bidir ? kMinCtas<true> : kMinCtas<false>,
                                                       device_smem_per_sm() / (long long)(smem + 1024)));
        const long long slots = sms * per_sm;
        const long long K0 = (L + (long long)WT * Tsub - 1) / ((long long)WT * Tsub);
        long long lo = std::max<long long>(kTS, Tsub / 2 / kTS * kTS);
        if (bidir) {  // keep the residency bound
            const long long rb = (L + (long long)WT * sms - 1) / ((long long)WT * sms);
            lo = std::max<long long>(lo, (rb + kTS - 1) / kTS * kTS);
        }
        const long long hi = bidir ? (Tsub + Tsub / 2) / kTS * kTS : Tsub;
        long long best_cost = -1, best_T = Tsub;
        // (within one wave there is nothing to fill: keep the plan)
        for (long long T = hi; pl.seqs * K0 > slots && T >= lo; T -= kTS) {
            const long long Kc = (L + (long long)WT * T - 1) / ((long long)WT * T);
            const long long waves = (pl.seqs * Kc + slots - 1) / slots;
            const long long cost = waves * (T + 16);
            if (best_cost < 0 || cost < best_cost) {
                best_cost = cost;
                best_T = T;
            }
        }
        Tsub = best_T;
    }
    if (ovr == 1) {  // test override of (warps per CTA, timesteps per warp)
        const int wv = g_ovr_a.load(), tv = g_ovr_b.load();
        if (wv >= 1 && wv <= kMaxWT && tv >= 1) {  // (0, 0): keep the planner's
            WT = wv;
            Tsub = tv;
        }
    }
    K = std::max<long long>(1, (L + (long long)WT * Tsub - 1) / ((long long)WT * Tsub));
    pl.WT = WT;
    pl.K = (int)K;
    pl.Tsub = (int)Tsub;
    const int NF = bidir ? 5 : 3;
    const int NSUB = bidir ? 3 : 2;
    if (pl.K > 1) {
        pl.flag_bytes = (size_t)pl.seqs * pl.K * 4 * sizeof(unsigned);
        pl.flag_bytes = (pl.flag_bytes + 255) / 256 * 256;
        pl.payload_bytes = (size_t)pl.seqs * pl.K * NF * 32 * pl.NG * sizeof(float);
    }
    pl.scratch_bytes = (bidir && io_bf16) ? (size_t)B * L * D * sizeof(float) : 0;
    pl.desc_bytes = pl.flag_bytes + pl.payload_bytes;
    pl.total = 0;
    if (pl.K > 1 || pl.scratch_bytes) pl.total = kWsHeaderBytes + pl.desc_bytes + pl.scratch_bytes;
    const size_t ring = io_bf16 ? Ring<__nv_bfloat16>::kWarp : Ring<float>::kWarp;
    pl.smem = 128 + (size_t)pl.WT * (ring + kMaxStages * sizeof(uint64_t)) +
              (size_t)(pl.WT * NSUB + (bidir ? 2 : 1)) * 32 * pl.NG * sizeof(float);

    // The time-parallel single pass computes each term's exp once and needs
    // no look-back, but its parallelism is one warp per G channels: it runs
    // forward shapes whose channels alone keep the SMs busy (tp_choose_plan).
    pl.tp = false;
    pl.tp_offset = 0;
    pl.ws = false;
    // The wavefront single pass computes each term's exp once, reads every
    // input once and needs no look-back; it takes forward shapes whose
    // channels fill the chip (ws_choose_plan), the chunked kernel the rest.
    if (!bidir && (ovr == 3 || ovr == 0)) {
        WSPlan wsp{};
        const bool ok = ovr == 3 ? ws_make_plan(B, L, D, N, io_bf16, g_ovr_a.load(),
                                                g_ovr_b.load(), &wsp)
                                 : ws_choose_plan(B, L, D, N, io_bf16, (int)sms, &wsp);
        if (ok) {
            pl.ws = true;
            pl.wsp = wsp;
            pl.total = std::max<size_t>(pl.total, kWsHeaderBytes);
            return pl;
        }
        if (ovr == 3) return pl;
    }
    if (!bidir && ovr != 1) {
        TPPlan tpp{};
        const bool ok = ovr == 2 ? tp_make_plan(B, L, D, N, io_bf16, g_ovr_a.load(),
                                                g_ovr_b.load(), g_ovr_c.load(), &tpp)
                                 : (kTPByDefault && tp_choose_plan(B, L, D, N, io_bf16, (int)sms, &tpp));
        if (ok) {
            pl.tp = true;
            pl.tpp = tpp;
            const size_t base = std::max<size_t>(pl.total, kWsHeaderBytes);
            pl.tp_offset = (base + 255) / 256 * 256;
            pl.total = pl.tp_offset + tpp.pack_bytes;
        }
    }
    return pl;
}

// Row-major 2D map over `rows` rows of `inner` elements, `ld` elements apart,
// box = box_inner x box_rows.
bool encode_2d(CUtensorMap *m, const void *base, bool bf16, uint64_t inner, uint64_t ld,
               uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
    const uint64_t es = bf16 ? 2 : 4;
    const uint64_t dims[2] = {inner, rows};
    const uint64_t strides[1] = {ld * es};
    const uint32_t box[2] = {box_inner, box_rows};
    return encode_tiled_map(m, base, bf16, 2, dims, strides, box);
}

template <int NG, int LPC, typename IO, bool SP, bool BIDIR>
ss_status launch_t(const S6Params &prm, const Plan &pl, cudaStream_t stream) {
    auto kern = s6_kernel<NG, LPC, IO, SP, BIDIR>;
    if (pl.smem > 48 * 1024 &&
        raise_smem_limit(reinterpret_cast<const void *>(kern), (int)pl.smem) != SS_OK)
        return SS_ERR_CUDA;
    if (BIDIR && pl.K > 1) {
        // every chunk of one sequence must be resident at the same time
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, pl.WT * 32, pl.smem) !=
            cudaSuccess)
            return SS_ERR_CUDA;
        if ((long long)per_sm * device_sm_count() < 2LL * pl.K) return SS_ERR_UNSUPPORTED;
    }
    const long long grid = pl.seqs * pl.K;
    if (grid > 0x7fffffffLL) return SS_ERR_UNSUPPORTED;
    kern<<<(unsigned)grid, pl.WT * 32, pl.smem, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <int NG, int LPC, typename IO>
ss_status launch_ng(const S6Params &prm, const Plan &pl, bool sp, bool bidir, cudaStream_t s) {
    if (bidir)
        return sp ? launch_t<NG, LPC, IO, true, true>(prm, pl, s)
                  : launch_t<NG, LPC, IO, false, true>(prm, pl, s);
    return sp ? launch_t<NG, LPC, IO, true, false>(prm, pl, s)
              : launch_t<NG, LPC, IO, false, false>(prm, pl, s);
}

template <typename IO>
ss_status launch_io(const S6Params &prm, const Plan &pl, bool sp, bool bidir, cudaStream_t s) {
    if (pl.LPC == 2) return launch_ng<8, 2, IO>(prm, pl, sp, bidir, s);
    if (pl.LPC == 4) return launch_ng<4, 4, IO>(prm, pl, sp, bidir, s);
    switch (pl.NG) {
        case 4: return launch_ng<4, 1, IO>(prm, pl, sp, bidir, s);
        case 8: return launch_ng<8, 1, IO>(prm, pl, sp, bidir, s);
        default: return launch_ng<16, 1, IO>(prm, pl, sp, bidir, s);
    }
}

}  // namespace

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (the library does not link libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *sym = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &sym, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(sym);
        cudaGetLastError();
    });
    return fn;
}

bool encode_tiled_map(void *map, const void *base, bool bf16, int rank, const uint64_t *dims,
                      const uint64_t *strides, const uint32_t *box, int swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return enc(static_cast<CUtensorMap *>(map),
               bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
               (cuuint32_t)rank, const_cast<void *>(base), d, st, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
               : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                               : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void s6_set_plan_override(int kind, int a, int b, int c) {
    g_ovr_a.store(a);
    g_ovr_b.store(b);
    g_ovr_c.store(c);
    g_ovr_kind.store(kind >= 0 && kind <= 3 ? kind : 0);
}

int s6_describe_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int bidir,
                     int64_t *out) {
    if (B <= 0 || L <= 0 || D <= 0 || N <= 0 || N > 16) return -1;
    const Plan pl = make_plan(B, L, D, N, io_bf16, bidir);
    if (pl.ws) {
        out[0] = pl.wsp.T;
        out[1] = pl.wsp.S;
        out[2] = 32;
        out[3] = pl.wsp.nblk;
        out[4] = pl.wsp.ctas;
        out[5] = pl.wsp.R;
        return 2;
    }
    if (pl.tp) {
        out[0] = pl.tpp.G;
        out[1] = pl.tpp.T;
        out[2] = pl.tpp.W;
        out[3] = pl.tpp.nblk;
        out[4] = pl.tpp.ctas;
        out[5] = pl.tpp.R;
        return 1;
    }
    out[0] = pl.LPC;
    out[1] = pl.WT;
    out[2] = pl.Tsub;
    out[3] = pl.K;
    out[4] = pl.seqs * pl.K;
    out[5] = pl.NG;
    return 0;
}

size_t s6_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int bidir) {
    if (B <= 0 || L <= 0 || D <= 0 || N <= 0) return 0;
    return make_plan(B, L, D, N, io_bf16, bidir).total;
}

ss_status s6_launch(const S6Args &a, void *workspace, size_t ws_bytes, cudaStream_t stream,
                    unsigned long long timeout_ns, long long skip_unit) {
    const Plan pl = make_plan(a.B, a.L, a.D, a.N, a.io_bf16, a.bidir);
    if (pl.total > 0) {
        if (workspace == nullptr || ws_bytes < pl.total ||
            (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return SS_ERR_WORKSPACE;
    }
    if (pl.ws) {
        // tile copies need 16-byte aligned rows and bases (else the chunked
        // kernel below runs, with its own section of the workspace)
        const size_t es = a.io_bf16 ? 2 : 4;
        const int64_t ldd = a.ld_delta > 0 ? a.ld_delta : a.D;
        const int64_t ldbc = a.ld_bc > 0 ? a.ld_bc : a.N;
        const uintptr_t al = reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.delta) |
                             reinterpret_cast<uintptr_t>(a.y) | reinterpret_cast<uintptr_t>(a.Bt) |
                             reinterpret_cast<uintptr_t>(a.Ct);
        if ((a.D * es) % 16 == 0 && (ldd * es) % 16 == 0 && (ldbc * es) % 16 == 0 && al % 16 == 0)
            return ws_launch(a, pl.wsp, workspace, stream, timeout_ns);
    }
    if (pl.tp) {
        // tile copies need 16-byte aligned rows and bases (else the chunked
        // kernel below runs, with its own section of the workspace)
        const size_t es = a.io_bf16 ? 2 : 4;
        const int64_t ldd = a.ld_delta > 0 ? a.ld_delta : a.D;
        const uintptr_t al = reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.delta) |
                             reinterpret_cast<uintptr_t>(a.y);
        if ((a.D * es) % 16 == 0 && (ldd * es) % 16 == 0 && al % 16 == 0) {
            return tp_launch(a, pl.tpp, workspace, pl.tp_offset, stream, timeout_ns);
        }
    }
    S6Params prm{};
    prm.x = a.x;
    prm.delta = a.delta;
    prm.Bt = a.Bt;
    prm.Ct = a.Ct;
    prm.A = a.A;
    prm.Dskip = a.Dskip;
    prm.y = a.y;
    prm.L = a.L;
    prm.D = a.D;
    prm.N = (int)a.N;
    prm.dtiles = pl.dtiles;
    prm.K = pl.K;
    prm.WT = pl.WT;
    prm.Tsub = pl.Tsub;
    const size_t es = a.io_bf16 ? 2 : 4;
    prm.ldd = a.ld_delta > 0 ? a.ld_delta : a.D;
    prm.ldbc = a.ld_bc > 0 ? a.ld_bc : a.N;
    const uintptr_t al = reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.delta) |
                         reinterpret_cast<uintptr_t>(a.Bt) | reinterpret_cast<uintptr_t>(a.Ct);
    prm.bulk = ((a.D * es) % 16 == 0) && ((a.N * es) % 16 == 0) && ((prm.ldd * es) % 16 == 0) &&
               ((prm.ldbc * es) % 16 == 0) && (al % 16 == 0) && (a.B * a.L < (1LL << 31)) &&
               (a.D < (1LL << 31));
    if (prm.bulk) {
        const bool bf = a.io_bf16 != 0;
        const uint64_t rows = (uint64_t)(a.B * a.L);
        const uint32_t cpw = 32u / (uint32_t)pl.LPC;
        const uint32_t kTS = bf ? Ring<__nv_bfloat16>::kTS : Ring<float>::kTS;
        prm.bulk = encode_2d(&prm.tm_x, a.x, bf, a.D, a.D, rows, cpw, kTS) &&
                   encode_2d(&prm.tm_d, a.delta, bf, a.D, prm.ldd, rows, cpw, kTS) &&
                   encode_2d(&prm.tm_b, a.Bt, bf, a.N, prm.ldbc, rows, (uint32_t)a.N, kTS) &&
                   encode_2d(&prm.tm_c, a.Ct, bf, a.N, prm.ldbc, rows, (uint32_t)a.N, kTS);
    }
    prm.timeout_ns = timeout_ns;
    prm.skip_unit = skip_unit;
    prm.delta_bias = a.delta_bias;
    prm.h0 = a.bidir ? nullptr : a.h0;
    prm.h_last = a.bidir ? nullptr : a.h_last;
    char *ws = static_cast<char *>(workspace);
    prm.ws = reinterpret_cast<WsHeader *>(ws);
    prm.flags = pl.K > 1 ? reinterpret_cast<unsigned *>(ws + kWsHeaderBytes) : nullptr;
    prm.payload = pl.K > 1 ? reinterpret_cast<float *>(ws + kWsHeaderBytes + pl.flag_bytes) : nullptr;
    prm.yscratch =
        pl.scratch_bytes ? reinterpret_cast<float *>(ws + kWsHeaderBytes + pl.desc_bytes) : nullptr;
    const bool sp = a.softplus != 0, bd = a.bidir != 0;
    return a.io_bf16 ? launch_io<__nv_bfloat16>(prm, pl, sp, bd, stream)
                     : launch_io<float>(prm, pl, sp, bd, stream);
}

}  // namespace ss
