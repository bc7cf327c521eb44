// Backward pass of the S6 selective scan (sm_103a).
//
// The forward pass ("POPCORNBENCH FW-GLM-5-1 l2_p30", forward-pass
// derivation) is, per channel (b, d) and state n,
//   dl_t = softplus(v_t) or v_t,  dA_t = exp(dl_t A),  u_t = dl_t B_t x_t,
//   h_t = dA_t h_{t-1} + u_t  (h_{-1} = h0),   y_t = sum_n C_t h_t + D x_t.
// Its exact derivative for the loss sum dy*y + sum dh_last*h_last needs the
// state h and the adjoint lam (the whole gradient of h_t) at the same t:
//   lam_t = dy_t C_t + mu_{t+1},  mu_t = dA_t lam_t  (mu_L = dh_last),
//   dC_t += dy_t h_t,  dB_t += lam_t dl_t x_t,  dx_t = D dy_t + sum lam dl B,
//   ddl_t = sum_n lam_t (B_t x_t + A (h_t - u_t)),  dA += lam (h_t - u_t) dl,
//   dh0 = mu_0,  and ddelta = ddl * sigmoid(v) under softplus.
// (h_t - u_t = dA_t h_{t-1}, so no earlier state is needed.)
//
// Layout of the gradients: time-parallel. A warp owns one channel of a
// 256-step chunk, lane l the 8 consecutive steps 8l .. 8l+7, and loops over
// the states n; h and mu for one n are warp scans (ordered shuffles) over
// the lanes' local affine maps, so no per-(t, n) tensor is stored. Four
// launches:
//   1. chunk aggregates (prod dA, forward end state from 0, adjoint entry
//      from 0) per (b, chunk, d, n), in the forward kernel's layout instead
//      (lane = channel, its 16 states in registers, steps in order);
//   2. carries: one thread per (b, d, n) walks the chunks forward (state
//      entering each chunk, from h0) and backward (adjoint leaving each
//      chunk, from dh_last; dh0 at the end);
//   3. gradients per chunk: warps of 8 consecutive channels in lockstep;
//      dB and dC, sums over d, go through shared memory in warp order into
//      per-CTA sums over the CTA's channel range;
//   4. fixed-order sums: dB, dC over the channel ranges; dA, dD over (b,
//      chunk).
// Every reduction has a fixed order, so results are bitwise reproducible.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>

#include "f32x2.cuh"
#include "s6_common.cuh"
#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr int kItems = 8;               // steps per lane
constexpr int kChunk = 32 * kItems;     // steps per chunk
constexpr int kWarps = 8;               // channels in flight per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxN = 16;
constexpr int kMaxP = kMaxN / 2;                // state pairs (f32x2)
constexpr u64 kOne2 = 0x3f8000003f800000ull;   // {1.0f, 1.0f}
constexpr unsigned kFull = 0xffffffffu;

struct BwdParams {
    const void *x, *delta, *Bt, *Ct, *dy;
    const float *A, *Dskip, *h0, *dh_last;
    void *dx, *ddelta;
    float *dA, *dBt, *dCt, *dDskip, *dh0;
    long long B, L, D;
    int N;
    int K;           // chunks per sequence
    int SD;          // channel ranges (CTAs per (b, chunk))
    int Dr;          // channels per range (multiple of kWarps)
    int softplus;
    int vec_rows;    // x, delta, dy, dx, ddelta 16-byte aligned with 16-byte rows
    int tma_rows;    // tm_x, tm_d, tm_dy hold valid tensor maps (aggregate launch)
    unsigned long long timeout_ns;
    CUtensorMap tm_x, tm_d, tm_dy;  // 3D (D, L, B) maps, box (32, kAggStage, 1)
    // workspace, each [B][K][D][N] unless noted
    float *aggP, *aggH, *aggM;   // chunk aggregates
    float *carH, *carM;          // state entering / adjoint leaving each chunk
    float *partA;                // dA partial per (b, chunk)
    float *partD;                // [B][K][D] dDskip partial per (b, chunk)
    float *partB, *partC;        // [SD][B][L][N] dB, dC partial per channel range
};

__device__ __forceinline__ float ld_io(const float *p, long long i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_io(const __nv_bfloat16 *p, long long i) {
    return __bfloat162float(p[i]);
}

// d softplus / dv = sigmoid(v); 1 above the pass-through threshold.
__device__ __forceinline__ float softplus_grad(float v) {
    return v > 20.0f ? 1.0f : 1.0f / (1.0f + ex2_approx(-v * kLog2e));
}

struct Map {  // x -> a x + b
    float a, b;
};
// p then q (p earlier in time for the forward state, the reverse order for
// the adjoint: the caller passes the map applied first as p).
__device__ __forceinline__ Map then(Map p, Map q) { return {p.a * q.a, fmaf(q.a, p.b, q.b)}; }

// Exclusive scan over lanes of maps applied in lane order (lane 0 first):
// returns the composition of lanes 0 .. l-1 (identity for lane 0).
__device__ __forceinline__ Map warp_exclusive_fwd(Map m, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float a = __shfl_up_sync(kFull, m.a, off);
        const float b = __shfl_up_sync(kFull, m.b, off);
        if (lane >= off) m = then({a, b}, m);
    }
    Map e;
    e.a = __shfl_up_sync(kFull, m.a, 1);
    e.b = __shfl_up_sync(kFull, m.b, 1);
    if (lane == 0) e = {1.0f, 0.0f};
    return e;
}
// Exclusive scan over lanes of maps applied in reverse lane order (lane 31
// first): returns the composition of lanes 31 .. l+1 (identity for lane 31).
__device__ __forceinline__ Map warp_exclusive_rev(Map m, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float a = __shfl_down_sync(kFull, m.a, off);
        const float b = __shfl_down_sync(kFull, m.b, off);
        if (lane + off < 32) m = then({a, b}, m);
    }
    Map e;
    e.a = __shfl_down_sync(kFull, m.a, 1);
    e.b = __shfl_down_sync(kFull, m.b, 1);
    if (lane == 31) e = {1.0f, 0.0f};
    return e;
}
// Sum over lanes in a fixed tree order (lane 0's result is used).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}
// One CTA: chunk k of batch b, channel range r. Shared Bt / Ct tiles of the
// chunk laid out [n][item][lane], so lane reads are conflict-free.
struct ChunkCtx {
    long long b, t0;
    int k, d0, d1;  // channels [d0, d1)
};
__device__ __forceinline__ ChunkCtx chunk_ctx(const BwdParams &p) {
    ChunkCtx c;
    const long long bk = blockIdx.x / p.SD;
    const int r = (int)(blockIdx.x % p.SD);
    c.b = bk / p.K;
    c.k = (int)(bk % p.K);
    c.t0 = (long long)c.k * kChunk;
    c.d0 = r * p.Dr;
    c.d1 = (int)min((long long)(c.d0 + p.Dr), p.D);
    return c;
}
__device__ __forceinline__ void load_bc_tiles(const BwdParams &p, const ChunkCtx &c, float *Bs,
                                              float *Cs, bool bf16) {
    const int N = p.N;
    for (int idx = threadIdx.x; idx < kChunk * N; idx += kThreads) {
        const int tl = idx / N, n = idx - tl * N;
        const long long t = c.t0 + tl;
        float bv = 0.0f, cv = 0.0f;
        if (t < p.L) {
            const long long g = (c.b * p.L + t) * N + n;
            if (bf16) {
                bv = ld_io(static_cast<const __nv_bfloat16 *>(p.Bt), g);
                cv = ld_io(static_cast<const __nv_bfloat16 *>(p.Ct), g);
            } else {
                bv = ld_io(static_cast<const float *>(p.Bt), g);
                cv = ld_io(static_cast<const float *>(p.Ct), g);
            }
        }
        const int s = n * kChunk + (tl & (kItems - 1)) * 32 + tl / kItems;  // [n][item][lane]
        Bs[s] = bv;
        Cs[s] = cv;
    }
}

// Row segments of kWarps consecutive channels (warp w takes channel
// dbase + w) for the chunk's 256 steps go through shared memory, so global
// memory sees whole segments: thread j moves step j's kWarps values of an
// array with vector accesses (8 channels: 32 B in fp32, 16 B in bf16), where
// the time-parallel layout would touch one cache line per lane and value.
// Shared layout per array: [channel][kChunk], the value of step 8l + i (lane
// l, item i) in slot i*32 + (l ^ 4i): a permutation within each item's row
// under which both the staging threads (i = j % 8, l = j / 8) and the lanes
// reading item i hit 32 distinct banks.
__device__ __forceinline__ int stage_slot(int i, int l) { return i * 32 + (l ^ (4 * i)); }
constexpr int kStageFloats = 3 * kWarps * kChunk;  // delta (as given), x, dy

__device__ __forceinline__ void load8(const float *p, long long i, bool vec, int valid, float (&v)[8]) {
    if (vec) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p + i));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p + i) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) v[w] = w < valid ? __ldg(p + i + w) : 0.0f;
    }
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, long long i, bool vec, int valid,
                                      float (&v)[8]) {
    if (vec) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p + i));
        const unsigned w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w4[k] << 16);
            v[2 * k + 1] = __uint_as_float(w4[k] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) v[w] = w < valid ? __bfloat162float(p[i + w]) : 0.0f;
    }
}
__device__ __forceinline__ void store8(float *p, long long i, bool vec, int valid, const float (&v)[8]) {
    if (vec) {
        reinterpret_cast<float4 *>(p + i)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p + i)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
#pragma unroll
        for (int w = 0; w < 8; ++w)
            if (w < valid) p[i + w] = v[w];
    }
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, long long i, bool vec, int valid,
                                       const float (&v)[8]) {
    if (vec) {
        unsigned w4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w4[k] = *reinterpret_cast<const unsigned *>(&b2);
        }
        *reinterpret_cast<uint4 *>(p + i) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    } else {
#pragma unroll
        for (int w = 0; w < 8; ++w)
            if (w < valid) p[i + w] = __float2bfloat16_rn(v[w]);
    }
}

// Stages delta, x and dy of channels [dbase, dbase + kWarps) for the chunk
// (zeros past L and past the range's last channel d1).
template <typename IO>
__device__ __forceinline__ void stage_rows(const BwdParams &p, const ChunkCtx &c, int dbase,
                                           float *stg) {
    static_assert(kWarps == 8, "row segments of 8 channels");
    const int j = threadIdx.x;
    const long long t = c.t0 + j;
    const int valid = min(kWarps, c.d1 - dbase);
    const bool vec = p.vec_rows && valid == kWarps;
    const int slot = stage_slot(j & (kItems - 1), j / kItems);
    const void *src[3] = {p.delta, p.x, p.dy};
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        float v[8];
        if (t < p.L)
            load8(static_cast<const IO *>(src[a]), (c.b * p.L + t) * p.D + dbase, vec, valid, v);
        else
#pragma unroll
            for (int w = 0; w < 8; ++w) v[w] = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) stg[(a * kWarps + w) * kChunk + slot] = v[w];
    }
}

// Writes dx (staged in the x array) and ddelta (staged in the delta array)
// of channels [dbase, dbase + kWarps) that lie below d1.
template <typename IO>
__device__ __forceinline__ void store_rows(const BwdParams &p, const ChunkCtx &c, int dbase,
                                           const float *stg) {
    const int j = threadIdx.x;
    const long long t = c.t0 + j;
    if (t >= p.L) return;
    const int valid = min(kWarps, c.d1 - dbase);
    const bool vec = p.vec_rows && valid == kWarps;
    const int slot = stage_slot(j & (kItems - 1), j / kItems);
    const long long row = (c.b * p.L + t) * p.D + dbase;
    float v[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) v[w] = stg[(1 * kWarps + w) * kChunk + slot];
    store8(static_cast<IO *>(p.dx), row, vec, valid, v);
#pragma unroll
    for (int w = 0; w < 8; ++w) v[w] = stg[(0 * kWarps + w) * kChunk + slot];
    store8(static_cast<IO *>(p.ddelta), row, vec, valid, v);
}

// This lane's 8 steps of the warp's staged channel: discretisation step, x,
// dy and delta as given (zeros past L or for an absent channel, which makes
// every map the identity).
__device__ __forceinline__ void read_items(const BwdParams &p, const ChunkCtx &c, const float *stg,
                                           bool dok, int warp, int lane, float (&dl)[kItems],
                                           float (&x)[kItems], float (&gy)[kItems],
                                           float (&v)[kItems]) {
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const int s = stage_slot(i, lane);
        v[i] = stg[(0 * kWarps + warp) * kChunk + s];
        x[i] = stg[(1 * kWarps + warp) * kChunk + s];
        gy[i] = stg[(2 * kWarps + warp) * kChunk + s];
        const bool ok = dok && c.t0 + lane * kItems + i < p.L;  // else dA = 1: an identity step
        dl[i] = ok ? (p.softplus ? softplus_mufu(v[i]) : v[i]) : 0.0f;
    }
}

// ---- launch 1: per (b, chunk, d, n) the product of dA over the chunk, the
// forward end state from zero, and the adjoint entering the chunk from zero,
// mu_in = sum_t (dA_t0 ... dA_t) dy_t C_t (the adjoint recursion mu_t =
// dA_t (dy_t C_t + mu_t+1) unrolled from mu = 0 after the chunk). Lane =
// channel with all 16 states as 8 f32x2 pairs in registers, as in the
// forward kernel, sweeping steps in order (no warp scans). A CTA is 32
// consecutive channels of one chunk; its kAggWarps warps take consecutive
// quarters of the chunk's steps, and warp 0 folds the quarters' (P, H, M)
// in time order: (P, H, M) then (P', H', M') = (P P', P' H + H', M + P M').
constexpr int kAggWarps = 4;
constexpr int kAggSteps = kChunk / kAggWarps;  // steps per warp
constexpr int kAggStage = 32;                  // steps per staged tile of x, delta, dy
constexpr int kAggSmemBase =
    (2 * kChunk * kMaxN + 3 * (kAggWarps - 1) * 32 * kMaxN) * (int)sizeof(float);  // 50 KB
// plus, per warp, one staged tile of x, delta and dy (kAggStage rows of 32
// channels each) and its mbarrier
template <typename IO>
constexpr int agg_smem() {
    return kAggSmemBase + kAggWarps * (3 * kAggStage * 32 * (int)sizeof(IO) + 16);
}

template <typename IO>
__global__ void __launch_bounds__(32 * kAggWarps, 4)
bwd_aggregate_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ __align__(128) float smem[];  // agg_smem<IO>() bytes
    float *sB = smem, *sC = smem + kChunk * kMaxN;  // [step][16], zeros past N and L
    u64 *fold = reinterpret_cast<u64 *>(sC + kChunk * kMaxN);  // [warp-1][P, H, M][pair][lane]
    const long long groups = (p.D + 31) / 32;
    const long long bk = blockIdx.x / groups;
    const long long b = bk / p.K;
    const int k = (int)(bk % p.K);
    const long long t0 = (long long)k * kChunk;
    const int steps = (int)min((long long)kChunk, p.L - t0);
    const int N = p.N;
    for (int idx = threadIdx.x; idx < kChunk * kMaxN; idx += 32 * kAggWarps) {
        const int tl = idx / kMaxN, n = idx - tl * kMaxN;
        float bv = 0.0f, cv = 0.0f;
        if (tl < steps && n < N) {
            const long long g = (b * p.L + t0 + tl) * N + n;
            bv = ld_io(static_cast<const IO *>(p.Bt), g);
            cv = ld_io(static_cast<const IO *>(p.Ct), g);
        }
        sB[idx] = bv;
        sC[idx] = cv;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long d = (blockIdx.x % groups) * 32 + lane;
    const bool dok = d < p.D;
    u64 A2[kMaxP], P[kMaxP], H[kMaxP], M[kMaxP];
#pragma unroll
    for (int q = 0; q < kMaxP; ++q) {
        const int n0 = 2 * q;
        const float a0 = dok && n0 < N ? p.A[d * N + n0] * kLog2e : 0.0f;
        const float a1 = dok && n0 + 1 < N ? p.A[d * N + n0 + 1] * kLog2e : 0.0f;
        A2[q] = f2(a0, a1);  // a missing state: dA = 1, B = C = 0, so it stays (1, 0, 0)
        P[q] = kOne2;
        H[q] = M[q] = 0ull;
    }
    // this warp's staged tiles: [x | delta | dy][kAggStage rows][32 channels]
    IO *stile = reinterpret_cast<IO *>(reinterpret_cast<unsigned char *>(smem) + kAggSmemBase) +
                warp * 3 * kAggStage * 32;
    uint64_t *sbar = reinterpret_cast<uint64_t *>(
        reinterpret_cast<unsigned char *>(smem) + kAggSmemBase +
        kAggWarps * 3 * kAggStage * 32 * (int)sizeof(IO)) + warp;
    if (p.tma_rows && lane == 0) {
        mbar_init(sbar, 1);
        fence_mbar_init();
    }
    __syncthreads();  // the Bt, Ct rows are in place
    const IO *xp = static_cast<const IO *>(p.x);
    const IO *dp = static_cast<const IO *>(p.delta);
    const IO *yp = static_cast<const IO *>(p.dy);
    const int s0 = warp * kAggSteps, s1 = min(steps, s0 + kAggSteps);
    const int d0 = (int)((blockIdx.x % groups) * 32);
    unsigned use = 0;  // staged tiles consumed (the barrier's phase)
#pragma unroll 4
    for (int tl = s0; tl < s1; ++tl) {
        float v = 0.0f, x = 0.0f, gy = 0.0f;
        if (p.tma_rows) {
            // rows of x, delta, dy of the next kAggStage steps: three tile
            // copies issued at once by one lane (zero-filled past D and L)
            const int r = (tl - s0) % kAggStage;
            if (r == 0) {
                __syncwarp();  // every lane is done with the previous tile
                if (lane == 0) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(sbar, 3u * kAggStage * 32 * (unsigned)sizeof(IO));
                    const int ty = (int)(t0 + tl);
                    tma_load_3d(stile, &p.tm_x, d0, ty, (int)b, sbar);
                    tma_load_3d(stile + kAggStage * 32, &p.tm_d, d0, ty, (int)b, sbar);
                    tma_load_3d(stile + 2 * kAggStage * 32, &p.tm_dy, d0, ty, (int)b, sbar);
                }
                mbar_wait_bounded(sbar, use & 1u, p.timeout_ns);
                ++use;
            }
            x = to_f32(stile[r * 32 + lane]);
            v = to_f32(stile[(kAggStage + r) * 32 + lane]);
            gy = to_f32(stile[(2 * kAggStage + r) * 32 + lane]);
        } else if (dok) {
            const long long g = (b * p.L + t0 + tl) * p.D + d;
            v = ld_io(dp, g);
            x = ld_io(xp, g);
            gy = ld_io(yp, g);
        }
        const float dl = dok ? (p.softplus ? softplus_mufu(v) : v) : 0.0f;
        const float u = dl * x;
        const u64 dd = f2(dl, dl), uu = f2(u, u), gg = f2(gy, gy);
        const float4 *Bq = reinterpret_cast<const float4 *>(sB + tl * kMaxN);
        const float4 *Cq = reinterpret_cast<const float4 *>(sC + tl * kMaxN);
#pragma unroll
        for (int h4 = 0; h4 < kMaxN / 4; ++h4) {
            const float4 b4 = Bq[h4], c4 = Cq[h4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q = 2 * h4 + e;
                const u64 Bp = e ? f2(b4.z, b4.w) : f2(b4.x, b4.y);
                const u64 Cp = e ? f2(c4.z, c4.w) : f2(c4.x, c4.y);
                const u64 dA = f2_exp2_scaled(dd, A2[q]);
                H[q] = f2fma(dA, H[q], f2mul(uu, Bp));
                P[q] = f2mul(P[q], dA);
                M[q] = f2fma(P[q], f2mul(gg, Cp), M[q]);
            }
        }
    }
    if (warp > 0) {
        u64 *f = fold + (warp - 1) * 3 * kMaxP * 32;
#pragma unroll
        for (int q = 0; q < kMaxP; ++q) {
            f[(0 * kMaxP + q) * 32 + lane] = P[q];
            f[(1 * kMaxP + q) * 32 + lane] = H[q];
            f[(2 * kMaxP + q) * 32 + lane] = M[q];
        }
    }
    __syncthreads();
    if (warp > 0 || !dok) return;
#pragma unroll
    for (int w = 1; w < kAggWarps; ++w) {
        const u64 *f = fold + (w - 1) * 3 * kMaxP * 32;
#pragma unroll
        for (int q = 0; q < kMaxP; ++q) {
            const u64 P2 = f[(0 * kMaxP + q) * 32 + lane];
            const u64 H2 = f[(1 * kMaxP + q) * 32 + lane];
            const u64 M2 = f[(2 * kMaxP + q) * 32 + lane];
            M[q] = f2fma(P[q], M2, M[q]);
            H[q] = f2fma(P2, H[q], H2);
            P[q] = f2mul(P[q], P2);
        }
    }
    const long long base = ((b * p.K + k) * p.D + d) * N;
#pragma unroll
    for (int q = 0; q < kMaxP; ++q) {
        const int n0 = 2 * q;
        if (n0 < N) {
            p.aggP[base + n0] = f2lo(P[q]);
            p.aggH[base + n0] = f2lo(H[q]);
            p.aggM[base + n0] = f2lo(M[q]);
        }
        if (n0 + 1 < N) {
            p.aggP[base + n0 + 1] = f2hi(P[q]);
            p.aggH[base + n0 + 1] = f2hi(H[q]);
            p.aggM[base + n0 + 1] = f2hi(M[q]);
        }
    }
}

// ---- launch 2: per (b, d, n), the state entering each chunk (from h0) and
// the adjoint leaving each chunk (from dh_last), chunk by chunk in order;
// dh0 is the adjoint left at the sequence's start.
__global__ void bwd_carry_kernel(const BwdParams p) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = p.B * p.D * p.N;
    if (i >= total) return;
    const long long b = i / (p.D * p.N), dn = i - b * p.D * p.N;  // dn = d*N + n
    const long long stride = p.D * p.N;
    const long long base = b * p.K * stride + dn;
    float h = p.h0 ? p.h0[i] : 0.0f;
    for (int k = 0; k < p.K; ++k) {
        const long long idx = base + k * stride;
        p.carH[idx] = h;
        h = fmaf(p.aggP[idx], h, p.aggH[idx]);
    }
    float mu = p.dh_last ? p.dh_last[i] : 0.0f;
    for (int k = p.K - 1; k >= 0; --k) {
        const long long idx = base + k * stride;
        p.carM[idx] = mu;
        mu = fmaf(p.aggP[idx], mu, p.aggM[idx]);
    }
    if (p.dh0) p.dh0[i] = mu;
}

constexpr int kGradSmem =
    ((4 * kMaxN + 2 * kWarps) * kChunk + kWarps * 3 * kMaxN + kStageFloats) *
    (int)sizeof(float);  // 105.5 KB

// ---- launch 3: gradients of one chunk for a channel range. Warp w takes
// channels d0 + w, d0 + w + 8, ...; per state n each warp rebuilds h over its
// steps (warp scan from the chunk's entering state) and runs the adjoint
// back over them (warp scan from the chunk's leaving adjoint), accumulating
// the per-step terms. dB and dC contributions of the 8 warps meet in shared
// memory and are added in warp order; the CTA's channel-range sums are
// written once at the end.
template <typename IO>
__global__ void __launch_bounds__(kThreads) bwd_grad_kernel(const BwdParams p) {
    extern __shared__ __align__(128) float smem[];  // kGradSmem bytes
    float *Bs = smem, *Cs = Bs + kMaxN * kChunk;
    float *accB = Cs + kMaxN * kChunk, *accC = accB + kMaxN * kChunk;  // [n][item][lane]
    float *redB = accC + kMaxN * kChunk, *redC = redB + kWarps * kChunk;  // [warp][item][lane]
    float *spar = redC + kWarps * kChunk;  // [warp][A, entering state, leaving adjoint][n]
    float *stg = spar + kWarps * 3 * kMaxN;  // staged rows of the current 8 channels
    const ChunkCtx c = chunk_ctx(p);
    load_bc_tiles(p, c, Bs, Cs, sizeof(IO) == 2);
    for (int i = threadIdx.x; i < kMaxN * kChunk; i += kThreads) accB[i] = accC[i] = 0.0f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N;
    float *par = spar + warp * 3 * kMaxN;

    for (int dbase = c.d0; dbase < c.d1; dbase += kWarps) {
        const int d = dbase + warp;
        const bool dok = d < c.d1;  // warp-uniform; absent channels add zeros
        // this channel's A and carries for every n, read once
        if (lane < N) {
            const long long cidx = ((c.b * p.K + c.k) * p.D + d) * N + lane;
            par[lane] = dok ? p.A[(long long)d * N + lane] : 0.0f;
            par[kMaxN + lane] = dok ? p.carH[cidx] : 0.0f;
            par[2 * kMaxN + lane] = dok ? p.carM[cidx] : 0.0f;
        }
        if (dbase > c.d0) __syncthreads();  // the previous block's rows are stored
        stage_rows<IO>(p, c, dbase, stg);
        __syncthreads();
        float dl[kItems], x[kItems], gy[kItems], v[kItems], xdl[kItems];
        read_items(p, c, stg, dok, warp, lane, dl, x, gy, v);
        // S = sum_n lam B (dx = dl S, ddelta gets x S), G = sum_n lam dA h_prev A
        float S[kItems], G[kItems];
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            xdl[i] = dl[i] * x[i];
            S[i] = G[i] = 0.0f;
        }
        __syncwarp();

        for (int n = 0; n < N; ++n) {
            const float An = par[n], A2 = An * kLog2e;
            const float hs = par[kMaxN + n];      // state entering the chunk
            const float me = par[2 * kMaxN + n];  // adjoint leaving it
            float dA[kItems], u[kItems], g[kItems], Bv[kItems], h[kItems];
            Map f = {1.0f, 0.0f};
#pragma unroll
            for (int i = 0; i < kItems; ++i) {
                Bv[i] = Bs[n * kChunk + i * 32 + lane];
                dA[i] = ex2_approx(dl[i] * A2);
                u[i] = xdl[i] * Bv[i];
                g[i] = gy[i] * Cs[n * kChunk + i * 32 + lane];
                f = {f.a * dA[i], fmaf(dA[i], f.b, u[i])};
            }
            const Map ef = warp_exclusive_fwd(f, lane);
            const float s = fmaf(ef.a, hs, ef.b);  // state before this lane's first step
            float hc = s;
#pragma unroll
            for (int i = 0; i < kItems; ++i) h[i] = hc = fmaf(dA[i], hc, u[i]);
            float m = 0.0f;  // adjoint map of the lane's steps: mu -> f.a mu + m
#pragma unroll
            for (int i = kItems - 1; i >= 0; --i) m = dA[i] * (g[i] + m);
            const Map er = warp_exclusive_rev({f.a, m}, lane);
            float mu = fmaf(er.a, me, er.b);  // adjoint after this lane's last step
            float dAp = 0.0f;
#pragma unroll
            for (int i = kItems - 1; i >= 0; --i) {
                const float lam = g[i] + mu;  // gradient of h_t
                const float tA = lam * (dA[i] * (i > 0 ? h[i - 1] : s));  // through dA_t
                S[i] = fmaf(lam, Bv[i], S[i]);
                G[i] = fmaf(tA, An, G[i]);
                dAp = fmaf(tA, dl[i], dAp);
                redB[warp * kChunk + i * 32 + lane] = lam * xdl[i];
                redC[warp * kChunk + i * 32 + lane] = gy[i] * h[i];
                mu = dA[i] * lam;
            }
            dAp = warp_sum(dAp);
            if (dok && lane == 0) p.partA[((c.b * p.K + c.k) * p.D + d) * N + n] = dAp;
            __syncthreads();
            // this chunk's dB, dC for state n: the 8 warps' terms in warp order
            {
                const int j = threadIdx.x;  // [item][lane] position
                float sb = accB[n * kChunk + j], sc = accC[n * kChunk + j];
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    sb += redB[w * kChunk + j];
                    sc += redC[w * kChunk + j];
                }
                accB[n * kChunk + j] = sb;
                accC[n * kChunk + j] = sc;
            }
            __syncthreads();
        }
        // dx and ddelta into this lane's staged x and delta slots (only its
        // own slots: no other thread reads them before the barrier below)
        const float Dd = dok && p.Dskip ? p.Dskip[d] : 0.0f;
        float sdx = 0.0f;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            const int sl = stage_slot(i, lane);
            const float gdl = fmaf(x[i], S[i], G[i]);
            sdx = fmaf(gy[i], x[i], sdx);
            stg[(1 * kWarps + warp) * kChunk + sl] = fmaf(gy[i], Dd, dl[i] * S[i]);
            stg[(0 * kWarps + warp) * kChunk + sl] = p.softplus ? gdl * softplus_grad(v[i]) : gdl;
        }
        sdx = warp_sum(sdx);
        if (dok && lane == 0) p.partD[(c.b * p.K + c.k) * p.D + d] = sdx;
        __syncthreads();  // the block's dx, ddelta are staged
        store_rows<IO>(p, c, dbase, stg);
    }
    // this channel range's dB, dC over the chunk
    const int r = (int)(blockIdx.x % p.SD);
    for (int idx = threadIdx.x; idx < N * kChunk; idx += kThreads) {
        const int n = idx / kChunk, j = idx - n * kChunk;
        const int tl = (j & 31) * kItems + (j >> 5);  // lane * 8 + item
        const long long t = c.t0 + tl;
        if (t < p.L) {
            const long long o = (((long long)r * p.B + c.b) * p.L + t) * N + n;
            p.partB[o] = accB[idx];
            p.partC[o] = accC[idx];
        }
    }
}

// ---- launch 4: the remaining sums, each in a fixed order: dBt, dCt over
// the channel ranges; dA and dDskip over (b, chunk).
__global__ void bwd_final_kernel(const BwdParams p) {
    const long long nBC = p.B * p.L * p.N, nA = p.D * p.N, nD = p.dDskip ? p.D : 0;
    const long long total = nBC + nA + nD;
    const long long BK = p.B * p.K;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        if (i < nBC) {
            float sb = 0.0f, sc = 0.0f;
            for (int r = 0; r < p.SD; ++r) {
                sb += p.partB[(long long)r * nBC + i];
                sc += p.partC[(long long)r * nBC + i];
            }
            p.dBt[i] = sb;
            p.dCt[i] = sc;
        } else if (i < nBC + nA) {
            const long long dn = i - nBC;
            float s = 0.0f;
            for (long long bk = 0; bk < BK; ++bk) s += p.partA[bk * nA + dn];
            p.dA[dn] = s;
        } else {
            const long long d = i - nBC - nA;
            float s = 0.0f;
            for (long long bk = 0; bk < BK; ++bk) s += p.partD[bk * p.D + d];
            p.dDskip[d] = s;
        }
    }
}

// ------------------------------------------------------------------ planning
struct BwdPlan {
    int K, SD, Dr;
    size_t off[9];  // section offsets: aggP aggH aggM carH carM partA partD partB partC
    size_t total;
};

BwdPlan bwd_plan(int64_t B, int64_t L, int64_t D, int64_t N) {
    BwdPlan pl{};
    pl.K = (int)((L + kChunk - 1) / kChunk);
    // Channel ranges per (b, chunk): the gradient launch (the longest) fits
    // 2 CTAs per SM (128 registers x 256 threads, and its shared memory), so
    // pick the split that minimises waves x (channels per CTA + 16, the
    // per-CTA tile loads and range sums in channel-equivalents): a last wave
    // that only a few CTAs occupy costs as much as a full one.
    const long long groups = (D + kWarps - 1) / kWarps;
    const long long per_sm =
        std::max<long long>(1, std::min<long long>(2, device_smem_per_sm() / (kGradSmem + 1024)));
    const long long slots = (long long)device_sm_count() * per_sm;
    long long best_cost = -1, best_Dr = groups * kWarps;
    for (long long sd = 1; sd <= std::min<long long>(groups, 64); ++sd) {
        const long long Dr = (groups + sd - 1) / sd * kWarps;
        const long long ctas = B * pl.K * ((D + Dr - 1) / Dr);
        const long long cost = (ctas + slots - 1) / slots * (Dr + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_Dr = Dr;
        }
    }
    pl.Dr = (int)best_Dr;
    pl.SD = (int)((D + pl.Dr - 1) / pl.Dr);
    const size_t bkdn = (size_t)B * pl.K * D * N * sizeof(float);
    const size_t sizes[9] = {bkdn, bkdn, bkdn, bkdn, bkdn, bkdn,
                             (size_t)B * pl.K * D * sizeof(float),
                             (size_t)pl.SD * B * L * N * sizeof(float),
                             (size_t)pl.SD * B * L * N * sizeof(float)};
    size_t o = 0;
    for (int i = 0; i < 9; ++i) {
        pl.off[i] = o;
        o += (sizes[i] + 255) / 256 * 256;
    }
    pl.total = o;
    return pl;
}

}  // namespace

size_t s6_bwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N) {
    if (B <= 0 || L <= 0 || D <= 0 || N <= 0) return 0;
    return bwd_plan(B, L, D, N).total;
}

ss_status s6_bwd_launch(const S6BwdArgs &a, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    const BwdPlan pl = bwd_plan(a.B, a.L, a.D, a.N);
    if (workspace == nullptr || ws_bytes < pl.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SS_ERR_WORKSPACE;
    BwdParams p{};
    p.x = a.x;
    p.delta = a.delta;
    p.Bt = a.Bt;
    p.Ct = a.Ct;
    p.dy = a.dy;
    p.A = a.A;
    p.Dskip = a.Dskip;
    p.h0 = a.h0;
    p.dh_last = a.dh_last;
    p.dx = a.dx;
    p.ddelta = a.ddelta;
    p.dA = a.dA;
    p.dBt = a.dBt;
    p.dCt = a.dCt;
    p.dDskip = a.dDskip;
    p.dh0 = a.dh0;
    p.B = a.B;
    p.L = a.L;
    p.D = a.D;
    p.N = (int)a.N;
    p.K = pl.K;
    p.SD = pl.SD;
    p.Dr = pl.Dr;
    p.softplus = a.softplus;
    {
        const uintptr_t es = a.io_bf16 ? 2 : 4;
        const uintptr_t ptrs = reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.delta) |
                               reinterpret_cast<uintptr_t>(a.dy) | reinterpret_cast<uintptr_t>(a.dx) |
                               reinterpret_cast<uintptr_t>(a.ddelta);
        p.vec_rows = (ptrs & 15u) == 0 && ((uintptr_t)a.D * es) % 16 == 0;
        p.timeout_ns = spin_timeout_ns();
        const uint64_t dims[3] = {(uint64_t)a.D, (uint64_t)a.L, (uint64_t)a.B};
        const uint64_t strides[2] = {(uint64_t)a.D * es, (uint64_t)(a.L * a.D) * es};
        const uint32_t box[3] = {32u, (uint32_t)kAggStage, 1u};
        const bool bf = a.io_bf16 != 0;
        p.tma_rows = p.vec_rows && encode_tiled_map(&p.tm_x, a.x, bf, 3, dims, strides, box) &&
                     encode_tiled_map(&p.tm_d, a.delta, bf, 3, dims, strides, box) &&
                     encode_tiled_map(&p.tm_dy, a.dy, bf, 3, dims, strides, box);
    }
    char *ws = static_cast<char *>(workspace);
    float **sec[9] = {&p.aggP, &p.aggH, &p.aggM, &p.carH, &p.carM, &p.partA, &p.partD, &p.partB, &p.partC};
    for (int i = 0; i < 9; ++i) *sec[i] = reinterpret_cast<float *>(ws + pl.off[i]);
    const long long grid = a.B * pl.K * pl.SD;
    if (grid > 0x7fffffffLL) return SS_ERR_UNSUPPORTED;
    const long long agg_grid = a.B * pl.K * ((a.D + 31) / 32);
    if (agg_grid > 0x7fffffffLL) return SS_ERR_UNSUPPORTED;
    auto agg = a.io_bf16 ? bwd_aggregate_kernel<__nv_bfloat16> : bwd_aggregate_kernel<float>;
    const int agg_smem_bytes = a.io_bf16 ? agg_smem<__nv_bfloat16>() : agg_smem<float>();
    if (raise_smem_limit(reinterpret_cast<const void *>(agg), agg_smem_bytes) != SS_OK)
        return SS_ERR_CUDA;
    agg<<<(unsigned)agg_grid, 32 * kAggWarps, agg_smem_bytes, stream>>>(p);
    const long long chains = a.B * a.D * a.N;
    bwd_carry_kernel<<<(unsigned)((chains + 255) / 256), 256, 0, stream>>>(p);
    auto grad = a.io_bf16 ? bwd_grad_kernel<__nv_bfloat16> : bwd_grad_kernel<float>;
    if (raise_smem_limit(reinterpret_cast<const void *>(grad), kGradSmem) != SS_OK)
        return SS_ERR_CUDA;
    grad<<<(unsigned)grid, kThreads, kGradSmem, stream>>>(p);
    bwd_final_kernel<<<device_sm_count() * 8, 256, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace ss
