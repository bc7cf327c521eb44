// Single-pass S6 selective-scan forward on a skewed wavefront (sm_103a).
//
// "POPCORNBENCH FW-GLM-5-1 l2_p30" (arjun-banerjee.github.io), forward-pass
// derivation: dA = exp(delta*A), dBx = delta*B_t*x, h = dA*h + dBx,
// y_t = sum_n h*C_t + D*x. Every (b, t, d, n) term's exp is computed once and
// every input is read once:
//
//  * a CTA owns 32 channels (lane = channel) and walks all of L in blocks of
//    R = S*T steps; warp s owns the T steps [s*T, s*T + T) of every block
//    (its time slice), so the 32 channels' rows are read by one warp at a
//    time: x / delta / y accesses are conflict-free and the B_t / C_t values
//    of a step are one broadcast load for the whole warp;
//  * the 16 states are taken as 8 pairs (one f32x2 register each), handled
//    two at a time (pairs k and k + 4: an item, two independent chains). The
//    state of an item's pairs leaving slice s of block j is the state
//    entering slice s + 1 (or slice 0 of block j + 1), so the work is
//    pipelined as a skewed wavefront: warp s handles item k of block j
//    (m = 4j + k) one item after warp s - 1 did. Its entering state comes
//    from warp s - 1 through shared memory (double-buffered, with full /
//    empty mbarriers between the two warps only), or for slice 0 from the
//    last warp's item four items earlier (kept per channel and pair), so
//    every warp runs the plain recurrence over its T steps from the exact
//    state: no second pass, no scan, no stored dA (issuing an item's exps
//    before its wait for the entering state measured slower: the registers
//    they hold cost more than the latency they hide);
//  * a warp enters block j all its lanes at once: it stores y of block
//    j - 1 and loads delta, x and its slice of B_t / C_t of block j;
//  * x and delta tiles (R rows x 32 channels) arrive by 3D TMA tile copies
//    into a 2-stage ring, B_t / C_t tiles (R rows x 16 states) likewise into
//    a 2-stage staging ring, from which each warp writes its slice as fp32
//    laid out per pair so that one broadcast 16-byte load gives a pair's
//    values for two steps; y leaves by 3D TMA tile stores (clipped at L and
//    D). One thread issues every copy, when the last warp has entered a
//    block (so every warp is done with the stage it refills).
//
// Results are bitwise reproducible: the order of every operation is fixed.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "f32x2.cuh"
#include "s6_common.cuh"
#include "s6_ws.h"
#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr int kCH = 32;     // channels per CTA (lane = channel)
constexpr int kPairs = 8;   // state pairs (16 states; fewer are zero-padded)
constexpr int kItems = 4;   // wavefront items per block (two state pairs each)
constexpr int kNX = 2;      // x / delta stages
constexpr int kNBS = 2;     // B_t / C_t staging stages
constexpr int kNY = 3;      // y tiles

template <int T, int S> struct WSShape {
    static_assert(S >= 2 && S <= kItems, "the skew needs items per block >= slices");
    static constexpr int R = S * T;          // steps per block
    static constexpr int P2 = (T + 1) / 2;   // step pairs per slice

};

struct WSParams {
    CUtensorMap tm_x, tm_d, tm_y, tm_b, tm_c;  // 3D (inner, L, B) maps
    const float *A, *Dskip, *delta_bias, *h0;
    float *h_last;
    WsHeader *ws;
    long long L, D;
    int N, nblk, dgroups;
    unsigned long long timeout_ns;
};

struct WSSmem {
    int xt, bt, wc, off_d, off_bs, off_bc, off_y, off_hs, off_cs, off_a2, off_dsk, off_db,
        off_bar, total;
};
// Barriers after the TMA ones: hand-off full / empty per (slice, parity),
// carry full per pair.
__host__ __device__ constexpr int ws_nbars(int S) { return kNX + kNBS + 4 * S + kItems; }
__host__ __device__ inline WSSmem ws_smem(int R, int S, int es, int wc) {
    WSSmem m;
    m.xt = (R * kCH * es + 127) / 128 * 128;  // one x (or delta, or y) tile
    m.bt = (R * 16 * es + 127) / 128 * 128;   // one B_t (or C_t) staging tile
    m.wc = wc;                                // one warp's fp32 B_t / C_t slice
    m.off_d = kNX * m.xt;
    m.off_bs = 2 * kNX * m.xt;
    m.off_bc = m.off_bs + kNBS * 2 * m.bt;
    m.off_y = m.off_bc + S * wc;
    m.off_hs = m.off_y + kNY * m.xt;
    m.off_cs = m.off_hs + 2 * S * 2 * kCH * 8;
    m.off_a2 = m.off_cs + kCH * kPairs * 8;
    m.off_dsk = m.off_a2 + kCH * kPairs * 8;
    m.off_db = m.off_dsk + kCH * 4;
    m.off_bar = (m.off_db + kCH * 4 + 7) / 8 * 8;
    m.total = m.off_bar + ws_nbars(S) * 8 + 16;  // + the abort word and the issue count
    return m;
}

__device__ __forceinline__ float ld_smem_io(const float *p) { return *p; }
__device__ __forceinline__ float ld_smem_io(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
// Two adjacent values (p aligned to two elements), widened to fp32.
__device__ __forceinline__ float2 ld_smem_io2(const float *p) {
    return *reinterpret_cast<const float2 *>(p);
}
__device__ __forceinline__ float2 ld_smem_io2(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

// 12 resident warps per SM (170 registers a thread): three four-warp CTAs.
template <typename IO, int T, int S, bool SP>
__global__ void __launch_bounds__(S * 32, 12 / S) s6_ws_kernel(const __grid_constant__ WSParams p) {
    static_assert(S >= 2, "the hand-off needs two warps or more");
    using C = WSShape<T, S>;
    constexpr int R = C::R, P2 = C::P2;
    constexpr int WC = 2 * kPairs * P2 * 16;  // a warp's fp32 B_t / C_t slice of a block
    constexpr int NT = S * 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    const WSSmem L_ = ws_smem(R, S, (int)sizeof(IO), WC);
    u64 *hs = reinterpret_cast<u64 *>(sm + L_.off_hs);    // [2][S][2][32] slice hand-off
    u64 *cs = reinterpret_cast<u64 *>(sm + L_.off_cs);    // [8][32] block carries, per pair
    u64 *a2s = reinterpret_cast<u64 *>(sm + L_.off_a2);   // [8][32] A * log2(e), per pair
    float *dsk = reinterpret_cast<float *>(sm + L_.off_dsk);
    float *dbs = reinterpret_cast<float *>(sm + L_.off_db);
    uint64_t *xbar = reinterpret_cast<uint64_t *>(sm + L_.off_bar);  // TMA: x, delta (kNX)
    uint64_t *bbar = xbar + kNX;                                      // TMA: B_t, C_t (kNBS)
    uint64_t *hfull = bbar + kNBS;                                    // [S][2] hand-off written
    uint64_t *hempty = hfull + 2 * S;                                 // [S][2] hand-off read
    uint64_t *cfull = hempty + 2 * S;                                 // [4] carries written
    volatile int *abort_word = reinterpret_cast<volatile int *>(cfull + kItems);
    volatile int *issued = abort_word + 1;  // blocks whose tiles were requested

    const int tid = threadIdx.x, s = tid >> 5, c = tid & 31;
    const long long b = blockIdx.x / p.dgroups;
    const long long d0 = (long long)(blockIdx.x % p.dgroups) * kCH;
    const int N = p.N;
    const long long D = p.D, L = p.L;
    const int nblk = p.nblk;

    for (int i = tid; i < kCH * kPairs; i += NT) {  // i = pair * 32 + channel
        const long long dd = d0 + (i & 31);
        const int n = 2 * (i >> 5);
        float a[2], h[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool ok = dd < D && n + e < N;
            a[e] = ok ? p.A[dd * N + n + e] * kLog2e : 0.0f;
            h[e] = (ok && p.h0) ? p.h0[(b * D + dd) * N + n + e] : 0.0f;
        }
        a2s[i] = f2(a[0], a[1]);
        cs[i] = f2(h[0], h[1]);
    }
    for (int i = tid; i < kCH; i += NT) {
        const long long dd = d0 + i;
        dsk[i] = (dd < D && p.Dskip) ? p.Dskip[dd] : 0.0f;
        dbs[i] = (dd < D && p.delta_bias) ? p.delta_bias[dd] : 0.0f;
    }
    if (tid == 0) {
        for (int k = 0; k < kNX + kNBS; ++k) mbar_init(xbar + k, 1);
        for (int k = 0; k < 4 * S + kItems; ++k) mbar_init(hfull + k, 32);  // one warp arrives
        *abort_word = 0;
        *issued = 0;
        fence_mbar_init();
    }
    __syncthreads();

    constexpr unsigned kXBytes = 2u * (unsigned)(R * kCH * (int)sizeof(IO));
    constexpr unsigned kBBytes = 2u * (unsigned)(R * 16 * (int)sizeof(IO));
    // block j's x, delta, B_t and C_t tiles into stage j % 2; one thread (the
    // first of the last warp) issues every tile copy and store of the CTA
    const bool issuer = tid == 32 * (S - 1);
    auto issue_tiles = [&](int j) {
        *issued = j + 1;
        const int st = j % kNX;
        mbar_arrive_expect_tx(xbar + st, kXBytes);
        tma_load_3d(sm + st * L_.xt, &p.tm_x, (int)d0, j * R, (int)b, xbar + st);
        tma_load_3d(sm + L_.off_d + st * L_.xt, &p.tm_d, (int)d0, j * R, (int)b, xbar + st);
        unsigned char *dst = sm + L_.off_bs + st * 2 * L_.bt;
        mbar_arrive_expect_tx(bbar + st, kBBytes);
        tma_load_3d(dst, &p.tm_b, 0, j * R, (int)b, bbar + st);
        tma_load_3d(dst + L_.bt, &p.tm_c, 0, j * R, (int)b, bbar + st);
    };
    if (issuer)
        for (int j = 0; j < kNX && j < nblk; ++j) issue_tiles(j);

    // Bounded wait that gives up at once when another warp already did.
    auto wait = [&](uint64_t *bar, unsigned parity, unsigned where) {
        if (mbar_try_wait(bar, parity)) return;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (*abort_word) return;
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                record_error(p.ws, SS_ERR_TIMEOUT, where, blockIdx.x, parity);
                *abort_word = 1;
                return;
            }
        }
    };

    const float Dd = dsk[c];
    const float dbias = dbs[c];
    // this lane's share of the B_t / C_t widening (the same every block):
    // entries it = c + 32 w of wbc, each from rows r, r + 1 (r = 2 ip) and
    // states 2k, 2k + 1 of tile m
    constexpr int kWiden = (2 * kPairs * P2 + 31) / 32;
    int wsrc[kWiden];
    bool wtwo[kWiden], wok[kWiden];
#pragma unroll
    for (int w = 0; w < kWiden; ++w) {
        const int it = c + 32 * w;
        const int ip = it % P2, k = (it / P2) % kPairs, m = it / (P2 * kPairs);
        wok[w] = it < 2 * kPairs * P2;
        wtwo[w] = 2 * ip + 1 < T;
        wsrc[w] = m * (L_.bt / (int)sizeof(IO)) + 2 * ip * 16 + 2 * k;
    }
    const int row0 = s * T;                                               // this slice's first row
    float4 *wbc = reinterpret_cast<float4 *>(sm + L_.off_bc + s * WC);   // this warp's B_t / C_t
    u64 ddl[T], uu[T], yv[T];

    // y of this warp's slice of block j (yv) into the y tile
    auto store_y = [&](int j) {
        IO *yt = reinterpret_cast<IO *>(sm + L_.off_y + (j % kNY) * L_.xt) + row0 * kCH + c;
#pragma unroll
        for (int i = 0; i < T; ++i) store_smem(yt + i * kCH, f2lo(yv[i]) + f2hi(yv[i]));
        fence_proxy_async_smem();
    };

    for (int j = 0; j < nblk; ++j) {
        // ---- entering block j: y of block j - 1 out; delta, x and this
        // slice's B_t / C_t of block j in
        if (j > 0) store_y(j - 1);
        const int st = j % kNX;
        wait(xbar + st, (unsigned)(j / kNX) & 1u, 11u);
        {
            const IO *xt = reinterpret_cast<const IO *>(sm + st * L_.xt) + row0 * kCH + c;
            const IO *dt = reinterpret_cast<const IO *>(sm + L_.off_d + st * L_.xt) + row0 * kCH + c;
            const long long lim = L - (long long)j * R - row0;  // steps of this slice inside L
            auto enter = [&](auto whole) {
#pragma unroll
                for (int i = 0; i < T; ++i) {
                    float dv = ld_smem_io(dt + i * kCH) + dbias;
                    if constexpr (SP) dv = softplus_mufu(dv);
                    if (!decltype(whole)::value && i >= lim) dv = 0.0f;  // past L: dA = 1, no input
                    const float xv = ld_smem_io(xt + i * kCH);
                    const float u = dv * xv;
                    ddl[i] = f2(dv, dv);
                    uu[i] = f2(u, u);
                    yv[i] = f2(Dd * xv, 0.0f);
                }
            };
            if (lim >= T)
                enter(std::true_type{});  // every block but possibly the last
            else
                enter(std::false_type{});
        }
        wait(bbar + st, (unsigned)(j / kNX) & 1u, 10u);
        {
            // widen this slice's rows into wbc[(m*kPairs + k)*P2 + ip] =
            // {M[r][2k], M[r][2k+1], M[r+1][2k], M[r+1][2k+1]}, r = 2*ip
            const IO *bs = reinterpret_cast<const IO *>(sm + L_.off_bs + st * 2 * L_.bt) + row0 * 16;
#pragma unroll
            for (int w = 0; w < kWiden; ++w) {
                if (!wok[w]) continue;
                const IO *M = bs + wsrc[w];
                const float2 r0 = ld_smem_io2(M);
                const float2 r1 = wtwo[w] ? ld_smem_io2(M + 16) : make_float2(0.0f, 0.0f);
                wbc[c + 32 * w] = make_float4(r0.x, r0.y, r1.x, r1.y);
            }
            __syncwarp();
        }
        // ---- the 4 items of block j, each two state pairs (k and k + 4):
        // two independent chains; item m = 4j + k
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            const int m = j * kItems + k;
            const int q = k & 1;  // == m & 1: the hand-off buffer of this item
            const u64 A2a = a2s[k * kCH + c], A2b = a2s[(k + kItems) * kCH + c];
            // the exps do not depend on the entering state: issued before
            // the hand-off wait
            u64 ha, hb;
            if (s == 0) {
                if (j > 0) wait(cfull + k, (unsigned)(j - 1) & 1u, 12u);
                ha = cs[k * kCH + c];
                hb = cs[(k + kItems) * kCH + c];
            } else {
                wait(hfull + (s - 1) * 2 + q, (unsigned)(m >> 1) & 1u, 13u);
                ha = hs[((q * S + s - 1) * 2) * kCH + c];
                hb = hs[((q * S + s - 1) * 2 + 1) * kCH + c];
                mbar_arrive(hempty + (s - 1) * 2 + q);
            }
            if (s == S - 1 && k == 0) {
                // every warp has entered block j (its item (j, 0) is done):
                // stage j % 2 takes block j + 2, and block j - 1's y tile is
                // complete
                if (issuer) {
                    if (j + kNX < nblk) issue_tiles(j + kNX);
                    if (j > 0) {
                        tma_store_3d(&p.tm_y, sm + L_.off_y + ((j - 1) % kNY) * L_.xt, (int)d0,
                                     (j - 1) * R, (int)b);
                        bulk_commit();
                        // every store but this one has read its tile: block j - 3's
                        // tile takes block j's y (written as warps enter j + 1, after
                        // this warp's item (j - 1, 0))
                        bulk_wait_read<1>();
                    }
                }
                __syncwarp();
            }
            const ulonglong2 *ba = reinterpret_cast<const ulonglong2 *>(wbc + k * P2);
            const ulonglong2 *bb = reinterpret_cast<const ulonglong2 *>(wbc + (k + kItems) * P2);
            const ulonglong2 *ca = reinterpret_cast<const ulonglong2 *>(wbc + (kPairs + k) * P2);
            const ulonglong2 *cb = reinterpret_cast<const ulonglong2 *>(wbc + (kPairs + k + kItems) * P2);
#pragma unroll
            for (int ip = 0; ip < P2; ++ip) {
                const ulonglong2 b4a = ba[ip], b4b = bb[ip], c4a = ca[ip], c4b = cb[ip];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = 2 * ip + e;
                    if (i < T) {
                        ha = f2fma(f2_exp2_scaled(ddl[i], A2a), ha, f2mul(uu[i], e ? b4a.y : b4a.x));
                        hb = f2fma(f2_exp2_scaled(ddl[i], A2b), hb, f2mul(uu[i], e ? b4b.y : b4b.x));
                        yv[i] = f2fma(e ? c4a.y : c4a.x, ha, yv[i]);
                        yv[i] = f2fma(e ? c4b.y : c4b.x, hb, yv[i]);
                    }
                }
            }
            if (s == S - 1) {
                cs[k * kCH + c] = ha;
                cs[(k + kItems) * kCH + c] = hb;
                mbar_arrive(cfull + k);
            } else {
                if (m >= 2) wait(hempty + s * 2 + q, (unsigned)((m >> 1) - 1) & 1u, 14u);
                hs[((q * S + s) * 2) * kCH + c] = ha;
                hs[((q * S + s) * 2 + 1) * kCH + c] = hb;
                mbar_arrive(hfull + s * 2 + q);
            }
        }
    }
    // the last block's y (every warp's slice), then its store
    store_y(nblk - 1);
    __syncthreads();
    const bool aborted = *abort_word != 0;
    if (issuer) {
        if (!aborted) {
            tma_store_3d(&p.tm_y, sm + L_.off_y + ((nblk - 1) % kNY) * L_.xt, (int)d0,
                         (nblk - 1) * R, (int)b);
            bulk_commit();
        }
        bulk_wait<0>();
        if (aborted) {
            // tile copies still in flight land before the CTA exits: the last
            // one issued into each stage (a wait on a phase that already
            // completed returns at once)
            const int n = *issued;
            for (int jj = n > kNX ? n - kNX : 0; jj < n; ++jj) {
                mbar_wait_bounded(xbar + jj % kNX, (unsigned)(jj / kNX) & 1u, p.timeout_ns);
                mbar_wait_bounded(bbar + jj % kNX, (unsigned)(jj / kNX) & 1u, p.timeout_ns);
            }
        }
    }
    __syncthreads();
    if (p.h_last && !aborted) {
        for (int i = tid; i < kCH * kPairs; i += NT) {
            const long long dd = d0 + (i & 31);
            const int n = 2 * (i >> 5);
            if (dd < D && n < N) p.h_last[(b * D + dd) * N + n] = f2lo(cs[i]);
            if (dd < D && n + 1 < N) p.h_last[(b * D + dd) * N + n + 1] = f2hi(cs[i]);
        }
    }
}

template <typename IO, int T, int S>
ss_status launch_shape(const S6Args &a, const WSPlan &pl, void *workspace, cudaStream_t stream,
                       unsigned long long timeout_ns) {
    using C = WSShape<T, S>;
    const bool bf = sizeof(IO) == 2;
    const uint64_t es = bf ? 2 : 4;
    WSParams prm{};
    const long long ldd = a.ld_delta > 0 ? a.ld_delta : a.D;
    const long long ldbc = a.ld_bc > 0 ? a.ld_bc : a.N;
    const uint64_t dx[3] = {(uint64_t)a.D, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t sx[2] = {(uint64_t)a.D * es, (uint64_t)(a.L * a.D) * es};
    const uint64_t sd[2] = {(uint64_t)ldd * es, (uint64_t)(a.L * ldd) * es};
    const uint64_t db[3] = {(uint64_t)a.N, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t sb[2] = {(uint64_t)ldbc * es, (uint64_t)(a.L * ldbc) * es};
    const uint32_t box[3] = {(uint32_t)kCH, (uint32_t)C::R, 1u};
    const uint32_t boxb[3] = {16u, (uint32_t)C::R, 1u};
    if (!encode_tiled_map(&prm.tm_x, a.x, bf, 3, dx, sx, box) ||
        !encode_tiled_map(&prm.tm_d, a.delta, bf, 3, dx, sd, box) ||
        !encode_tiled_map(&prm.tm_y, a.y, bf, 3, dx, sx, box) ||
        !encode_tiled_map(&prm.tm_b, a.Bt, bf, 3, db, sb, boxb) ||
        !encode_tiled_map(&prm.tm_c, a.Ct, bf, 3, db, sb, boxb))
        return SS_ERR_CUDA;
    prm.ws = static_cast<WsHeader *>(workspace);
    prm.A = a.A;
    prm.Dskip = a.Dskip;
    prm.delta_bias = a.delta_bias;
    prm.h0 = a.h0;
    prm.h_last = a.h_last;
    prm.L = a.L;
    prm.D = a.D;
    prm.N = (int)a.N;
    prm.nblk = pl.nblk;
    prm.dgroups = pl.dgroups;
    prm.timeout_ns = timeout_ns;
    auto kern = a.softplus ? s6_ws_kernel<IO, T, S, true> : s6_ws_kernel<IO, T, S, false>;
    if (raise_smem_limit(reinterpret_cast<const void *>(kern), (int)pl.smem) != SS_OK)
        return SS_ERR_CUDA;
    kern<<<(unsigned)pl.ctas, S * 32, pl.smem, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// Every built (T, S) variant.
#define WS_VARIANTS(X) X(9, 4) X(11, 4) X(13, 4) X(15, 4) X(9, 2) X(13, 2)

template <typename IO>
ss_status launch_io(const S6Args &a, const WSPlan &pl, void *ws, cudaStream_t st,
                    unsigned long long timeout_ns) {
#define WS_LAUNCH(T_, S_) \
    if (pl.T == T_ && pl.S == S_) return launch_shape<IO, T_, S_>(a, pl, ws, st, timeout_ns);
    WS_VARIANTS(WS_LAUNCH)
#undef WS_LAUNCH
    return SS_ERR_UNSUPPORTED;
}

}  // namespace

bool ws_make_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int T, int S,
                  WSPlan *out) {
    WSPlan pl{};
    pl.T = T;
    pl.S = S;
    bool built = false;
    const int es = io_bf16 ? 2 : 4;
#define WS_SIZES(T_, S_)                                                                  \
    if (T == T_ && S == S_) {                                                              \
        using C = WSShape<T_, S_>;                                                         \
        pl.R = C::R;                                                                       \
        pl.smem = (size_t)ws_smem(C::R, S_, es, 2 * kPairs * C::P2 * 16).total + 128;        \
        built = true;                                                                      \
    }
    WS_VARIANTS(WS_SIZES)
#undef WS_SIZES
    if (!built || N > 16) return false;
    pl.dgroups = (int)((D + kCH - 1) / kCH);
    pl.nblk = (int)((L + pl.R - 1) / pl.R);
    pl.ctas = B * pl.dgroups;
    if (pl.smem > 227 * 1024 || pl.ctas > 0x7fffffffLL || L + pl.R >= (1LL << 31) ||
        B >= (1LL << 31) || D >= (1LL << 31) || (long long)kPairs * pl.nblk + S >= (1LL << 31))
        return false;
    *out = pl;
    return true;
}

bool ws_choose_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int sms,
                    WSPlan *out) {
    // Every CTA walks all of L, so the shape needs channels for two CTAs
    // per SM (32 channels each) or more; 13 steps per slice and 4 slices
    // measured fastest on the bf16 forward workload (11: 4% slower, 15:
    // equal, 9 and 17: 5-10% slower).
    WSPlan pl{};
    if (N > 16 || !ws_make_plan(B, L, D, N, io_bf16, 13, 4, &pl)) return false;
    if (pl.ctas < 2LL * sms) return false;
    *out = pl;
    return true;
}

ss_status ws_launch(const S6Args &a, const WSPlan &pl, void *workspace, cudaStream_t stream,
                    unsigned long long timeout_ns) {
    return a.io_bf16 ? launch_io<__nv_bfloat16>(a, pl, workspace, stream, timeout_ns)
                     : launch_io<float>(a, pl, workspace, stream, timeout_ns);
}

}  // namespace ss
