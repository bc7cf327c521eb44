// Single-pass S6 selective-scan forward in a time-parallel layout (sm_103a).
//
// "POPCORNBENCH FW-GLM-5-1 l2_p30" (arjun-banerjee.github.io), forward-pass
// derivation: dA = exp(delta*A), dBx = delta*B_t*x, h = dA*h + dBx,
// y_t = sum_n h*C_t + D*x. Each (b, t, d, n) term's exp is computed once, and
// the inputs are read once:
//
//  * a warp owns G channels; lane (c, s) holds T consecutive timesteps of
//    channel c (slice s of S = 32 / G slices), so a warp block covers
//    R = S*T steps of its G channels. The warp walks its channels over all
//    of L block by block, so the state entering a block is the previous
//    block's last state (kept in shared memory), and no carry ever crosses
//    CTAs;
//  * states are taken two at a time (a pair n, n+1 in one f32x2 register):
//    for each pair the lane computes dA and dBx for its T steps (one ex2 each
//    on MUFU), folds them into its slice's map h -> P*h + H, an ordered
//    shuffle scan over the S slices (left operand earlier) turns the maps
//    into each slice's starting state, and a second pass over the T steps in
//    registers writes the states into y = sum_n h*C. exp runs once per term;
//    the product over a slice is 2^(A*log2e * sum(delta)), one MUFU op more
//    per pair and slice;
//  * x and delta tiles (R rows x the CTA's channels) arrive by 3D TMA tile
//    copies into a 2-stage ring; y leaves by a 3D TMA tile store, clipped at
//    L; B_t and C_t are first packed by a small kernel into fp32 slots laid
//    out for the lanes (two steps of a state pair per 16-byte load, slices
//    spread over the shared-memory banks) and stream in by bulk copies, four
//    state pairs per slot.
//
// Results are bitwise reproducible: every sum and scan has a fixed order.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>

#include "f32x2.cuh"
#include "s6_common.cuh"
#include "ss_common.cuh"
#include "ss_internal.h"
#include "s6_tp.h"

namespace ss {
namespace {

constexpr int kNSX = 2;           // x / delta tile stages
constexpr int kNSB = 2;           // B_t / C_t slots
constexpr int kPairsPerSlot = 4;  // state pairs per slot
constexpr unsigned kFull = 0xffffffffu;

template <int G, int T> struct TPShape {
    static_assert(G == 2 || G == 4 || G == 8, "channels per warp");
    static_assert(T % 2 == 1, "odd steps per lane keep slices on distinct banks");
    static constexpr int S = 32 / G;                         // slices per channel
    static constexpr int LOG2S = G == 2 ? 4 : (G == 4 ? 3 : 2);
    static constexpr int R = S * T;                          // steps per block
    static constexpr int P2 = (T + 1) / 2;                   // step pairs per slice
    // bytes per slice in a packed row; an odd count of 16-byte units puts the
    // slices of one quarter-warp on distinct banks
    static constexpr int SLS = (P2 & 1) ? P2 * 16 : P2 * 16 + 16;
    static constexpr int SLOT = 2 * kPairsPerSlot * S * SLS;  // B and C of kPairsPerSlot pairs
};

struct TPParams {
    CUtensorMap tm_x, tm_d, tm_y;  // 3D (D, L, B) maps, box (rowW, R, 1)
    const float4 *bc;              // packed B_t / C_t slots
    const float *A, *Dskip, *delta_bias, *h0;
    float *h_last;
    WsHeader *ws;
    long long L, D;
    int N, nsl, nblk, rowW, dgroups, softplus;
    unsigned long long timeout_ns;
};

// Shared-memory carve-up of one CTA (host and device agree on it).
struct TPSmem {
    int tile, off_d, off_bc, off_y, off_a2, off_cs, off_dsk, off_db, off_bar, total;
};
__host__ __device__ inline TPSmem tp_smem(int R, int rowW, int es, int slot) {
    TPSmem m;
    m.tile = (R * rowW * es + 127) / 128 * 128;
    m.off_d = kNSX * m.tile;
    m.off_bc = 2 * kNSX * m.tile;
    m.off_y = m.off_bc + kNSB * slot;
    m.off_a2 = m.off_y + 2 * m.tile;
    m.off_cs = m.off_a2 + rowW * 16 * 4;
    m.off_dsk = m.off_cs + rowW * 16 * 4;
    m.off_db = m.off_dsk + rowW * 4;
    m.off_bar = (m.off_db + rowW * 4 + 7) / 8 * 8;
    m.total = m.off_bar + (kNSX + kNSB) * 8;
    return m;
}

__device__ __forceinline__ u64 shfl_up64(u64 v, int delta) {
    const float lo = __shfl_up_sync(kFull, f2lo(v), delta);
    const float hi = __shfl_up_sync(kFull, f2hi(v), delta);
    return f2(lo, hi);
}

// ------------------------------------------------------------------ B_t / C_t packing
// out[((b*nblk + j)*nsl + q)*SLOT/16 + ((m*P + kk)*S + s)*SLS/16 + ip] =
//   {M[t][n], M[t][n+1], M[t+1][n], M[t+1][n+1]},  M = B_t (m = 0) or C_t,
//   P = kPairsPerSlot, t = j*R + s*T + 2*ip, n = 2*(P*q + kk); zero past L,
//   past the slice's T
//   steps and past N. One thread per (b, j, s, ip): it reads the four rows
//   t, t+1 of B_t and C_t and writes every state pair of them.
template <typename IO, int G, int T>
__global__ void __launch_bounds__(256) tp_pack_kernel(const IO *Bt, const IO *Ct, float4 *out,
                                                      long long L, int N, long long ldbc, int nblk,
                                                      int nsl, long long total) {
    griddep_launch_dependents();
    using C = TPShape<G, T>;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int ip = (int)(idx % C::P2);
    const int s = (int)((idx / C::P2) % C::S);
    const long long bj = idx / (C::P2 * C::S);  // b * nblk + j
    const long long j = bj % nblk, b = bj / nblk;
    float4 *dst = out + bj * nsl * (C::SLOT / 16) + s * (C::SLS / 16) + ip;
    const int npairs = nsl * kPairsPerSlot;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const IO *M = m ? Ct : Bt;
        float v[2][16];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = 2 * ip + e;
            const long long t = j * C::R + (long long)s * T + i;
            const bool ok = i < T && t < L;
            const IO *row = M + (b * L + t) * ldbc;
#pragma unroll
            for (int n = 0; n < 16; ++n) v[e][n] = (ok && n < N) ? to_f32(row[n]) : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < npairs) {
                const int q = k / kPairsPerSlot, kk = k % kPairsPerSlot;
                dst[q * (C::SLOT / 16) + (m * kPairsPerSlot + kk) * C::S * (C::SLS / 16)] =
                    make_float4(v[0][2 * k], v[0][2 * k + 1], v[1][2 * k], v[1][2 * k + 1]);
            }
        }
    }
}

// ------------------------------------------------------------------ scan steps
// One level of the ordered scan over slices, on the two states' scalars: a
// lane with `on` set combines its map (P, H) with the received map of the
// lane `off` slices earlier (left operand earlier): H = P*h + H, P = P*p.
// Predicated, so lanes without a left neighbour take no branch.
__device__ __forceinline__ void scan_level(float &Hl, float &Hh, float &Pl, float &Ph, float hl,
                                           float hh, float pl, float ph, unsigned on) {
    asm("{\n .reg .pred q;\n setp.ne.u32 q, %8, 0;\n"
        " @q fma.rn.f32 %0, %2, %4, %0;\n"
        " @q fma.rn.f32 %1, %3, %5, %1;\n"
        " @q mul.rn.f32 %2, %2, %6;\n"
        " @q mul.rn.f32 %3, %3, %7;\n}"
        : "+f"(Hl), "+f"(Hh), "+f"(Pl), "+f"(Ph)
        : "f"(hl), "f"(hh), "f"(pl), "f"(ph), "r"(on));
}
// The last level: H only (P is not needed after it).
__device__ __forceinline__ void scan_last(float &Hl, float &Hh, float Pl, float Ph, float hl,
                                          float hh, unsigned on) {
    asm("{\n .reg .pred q;\n setp.ne.u32 q, %6, 0;\n"
        " @q fma.rn.f32 %0, %2, %4, %0;\n"
        " @q fma.rn.f32 %1, %3, %5, %1;\n}"
        : "+f"(Hl), "+f"(Hh) : "f"(Pl), "f"(Ph), "f"(hl), "f"(hh), "r"(on));
}
// H = P*c + H on lanes with `on` set (the state entering the block folded into
// the first slice's map).
__device__ __forceinline__ u64 fold_if(u64 H, u64 P, u64 c, unsigned on) {
    asm("{\n .reg .pred q;\n setp.ne.u32 q, %3, 0;\n"
        " @q fma.rn.f32x2 %0, %1, %2, %0;\n}"
        : "+l"(H) : "l"(P), "l"(c), "r"(on));
    return H;
}
// (on ? c : {lo, hi})
__device__ __forceinline__ u64 select_pair(unsigned on, u64 c, float lo, float hi) {
    u64 r;
    asm("{\n .reg .pred q;\n .reg .f32 cl, ch, a, b;\n setp.ne.u32 q, %1, 0;\n"
        " mov.b64 {cl, ch}, %2;\n selp.f32 a, cl, %3, q;\n selp.f32 b, ch, %4, q;\n"
        " mov.b64 %0, {a, b};\n}"
        : "=l"(r) : "r"(on), "l"(c), "f"(lo), "f"(hi));
    return r;
}
// Stores (lo, hi) to the shared-memory pair at p on lanes with `on` set.
__device__ __forceinline__ void store_pair_if(float *p, float lo, float hi, unsigned on) {
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %3, 0;\n"
                 " @q st.shared.v2.f32 [%0], {%1, %2};\n}"
                 ::"r"(smem_addr(p)), "f"(lo), "f"(hi), "r"(on) : "memory");
}

// ------------------------------------------------------------------ per state pair
// Pass 1a for one state pair: dA = 2^(A2 * delta) of the lane's T steps (MUFU).
template <int T>
__device__ __forceinline__ void tp_pass1a(u64 A2, const u64 (&ddl)[T], u64 (&dA)[T]) {
#pragma unroll
    for (int i = 0; i < T; ++i) dA[i] = f2_exp2_scaled(ddl[i], A2);
}
// Pass 1b: dBx of the T steps (B_t pairs of two steps per 16-byte load from
// the slot row bp) and the slice's map (P, H): H = the state after the T
// steps from zero, P = 2^(A2 * sum of delta).
template <int T>
__device__ __forceinline__ void tp_pass1b(const unsigned char *bp, u64 A2, const u64 (&uu)[T],
                                          u64 sdl2, const u64 (&dA)[T], u64 (&bx)[T], u64 &H,
                                          u64 &P) {
    constexpr int P2 = (T + 1) / 2;
    H = 0ull;
#pragma unroll
    for (int ip = 0; ip < P2; ++ip) {
        const ulonglong2 b4 = *reinterpret_cast<const ulonglong2 *>(bp + ip * 16);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = 2 * ip + e;
            if (i < T) {
                bx[i] = f2mul(uu[i], e ? b4.y : b4.x);
                H = f2fma(dA[i], H, bx[i]);
            }
        }
    }
    P = f2_exp2_scaled(sdl2, A2);
}

// The ordered scan over the slices for one state pair: folds the block's
// entering state `cin` into slice 0's map, scans, and returns the state
// entering this lane's slice; the last slice stores the block's final state
// to `cout` (the next block's `cin`).
template <int G, int LOG2S>
__device__ __forceinline__ u64 tp_scan(u64 H, u64 P, u64 cin, const unsigned (&on_lv)[LOG2S],
                                       unsigned first, unsigned last, float *cout) {
    H = fold_if(H, P, cin, first);
    float Hl = f2lo(H), Hh = f2hi(H), Pl = f2lo(P), Ph = f2hi(P);
#pragma unroll
    for (int lv = 0; lv < LOG2S; ++lv) {
        const int off = (1 << lv) * G;
        const float hl = __shfl_up_sync(kFull, Hl, off);
        const float hh = __shfl_up_sync(kFull, Hh, off);
        if (lv + 1 < LOG2S) {
            const float pl = __shfl_up_sync(kFull, Pl, off);
            const float ph = __shfl_up_sync(kFull, Ph, off);
            scan_level(Hl, Hh, Pl, Ph, hl, hh, pl, ph, on_lv[lv]);
        } else {
            scan_last(Hl, Hh, Pl, Ph, hl, hh, on_lv[lv]);
        }
    }
    const float sl = __shfl_up_sync(kFull, Hl, G);
    const float sh = __shfl_up_sync(kFull, Hh, G);
    store_pair_if(cout, Hl, Hh, last);
    return select_pair(first, cin, sl, sh);
}

// Pass 2 for one state pair: the states of the T steps from h, into y.
template <int T>
__device__ __forceinline__ void tp_pass2(const unsigned char *cp, const u64 (&dA)[T],
                                         const u64 (&bx)[T], u64 h, u64 (&yp)[T]) {
    constexpr int P2 = (T + 1) / 2;
#pragma unroll
    for (int ip = 0; ip < P2; ++ip) {
        const ulonglong2 c4 = *reinterpret_cast<const ulonglong2 *>(cp + ip * 16);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = 2 * ip + e;
            if (i < T) {
                h = f2fma(dA[i], h, bx[i]);
                yp[i] = f2fma(e ? c4.y : c4.x, h, yp[i]);
            }
        }
    }
}

// ------------------------------------------------------------------ main kernel
// Resident warps per SM the launch bounds ask registers for: 16 for two and
// four channels per warp (128 registers a thread), 12 for eight (170): shapes
// with eight channels per warp have the channels for fewer warps per SM.
template <int G, int W> constexpr int kTPMinBlocks = (G == 8 ? 12 : 16) / W;

template <typename IO, int G, int T, int W>
__global__ void __launch_bounds__(W * 32, (kTPMinBlocks<G, W>)) s6_tp_kernel(const __grid_constant__ TPParams p) {
    using C = TPShape<G, T>;
    constexpr int S = C::S, R = C::R, P2 = C::P2, SLS = C::SLS, SLOT = C::SLOT;
    constexpr int LOG2S = C::LOG2S;
    constexpr int RW = G * W;  // channels per CTA (a tile row)
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);

    const TPSmem L_ = tp_smem(R, RW, (int)sizeof(IO), SLOT);
    float *a2s = reinterpret_cast<float *>(sm + L_.off_a2);
    float *cs = reinterpret_cast<float *>(sm + L_.off_cs);
    float *dsk = reinterpret_cast<float *>(sm + L_.off_dsk);
    float *dbs = reinterpret_cast<float *>(sm + L_.off_db);
    uint64_t *xbar = reinterpret_cast<uint64_t *>(sm + L_.off_bar);
    uint64_t *bcbar = xbar + kNSX;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = lane & (G - 1), s = lane / G;
    const int ch = warp * G + c;  // channel within the CTA
    const long long b = blockIdx.x / p.dgroups;
    const long long d0 = (long long)(blockIdx.x % p.dgroups) * RW;
    const int N = p.N;
    const long long D = p.D, L = p.L;

    for (int i = tid; i < RW * 16; i += W * 32) {
        const long long dd = d0 + (i >> 4);
        const int n = i & 15;
        const bool ok = dd < D && n < N;
        a2s[i] = ok ? p.A[dd * N + n] * kLog2e : 0.0f;
        cs[i] = (ok && p.h0) ? p.h0[(b * D + dd) * N + n] : 0.0f;
    }
    for (int i = tid; i < RW; i += W * 32) {
        const long long dd = d0 + i;
        dsk[i] = (dd < D && p.Dskip) ? p.Dskip[dd] : 0.0f;
        dbs[i] = (dd < D && p.delta_bias) ? p.delta_bias[dd] : 0.0f;
    }
    if (tid == 0) {
        for (int k = 0; k < kNSX + kNSB; ++k) mbar_init(xbar + k, 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int nblk = p.nblk, nsl = p.nsl;
    const long long total_slots = (long long)nblk * nsl;
    const float4 *bcg = p.bc + (long long)b * total_slots * (SLOT / 16);
    constexpr unsigned kXBytes = 2u * (unsigned)(R * RW * (int)sizeof(IO));

    auto issue_x = [&](int j) {
        const int st = j % kNSX;
        mbar_arrive_expect_tx(xbar + st, kXBytes);
        tma_load_3d(sm + st * L_.tile, &p.tm_x, (int)d0, j * R, (int)b, xbar + st);
        tma_load_3d(sm + L_.off_d + st * L_.tile, &p.tm_d, (int)d0, j * R, (int)b, xbar + st);
    };
    auto issue_bc = [&](long long gq) {
        const int sl = (int)(gq % kNSB);
        mbar_arrive_expect_tx(bcbar + sl, (unsigned)SLOT);
        bulk_g2s(sm + L_.off_bc + sl * SLOT, bcg + gq * (SLOT / 16), (unsigned)SLOT, bcbar + sl);
    };
    int x_issued = 0;
    long long bc_issued = 0;
    if (tid == 0) {
        for (; x_issued < kNSX && x_issued < nblk; ++x_issued) issue_x(x_issued);
        griddep_wait();  // the packed B_t / C_t come from the kernel before this one
        for (; bc_issued < kNSB && bc_issued < total_slots; ++bc_issued) issue_bc(bc_issued);
    }

    const float Dd = dsk[ch];
    const float dbias = dbs[ch];
    const bool sp = p.softplus != 0;
    float *csc = cs + ch * 16;           // this channel's carries
    const float *a2c = a2s + ch * 16;    // this channel's A * log2(e)
    const int lane_off = s * T * RW + ch;  // this lane's first element in a tile
    unsigned on_lv[LOG2S];                 // scan level lv: a left neighbour exists
#pragma unroll
    for (int lv = 0; lv < LOG2S; ++lv) on_lv[lv] = s >= (1 << lv);
    const unsigned first = s == 0, last = s == S - 1;
    bool bad = false;      // a wait of this thread ran out
    bool aborted = false;  // some thread's did (uniform across the CTA)
    int j = 0;
    for (; j < nblk; ++j) {
        // ---- x and delta of this lane's T steps
        const int xst = j % kNSX;
        if (!mbar_wait_bounded(xbar + xst, (unsigned)(j / kNSX) & 1u, p.timeout_ns)) {
            record_error(p.ws, SS_ERR_TIMEOUT, 8u, blockIdx.x, (unsigned)j);
            bad = true;
        }
        const IO *xt = reinterpret_cast<const IO *>(sm + xst * L_.tile) + lane_off;
        const IO *dt = reinterpret_cast<const IO *>(sm + L_.off_d + xst * L_.tile) + lane_off;
        u64 ddl[T], uu[T], yp[T];
        float sdl = 0.0f;
        const long long lim = L - (long long)j * R - (long long)s * T;  // steps of this slice in L
#pragma unroll
        for (int i = 0; i < T; ++i) {
            float dv = to_f32(dt[i * RW]) + dbias;
            if (sp) dv = softplus_mufu(dv);
            if (i >= lim) dv = 0.0f;  // past L: dA = 1, no input
            const float xv = to_f32(xt[i * RW]);
            const float u = dv * xv;
            ddl[i] = f2(dv, dv);
            uu[i] = f2(u, u);
            yp[i] = f2(Dd * xv, 0.0f);
            sdl += dv;
        }
        const u64 sdl2 = f2(sdl, sdl);

        // ---- the state pairs, software-pipelined: pass 1 of pair k + 1 is
        // issued ahead of the scan and pass 2 of pair k, so the two chains
        // overlap. Pair k lives in slot k / kPairsPerSlot of this block.
        const int np = nsl * kPairsPerSlot;
        auto wait_slot = [&](int q) {
            const long long gq = (long long)j * nsl + q;
            if (!mbar_wait_bounded(bcbar + (int)(gq % kNSB), (unsigned)(gq / kNSB) & 1u,
                                   p.timeout_ns)) {
                record_error(p.ws, SS_ERR_TIMEOUT, 9u, blockIdx.x, (unsigned)gq);
                bad = true;
            }
        };
        auto slot_row = [&](int k) {  // this lane's slice row of pair k's slot
            const long long gq = (long long)j * nsl + k / kPairsPerSlot;
            return sm + L_.off_bc + (int)(gq % kNSB) * SLOT + s * SLS;
        };
        wait_slot(0);
        u64 dA0[T];
        tp_pass1a<T>(*reinterpret_cast<const u64 *>(a2c), ddl, dA0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k >= np) break;
            const int kk = k % kPairsPerSlot;
            const u64 A2 = *reinterpret_cast<const u64 *>(a2c + 2 * k);
            u64 bx[T], H, P;
            tp_pass1b<T>(slot_row(k) + kk * S * SLS, A2, uu, sdl2, dA0, bx, H, P);
            // the next pair's exps are issued ahead of this pair's scan
            u64 dA1[T];
            if (k + 1 < np)
                tp_pass1a<T>(*reinterpret_cast<const u64 *>(a2c + 2 * (k + 1)), ddl, dA1);
            const u64 cin = *reinterpret_cast<const u64 *>(csc + 2 * k);
            const u64 h = tp_scan<G, LOG2S>(H, P, cin, on_lv, first, last, csc + 2 * k);
            tp_pass2<T>(slot_row(k) + (kPairsPerSlot + kk) * S * SLS, dA0, bx, h, yp);
            if (kk == kPairsPerSlot - 1 || k + 1 == np) {
                // slot (and, for the first, the x / delta stage) consumed
                aborted = __syncthreads_or(bad) != 0;
                if (aborted) break;
                if (tid == 0) {
                    if (bc_issued < total_slots) issue_bc(bc_issued++);
                    if (k < kPairsPerSlot && x_issued < nblk) issue_x(x_issued++);
                }
                if (k + 1 < np) wait_slot((k + 1) / kPairsPerSlot);
            }
#pragma unroll
            for (int i = 0; i < T; ++i) dA0[i] = dA1[i];
        }
        if (aborted) break;

        // ---- y: the block's tile, then one TMA store (clipped at L and D)
        IO *yt = reinterpret_cast<IO *>(sm + L_.off_y + (j & 1) * L_.tile);
#pragma unroll
        for (int i = 0; i < T; ++i) store_smem(yt + lane_off + i * RW, f2lo(yp[i]) + f2hi(yp[i]));
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&p.tm_y, yt, (int)d0, j * R, (int)b);
            bulk_commit();
            bulk_wait_read<1>();  // the other y buffer is free again
        }
    }

    if (tid == 0) {
        bulk_wait<0>();
        // after an abort, copies still in flight land before the CTA exits
        // (a wait on a phase that already completed returns at once)
        for (int jj = j; jj < x_issued; ++jj)
            mbar_wait_bounded(xbar + jj % kNSX, (unsigned)(jj / kNSX) & 1u, p.timeout_ns);
        for (long long g = (long long)j * nsl; g < bc_issued; ++g)
            mbar_wait_bounded(bcbar + g % kNSB, (unsigned)(g / kNSB) & 1u, p.timeout_ns);
    }
    __syncthreads();
    if (p.h_last && !aborted) {
        for (int i = tid; i < RW * 16; i += W * 32) {
            const long long dd = d0 + (i >> 4);
            const int n = i & 15;
            if (dd < D && n < N) p.h_last[(b * D + dd) * N + n] = cs[i];
        }
    }
}

template <typename IO, int G, int T, int W>
ss_status launch_shape(const S6Args &a, const TPPlan &pl, void *workspace, size_t pack_offset,
                       cudaStream_t stream, unsigned long long timeout_ns) {
    using C = TPShape<G, T>;
    const bool bf = sizeof(IO) == 2;
    const uint64_t es = bf ? 2 : 4;
    TPParams prm{};
    const long long ldd = a.ld_delta > 0 ? a.ld_delta : a.D;
    const long long ldbc = a.ld_bc > 0 ? a.ld_bc : a.N;
    const uint64_t dx[3] = {(uint64_t)a.D, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t sx[2] = {(uint64_t)a.D * es, (uint64_t)(a.L * a.D) * es};
    const uint64_t sd[2] = {(uint64_t)ldd * es, (uint64_t)(a.L * ldd) * es};
    const uint32_t box[3] = {(uint32_t)pl.rowW, (uint32_t)C::R, 1u};
    if (!encode_tiled_map(&prm.tm_x, a.x, bf, 3, dx, sx, box) ||
        !encode_tiled_map(&prm.tm_d, a.delta, bf, 3, dx, sd, box) ||
        !encode_tiled_map(&prm.tm_y, a.y, bf, 3, dx, sx, box))
        return SS_ERR_CUDA;
    char *ws = static_cast<char *>(workspace);
    prm.ws = reinterpret_cast<WsHeader *>(ws);
    prm.bc = reinterpret_cast<const float4 *>(ws + pack_offset);
    prm.A = a.A;
    prm.Dskip = a.Dskip;
    prm.delta_bias = a.delta_bias;
    prm.h0 = a.h0;
    prm.h_last = a.h_last;
    prm.L = a.L;
    prm.D = a.D;
    prm.N = (int)a.N;
    prm.nsl = pl.nsl;
    prm.nblk = pl.nblk;
    prm.rowW = G * W;
    prm.dgroups = pl.dgroups;
    prm.softplus = a.softplus;
    prm.timeout_ns = timeout_ns;

    // 1) pack B_t, C_t
    const long long total = (long long)a.B * pl.nblk * C::S * C::P2;
    const long long pack_blocks = (total + 255) / 256;
    if (pack_blocks > 0x7fffffffLL) return SS_ERR_UNSUPPORTED;
    tp_pack_kernel<IO, G, T><<<(unsigned)pack_blocks, 256, 0, stream>>>(
        static_cast<const IO *>(a.Bt), static_cast<const IO *>(a.Ct),
        reinterpret_cast<float4 *>(ws + pack_offset), a.L, (int)a.N, ldbc, pl.nblk, pl.nsl, total);
    if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;

    // 2) the scan, launched as a programmatic dependent of the packing kernel
    auto kern = s6_tp_kernel<IO, G, T, W>;
    if (raise_smem_limit(reinterpret_cast<const void *>(kern), (int)pl.smem) != SS_OK)
        return SS_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)pl.ctas);
    cfg.blockDim = dim3((unsigned)(pl.W * 32));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) return SS_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// Every built (G, T, W) variant: X(G, T, W) for each.
#define TP_VARIANTS(X)                                                                     \
    X(2, 9, 2) X(2, 9, 4) X(4, 9, 2) X(4, 9, 4) X(8, 9, 1) X(8, 9, 2) X(8, 9, 4) X(2, 7, 4)  \
    X(2, 7, 2) X(4, 7, 4) X(4, 7, 2) X(8, 7, 2) X(8, 7, 4)

template <typename IO>
ss_status launch_io(const S6Args &a, const TPPlan &pl, void *ws, size_t off, cudaStream_t s,
                    unsigned long long timeout_ns) {
#define TP_LAUNCH(G_, T_, W_)                                                      \
    if (pl.G == G_ && pl.T == T_ && pl.W == W_)                                   \
        return launch_shape<IO, G_, T_, W_>(a, pl, ws, off, s, timeout_ns);
    TP_VARIANTS(TP_LAUNCH)
#undef TP_LAUNCH
    return SS_ERR_UNSUPPORTED;
}

template <int G, int T>
void shape_sizes(TPPlan &pl, int es) {
    using C = TPShape<G, T>;
    pl.S = C::S;
    pl.R = C::R;
    pl.slot_bytes = C::SLOT;
    pl.smem = (size_t)tp_smem(C::R, pl.rowW, es, C::SLOT).total + 128;
}

}  // namespace

bool tp_make_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int G, int T, int W,
                  TPPlan *out) {
    TPPlan pl{};
    pl.G = G;
    pl.T = T;
    pl.W = W;
    pl.rowW = G * W;
    const int es = io_bf16 ? 2 : 4;
    if ((pl.rowW * es) % 16 != 0) return false;
    bool built = false;
#define TP_SIZES(G_, T_, W_)                          \
    if (G == G_ && T == T_ && W == W_) {              \
        shape_sizes<G_, T_>(pl, es);                  \
        built = true;                                 \
    }
    TP_VARIANTS(TP_SIZES)
#undef TP_SIZES
    if (!built) return false;
    pl.dgroups = (int)((D + pl.rowW - 1) / pl.rowW);
    pl.nblk = (int)((L + pl.R - 1) / pl.R);
    pl.nsl = (int)(((N + 1) / 2 + kPairsPerSlot - 1) / kPairsPerSlot);
    pl.ctas = B * pl.dgroups;
    pl.pack_bytes = (size_t)B * pl.nblk * pl.nsl * pl.slot_bytes;
    if (pl.smem > 227 * 1024 || pl.ctas > 0x7fffffffLL || L + pl.R >= (1LL << 31) ||
        B >= (1LL << 31) || D >= (1LL << 31))
        return false;
    *out = pl;
    return true;
}

int tp_ctas_per_sm(const TPPlan &pl, int io_bf16) {
    const void *fn = nullptr;
#define TP_FN(G_, T_, W_)                                                                    \
    if (pl.G == G_ && pl.T == T_ && pl.W == W_)                                              \
        fn = io_bf16 ? reinterpret_cast<const void *>(s6_tp_kernel<__nv_bfloat16, G_, T_, W_>) \
                     : reinterpret_cast<const void *>(s6_tp_kernel<float, G_, T_, W_>);
    TP_VARIANTS(TP_FN)
#undef TP_FN
    int n = 0;
    if (!fn ||
        raise_smem_limit(reinterpret_cast<const void *>(fn), (int)pl.smem) != SS_OK ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, pl.W * 32, pl.smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

bool tp_choose_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int sms,
                    TPPlan *out) {
    // Each CTA walks all of L, so a CTA's lifetime is the kernel's: the
    // busiest SM sets the time. For every built variant, estimate the
    // busiest SM's instructions (CTAs on it x channels per CTA x
    // instructions per (t, d) of the variant: per state pair and lane, about
    // 9 per step plus 6 per scan level and 8 more, over T steps), divided by
    // an issue efficiency that falls off below 12 resident warps per SM.
    // Channels per CTA stay >= 32 bytes of a row, as every CTA reloads the
    // packed B_t / C_t.
    const int es = io_bf16 ? 2 : 4;
    const int Gs[3] = {2, 4, 8}, Ts[2] = {9, 7}, Ws[3] = {1, 2, 4};
    double best = -1.0;
    TPPlan bp{};
    for (int G : Gs)
        for (int T : Ts)
            for (int W : Ws) {
                TPPlan pl{};
                if (G * W * es < 32 || !tp_make_plan(B, L, D, N, io_bf16, G, T, W, &pl)) continue;
                int per_sm = tp_ctas_per_sm(pl, io_bf16);
                if (per_sm <= 0) {  // no device to ask: 128 registers, shared memory
                    per_sm = std::min<long long>(65536 / (W * 32 * 128),
                                                 (228LL * 1024) / ((long long)pl.smem + 1024));
                }
                if (per_sm <= 0) continue;
                const long long load = (pl.ctas + sms - 1) / sms;  // CTAs on the busiest SM
                const long long rounds = (load + per_sm - 1) / per_sm;
                const long long conc = std::min<long long>(load, per_sm);
                const int log2s = G == 2 ? 4 : (G == 4 ? 3 : 2);
                const double ipt = 8.0 * (9.0 * T + 6.0 * log2s + 8.0) / T;
                const double eff = std::min(1.0, conc * W / 12.0);
                const double cost = rounds * conc * (double)pl.rowW * ipt / eff;
                // too few warps, idle SMs or a lopsided last round: the
                // chunked kernel, which splits L, does better
                if (conc * W < 8 || pl.ctas < sms || (double)pl.ctas / sms / load < 0.6) continue;
                if (best < 0 || cost < best * 0.999 ||
                    (cost <= best * 1.001 && pl.rowW > bp.rowW)) {
                    best = cost;
                    bp = pl;
                }
            }
    if (best < 0) return false;
    *out = bp;
    return true;
}

ss_status tp_launch(const S6Args &a, const TPPlan &pl, void *workspace, size_t pack_offset,
                    cudaStream_t stream, unsigned long long timeout_ns) {
    return a.io_bf16 ? launch_io<__nv_bfloat16>(a, pl, workspace, pack_offset, stream, timeout_ns)
                     : launch_io<float>(a, pl, workspace, pack_offset, stream, timeout_ns);
}

}  // namespace ss
