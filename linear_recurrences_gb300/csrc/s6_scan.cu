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
//  * lane = one channel d with NG of its N states in registers; a warp is
//    32 consecutive channels, so x, delta and y accesses are coalesced;
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
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxWT = 8;       // warps per CTA along time
constexpr int kMaxWindows = 4;  // look-back holds up to 128 predecessor chunks
constexpr unsigned kFull = 0xffffffffu;

// Descriptor payload fields, each [32 lanes][NG] floats per (sequence, chunk).
enum { F_P = 0, F_H = 1, F_INC = 2, F_HR = 3, F_RINC = 4 };
// Descriptor flags per (sequence, chunk).
enum { FL_AGG = 0, FL_INC = 1, FL_RINC = 2, FL_PAD = 3 };

struct S6Params {
    const void *x, *delta, *Bt, *Ct;
    const float *A, *Dskip;
    void *y;
    float *yscratch;   // bidirectional bf16: fp32 forward outputs (B, L, D)
    long long L, D;
    int N;
    int dtiles;        // ceil(D / 32)
    int K;             // chunks per sequence
    int WT;            // warps per CTA
    int Tsub;          // timesteps per warp
    int vecBC;         // Bt, Ct rows readable with 16-byte vector loads
    WsHeader *ws;
    unsigned *flags;   // [(seq*K + k)*4 + FL_*]
    float *payload;    // [((seq*K + k)*NF + field)*32*NG + lane*NG + i]
    unsigned long long timeout_ns;
    long long skip_unit;  // test hook: this unit publishes nothing (-1: none)
};

// ------------------------------------------------------------------ io helpers
template <typename IO> struct Io;
template <> struct Io<float> {
    static __device__ __forceinline__ float ld(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ void st(float *p, float v) { __stcs(p, v); }
};
template <> struct Io<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) {
        return __bfloat162float(__ldg(p));
    }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

__device__ __forceinline__ float bf16lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }

// NG consecutive values of a (B, L, N) row starting at p (element g*NG).
template <int NG, typename IO>
__device__ __forceinline__ void load_states(const IO *p, int nvalid, bool vec, float (&v)[NG]) {
    if (vec) {
        if constexpr (sizeof(IO) == 4) {
#pragma unroll
            for (int q = 0; q < NG / 4; ++q) {
                const float4 f = __ldg(reinterpret_cast<const float4 *>(p) + q);
                v[4 * q + 0] = f.x;
                v[4 * q + 1] = f.y;
                v[4 * q + 2] = f.z;
                v[4 * q + 3] = f.w;
            }
        } else if constexpr (NG % 8 == 0) {
#pragma unroll
            for (int q = 0; q < NG / 8; ++q) {
                const uint4 w = __ldg(reinterpret_cast<const uint4 *>(p) + q);
                v[8 * q + 0] = bf16lo(w.x);
                v[8 * q + 1] = bf16hi(w.x);
                v[8 * q + 2] = bf16lo(w.y);
                v[8 * q + 3] = bf16hi(w.y);
                v[8 * q + 4] = bf16lo(w.z);
                v[8 * q + 5] = bf16hi(w.z);
                v[8 * q + 6] = bf16lo(w.w);
                v[8 * q + 7] = bf16hi(w.w);
            }
        } else {
            const uint2 w = __ldg(reinterpret_cast<const uint2 *>(p));
            v[0] = bf16lo(w.x);
            v[1] = bf16hi(w.x);
            v[2] = bf16lo(w.y);
            v[3] = bf16hi(w.y);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NG; ++i) v[i] = i < nvalid ? Io<IO>::ld(p + i) : 0.0f;
    }
}

// softplus(v) = log(1 + exp(v)); v > 20 returns v. exp and log on MUFU; for
// exp(v) < 1/64 the log is replaced by its alternating series so that the
// rounding of 1 + exp(v) does not swamp small results.
__device__ __forceinline__ float softplus_mufu(float v) {
    if (v > 20.0f) return v;
    const float e = ex2_approx(v * kLog2e);
    if (e < 0.015625f) return e * (1.0f - e * (0.5f - e * (1.0f / 3.0f - 0.25f * e)));
    return lg2_approx(1.0f + e) * kLn2;
}

template <int NG>
__device__ __forceinline__ float *field_ptr(const S6Params &p, int NF, long long unit, int field,
                                            int lane) {
    return p.payload + ((unit * NF + field) * 32 + lane) * NG;
}

template <int NG>
__device__ __forceinline__ void store_field(float *dst, const float (&v)[NG]) {
#pragma unroll
    for (int q = 0; q < NG / 4; ++q)
        __stcg(reinterpret_cast<float4 *>(dst) + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
}
template <int NG>
__device__ __forceinline__ void load_field(const float *src, float (&v)[NG]) {
#pragma unroll
    for (int q = 0; q < NG / 4; ++q) {
        const float4 f = ld_cg_f32x4(reinterpret_cast<const float4 *>(src) + q);
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
}

// Publishes flag `which` of `unit` after every lane of the warp has written
// its payload (each lane fences its own writes first).
__device__ __forceinline__ void publish_flag(const S6Params &p, long long unit, int which,
                                             unsigned tag, int lane) {
    __threadfence();
    __syncwarp();
    if (lane == 0 && unit != p.skip_unit) st_release_u32(p.flags + unit * 4 + which, tag);
}

// ------------------------------------------------------------------ sweeps
// One pass of this lane's chains over timesteps [t0, t1).
// MODE_AGG: from a zero state, accumulate the sub-chunk aggregate.
// MODE_OUT: from the state in h, write outputs.
enum { MODE_AGG = 0, MODE_OUT = 1 };

template <int NG, typename IO, bool SP, bool BIDIR, int MODE, bool REV>
__device__ __forceinline__ void sweep(const S6Params &p, long long b, long long d, bool dvalid,
                                      long long t0, long long t1, const float (&A2)[NG], float Dd,
                                      float (&h)[NG], float (&hr)[NG], float (&Q)[NG], float &sdel,
                                      float *yf, bool final_out) {
    const IO *xp = static_cast<const IO *>(p.x);
    const IO *dp = static_cast<const IO *>(p.delta);
    const IO *bp = static_cast<const IO *>(p.Bt);
    const IO *cp = static_cast<const IO *>(p.Ct);
    const long long L = p.L, D = p.D;
    const int N = p.N;
    const bool vec = p.vecBC != 0;
    const long long nsteps = t1 - t0;
#pragma unroll 2
    for (long long s = 0; s < nsteps; ++s) {
        const long long t = REV ? (t1 - 1 - s) : (t0 + s);
        const long long row = b * L + t;
        const long long xi = row * D + d;
        float xv = 0.0f, dv = 0.0f;
        if (dvalid) {
            xv = Io<IO>::ld(xp + xi);
            dv = Io<IO>::ld(dp + xi);
        }
        const float dl = SP ? softplus_mufu(dv) : dv;
        float Bv[NG];
        load_states<NG, IO>(bp + row * N, N, vec, Bv);
        const float u = dl * xv;
        if constexpr (MODE == MODE_AGG) {
#pragma unroll
            for (int i = 0; i < NG; ++i) {
                const float dA = ex2_approx(dl * A2[i]);
                const float dbx = u * Bv[i];
                h[i] = fmaf(dA, h[i], dbx);
                if constexpr (BIDIR) {
                    hr[i] = fmaf(Q[i], dbx, hr[i]);
                    Q[i] *= dA;
                }
            }
            sdel += dl;
        } else {
            float Cv[NG];
            load_states<NG, IO>(cp + row * N, N, vec, Cv);
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < NG; ++i) {
                const float dA = ex2_approx(dl * A2[i]);
                h[i] = fmaf(dA, h[i], u * Bv[i]);
                acc = fmaf(h[i], Cv[i], acc);
            }
            float yv = fmaf(Dd, xv, acc);
            if (dvalid) {
                if (yf == nullptr) {
                    Io<IO>::st(static_cast<IO *>(p.y) + xi, yv);
                } else if (!final_out) {
                    yf[xi] = yv;  // forward half of a bidirectional output
                } else {
                    yv += yf[xi];
                    Io<IO>::st(static_cast<IO *>(p.y) + xi, yv);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ look-back
// Warp-parallel walk over the nearest predecessor (FWD) or successor (!FWD)
// chunks of the same sequence. Lane l examines chunk k -/+ (1 + l + 32*win).
// Returns the chunk index of the nearest published inclusive state (-1 or K
// for the sequence boundary, whose state is zero), or -2 on timeout.
template <bool FWD>
__device__ int find_anchor(const S6Params &p, long long seq, int k, unsigned tag, int lane) {
    const uint64_t t0 = globaltimer_ns();
    int win = 0;
    for (;;) {
        const int m = FWD ? k - 1 - (lane + 32 * win) : k + 1 + (lane + 32 * win);
        bool is_inc;
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
                if (ld_acquire_u32(fl + FL_AGG) == tag) {
                    is_inc = false;
                    break;
                }
                if ((it & 63u) == 63u &&
                    (globaltimer_ns() - t0 > p.timeout_ns || ld_relaxed_u32(&p.ws->error) != 0u)) {
                    is_inc = false;
                    it = 0xffffffffu;  // timed out
                    break;
                }
            }
            // a lane that gave up is reported through the timer check below
        }
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

// ------------------------------------------------------------------ kernel
template <int NG, typename IO, bool SP, bool BIDIR>
__global__ void __launch_bounds__(kMaxWT * 32)
s6_kernel(const S6Params p) {
    constexpr int NSUB = BIDIR ? 3 : 2;  // sub-aggregate fields: P, H (, Hr)
    constexpr int NF = BIDIR ? 5 : 3;    // descriptor fields
    extern __shared__ __align__(16) float smem[];
    float *s_sub = smem;                               // [WT][NSUB][32][NG]
    float *s_car = smem + p.WT * NSUB * 32 * NG;       // [2][32][NG]

    const bool chunked = p.K > 1;
    unsigned ticket, tag = 0;
    if (chunked) {
        take_ticket(p.ws, ticket, tag);
    } else {
        ticket = blockIdx.x;
    }
    const long long seq = ticket / (unsigned)p.K;
    const int k = (int)(ticket % (unsigned)p.K);
    const long long b = seq / p.dtiles;
    const int dt = (int)(seq % p.dtiles);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long d = (long long)dt * 32 + lane;
    const bool dvalid = d < p.D;
    const long long tc0 = (long long)k * p.WT * p.Tsub;
    const long long t0 = min(tc0 + (long long)warp * p.Tsub, p.L);
    const long long t1 = min(t0 + (long long)p.Tsub, p.L);

    float A2[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) A2[i] = (dvalid && i < p.N) ? p.A[d * p.N + i] * kLog2e : 0.0f;
    const float Dd = (dvalid && p.Dskip) ? p.Dskip[d] : 0.0f;

    float h[NG], hr[NG], Q[NG];
    float sdel = 0.0f;
    float cf[NG], cr[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) cf[i] = cr[i] = 0.0f;

    if (chunked || p.WT > 1) {
        // ---- sub-chunk aggregate from a zero state
#pragma unroll
        for (int i = 0; i < NG; ++i) {
            h[i] = 0.0f;
            hr[i] = 0.0f;
            Q[i] = 1.0f;
        }
        sweep<NG, IO, SP, BIDIR, MODE_AGG, false>(p, b, d, dvalid, t0, t1, A2, Dd, h, hr, Q, sdel,
                                                 nullptr, false);
        float *mine = s_sub + ((warp * NSUB) * 32 + lane) * NG;
#pragma unroll
        for (int i = 0; i < NG; ++i) {
            mine[i] = ex2_approx(A2[i] * sdel);  // prod of dA over the sub-chunk
            mine[32 * NG + i] = h[i];
            if constexpr (BIDIR) mine[2 * 32 * NG + i] = hr[i];
        }
        __syncthreads();

        if (warp == 0) {
            if (chunked) {
                // chunk aggregate: fold the sub-chunks in order
                float Pc[NG], Hc[NG], Hrc[NG];
#pragma unroll
                for (int i = 0; i < NG; ++i) {
                    Pc[i] = 1.0f;
                    Hc[i] = 0.0f;
                    Hrc[i] = 0.0f;
                }
                for (int w = 0; w < p.WT; ++w) {
                    const float *s = s_sub + ((w * NSUB) * 32 + lane) * NG;
#pragma unroll
                    for (int i = 0; i < NG; ++i) {
                        Pc[i] *= s[i];
                        Hc[i] = fmaf(s[i], Hc[i], s[32 * NG + i]);
                    }
                }
                if constexpr (BIDIR) {
                    for (int w = p.WT - 1; w >= 0; --w) {
                        const float *s = s_sub + ((w * NSUB) * 32 + lane) * NG;
#pragma unroll
                        for (int i = 0; i < NG; ++i) Hrc[i] = fmaf(s[i], Hrc[i], s[2 * 32 * NG + i]);
                    }
                }
                const long long unit = seq * p.K + k;
                store_field<NG>(field_ptr<NG>(p, NF, unit, F_P, lane), Pc);
                store_field<NG>(field_ptr<NG>(p, NF, unit, F_H, lane), Hc);
                if constexpr (BIDIR) store_field<NG>(field_ptr<NG>(p, NF, unit, F_HR, lane), Hrc);
                publish_flag(p, unit, FL_AGG, tag, lane);

                // forward carry: nearest inclusive state on the left, then the
                // aggregates after it applied one by one in sequence order
                const int j = find_anchor<true>(p, seq, k, tag, lane);
                if (j == -2) {
                    if (lane == 0) record_error(p.ws, SS_ERR_TIMEOUT, 3u, (unsigned)unit, 0u);
                } else {
                    if (j >= 0) load_field<NG>(field_ptr<NG>(p, NF, seq * p.K + j, F_INC, lane), cf);
                    for (int m = j + 1; m < k; ++m) {
                        float Pm[NG], Hm[NG];
                        load_field<NG>(field_ptr<NG>(p, NF, seq * p.K + m, F_P, lane), Pm);
                        load_field<NG>(field_ptr<NG>(p, NF, seq * p.K + m, F_H, lane), Hm);
#pragma unroll
                        for (int i = 0; i < NG; ++i) cf[i] = fmaf(Pm[i], cf[i], Hm[i]);
                    }
                }
                float inc[NG];
#pragma unroll
                for (int i = 0; i < NG; ++i) inc[i] = fmaf(Pc[i], cf[i], Hc[i]);
                store_field<NG>(field_ptr<NG>(p, NF, unit, F_INC, lane), inc);
                publish_flag(p, unit, FL_INC, tag, lane);

                if constexpr (BIDIR) {
                    // reverse carry: nearest reverse inclusive state on the right
                    const int jr = find_anchor<false>(p, seq, k, tag, lane);
                    if (jr == -2) {
                        if (lane == 0) record_error(p.ws, SS_ERR_TIMEOUT, 4u, (unsigned)unit, 0u);
                    } else {
                        if (jr < p.K)
                            load_field<NG>(field_ptr<NG>(p, NF, seq * p.K + jr, F_RINC, lane), cr);
                        for (int m = jr - 1; m > k; --m) {
                            float Pm[NG], Hm[NG];
                            load_field<NG>(field_ptr<NG>(p, NF, seq * p.K + m, F_P, lane), Pm);
                            load_field<NG>(field_ptr<NG>(p, NF, seq * p.K + m, F_HR, lane), Hm);
#pragma unroll
                            for (int i = 0; i < NG; ++i) cr[i] = fmaf(Pm[i], cr[i], Hm[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < NG; ++i) inc[i] = fmaf(Pc[i], cr[i], Hrc[i]);
                    store_field<NG>(field_ptr<NG>(p, NF, unit, F_RINC, lane), inc);
                    publish_flag(p, unit, FL_RINC, tag, lane);
                }
            }
#pragma unroll
            for (int i = 0; i < NG; ++i) {
                s_car[lane * NG + i] = cf[i];
                s_car[(32 + lane) * NG + i] = cr[i];
            }
        }
        __syncthreads();

        // this warp's carries: the chunk carry moved across the earlier
        // (forward) or later (reverse) sub-chunks of the CTA, in order
#pragma unroll
        for (int i = 0; i < NG; ++i) {
            cf[i] = s_car[lane * NG + i];
            cr[i] = s_car[(32 + lane) * NG + i];
        }
        for (int w = 0; w < warp; ++w) {
            const float *s = s_sub + ((w * NSUB) * 32 + lane) * NG;
#pragma unroll
            for (int i = 0; i < NG; ++i) cf[i] = fmaf(s[i], cf[i], s[32 * NG + i]);
        }
        if constexpr (BIDIR) {
            for (int w = p.WT - 1; w > warp; --w) {
                const float *s = s_sub + ((w * NSUB) * 32 + lane) * NG;
#pragma unroll
                for (int i = 0; i < NG; ++i) cr[i] = fmaf(s[i], cr[i], s[2 * 32 * NG + i]);
            }
        }
    }

    // ---- outputs: forward sweep from the carry (and the reverse sweep)
#pragma unroll
    for (int i = 0; i < NG; ++i) h[i] = cf[i];
    float *yf = nullptr;
    if constexpr (BIDIR) yf = p.yscratch ? p.yscratch : static_cast<float *>(p.y);
    sweep<NG, IO, SP, BIDIR, MODE_OUT, false>(p, b, d, dvalid, t0, t1, A2, Dd, h, hr, Q, sdel, yf,
                                             false);
    if constexpr (BIDIR) {
#pragma unroll
        for (int i = 0; i < NG; ++i) h[i] = cr[i];
        sweep<NG, IO, SP, BIDIR, MODE_OUT, true>(p, b, d, dvalid, t0, t1, A2, Dd, h, hr, Q, sdel, yf,
                                                true);
    }

    if (chunked) finish_launch(p.ws, tag);
}

// ------------------------------------------------------------------ planning
struct Plan {
    int NG, WT, K, Tsub, dtiles;
    long long seqs;
    size_t desc_bytes, flag_bytes, payload_bytes, scratch_bytes, total;
    size_t smem;
};

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return 152;
    }
    return sms;
}

Plan make_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int bidir) {
    Plan pl{};
    pl.NG = N <= 4 ? 4 : (N <= 8 ? 8 : 16);
    pl.dtiles = (int)((D + 31) / 32);
    pl.seqs = B * pl.dtiles;
    const long long sms = device_sm_count();
    const long long target_warps = sms * 16;
    long long S = (target_warps + pl.seqs - 1) / std::max<long long>(pl.seqs, 1);
    S = std::max<long long>(1, std::min<long long>(S, (L + 31) / 32));
    int WT = (int)std::min<long long>(S, kMaxWT);
    long long K = (S + WT - 1) / WT;
    long long Tsub = (L + K * WT - 1) / (K * WT);
    Tsub = (Tsub + 3) / 4 * 4;
    if (const char *e = std::getenv("SS_S6_WT_TSUB")) {  // tuning override "WT,Tsub"
        int w = 0, t = 0;
        if (std::sscanf(e, "%d,%d", &w, &t) == 2 && w >= 1 && w <= kMaxWT && t >= 1) {
            WT = w;
            Tsub = t;
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
    pl.smem = (size_t)(pl.WT * NSUB + 2) * 32 * pl.NG * sizeof(float);
    return pl;
}

template <int NG, typename IO, bool SP, bool BIDIR>
ss_status launch_t(const S6Params &prm, const Plan &pl, cudaStream_t stream) {
    auto kern = s6_kernel<NG, IO, SP, BIDIR>;
    if (pl.smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) !=
            cudaSuccess)
            return SS_ERR_CUDA;
    }
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

template <int NG, typename IO>
ss_status launch_ng(const S6Params &prm, const Plan &pl, bool sp, bool bidir, cudaStream_t s) {
    if (bidir) return sp ? launch_t<NG, IO, true, true>(prm, pl, s) : launch_t<NG, IO, false, true>(prm, pl, s);
    return sp ? launch_t<NG, IO, true, false>(prm, pl, s) : launch_t<NG, IO, false, false>(prm, pl, s);
}

template <typename IO>
ss_status launch_io(const S6Params &prm, const Plan &pl, bool sp, bool bidir, cudaStream_t s) {
    switch (pl.NG) {
        case 4: return launch_ng<4, IO>(prm, pl, sp, bidir, s);
        case 8: return launch_ng<8, IO>(prm, pl, sp, bidir, s);
        default: return launch_ng<16, IO>(prm, pl, sp, bidir, s);
    }
}

}  // namespace

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
    const uintptr_t al = reinterpret_cast<uintptr_t>(a.Bt) | reinterpret_cast<uintptr_t>(a.Ct);
    prm.vecBC = (a.N == pl.NG) && ((a.N * es) % 16 == 0) && (al % 16 == 0);
    prm.timeout_ns = timeout_ns;
    prm.skip_unit = skip_unit;
    char *ws = static_cast<char *>(workspace);
    prm.ws = reinterpret_cast<WsHeader *>(ws);
    prm.flags = pl.K > 1 ? reinterpret_cast<unsigned *>(ws + kWsHeaderBytes) : nullptr;
    prm.payload = pl.K > 1 ? reinterpret_cast<float *>(ws + kWsHeaderBytes + pl.flag_bytes) : nullptr;
    prm.yscratch = pl.scratch_bytes ? reinterpret_cast<float *>(ws + kWsHeaderBytes + pl.desc_bytes) : nullptr;
    const bool sp = a.softplus != 0, bd = a.bidir != 0;
    return a.io_bf16 ? launch_io<__nv_bfloat16>(prm, pl, sp, bd, stream)
                     : launch_io<float>(prm, pl, sp, bd, stream);
}

}  // namespace ss
