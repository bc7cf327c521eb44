// C ABI of libss.so: argument validation, workspace checks, dispatch.
// The arithmetic lives in affine_scan.cu and s6_scan.cu.
#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "ss_common.cuh"
#include "ss_internal.h"
#include "ss_testing.h"

namespace {

std::atomic<unsigned long long> g_timeout_ns{1000000000ull};
std::atomic<long long> g_skip_unit{-1};

using ss::take_skip_unit;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ss_status s6_entry(const void *x, const void *delta, const void *Bt, const void *Ct, const float *A,
                   const float *Dskip, void *y, int64_t B, int64_t L, int64_t D, int64_t N,
                   int io_dtype, int delta_softplus, void *workspace, size_t workspace_bytes,
                   void *stream, int bidir, const float *h0 = nullptr, float *h_last = nullptr) {
    if (B < 0 || L < 0 || D < 0 || N < 0) return SS_ERR_INVALID;
    if (io_dtype != SS_F32 && io_dtype != SS_BF16) return SS_ERR_INVALID;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    if (B == 0 || L == 0 || D == 0) return SS_OK;
    if (!x || !delta || !Bt || !Ct || !A || !y) return SS_ERR_INVALID;
    const uintptr_t es = io_dtype == SS_BF16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(delta, es) || !aligned(Bt, es) || !aligned(Ct, es) ||
        !aligned(y, es) || !aligned(A, 4) || (Dskip && !aligned(Dskip, 4)) ||
        (h0 && !aligned(h0, 4)) || (h_last && !aligned(h_last, 4)))
        return SS_ERR_INVALID;
    if (B > (1LL << 31) || L > (1LL << 40) || D > (1LL << 31) || B * L > (1LL << 48))
        return SS_ERR_UNSUPPORTED;
    ss::S6Args a;
    a.x = x;
    a.delta = delta;
    a.Bt = Bt;
    a.Ct = Ct;
    a.A = A;
    a.Dskip = Dskip;
    a.y = y;
    a.h0 = h0;
    a.h_last = h_last;
    a.B = B;
    a.L = L;
    a.D = D;
    a.N = N;
    a.io_bf16 = io_dtype == SS_BF16;
    a.softplus = delta_softplus != 0;
    a.bidir = bidir;
    return ss::s6_launch(a, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                         g_timeout_ns.load(), take_skip_unit());
}

ss_status affine_entry(const float *a, const float *b, float *h, int64_t n, void *workspace,
                       size_t workspace_bytes, void *stream, bool log_step,
                       const float *h0 = nullptr) {
    if (n < 0) return SS_ERR_INVALID;
    if (n == 0) return SS_OK;
    if (!a || !b || !h) return SS_ERR_INVALID;
    if (!aligned(a, 4) || !aligned(b, 4) || !aligned(h, 4) || (h0 && !aligned(h0, 4)))
        return SS_ERR_INVALID;
    if (h0 && h0 >= h && h0 < h + n) return SS_ERR_INVALID;  // the kernel writes h
    const size_t need = ss::affine_workspace_bytes(n);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SS_ERR_WORKSPACE;
    return ss::affine_launch(a, b, h, n, workspace, static_cast<cudaStream_t>(stream),
                             g_timeout_ns.load(), take_skip_unit(), log_step, h0);
}

}  // namespace

namespace ss {
unsigned long long spin_timeout_ns() { return g_timeout_ns.load(); }

ss_status raise_smem_limit(const void *fn, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> limits;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SS_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    int &cur = limits[{dev, fn}];
    if (bytes <= cur) return SS_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return SS_ERR_CUDA;
    }
    cur = bytes;
    return SS_OK;
}
long long take_skip_unit() { return g_skip_unit.exchange(-1); }
}  // namespace ss

extern "C" {

const char *ss_status_string(int status) {
    switch (status) {
        case SS_OK: return "SS_OK";
        case SS_ERR_INVALID: return "SS_ERR_INVALID";
        case SS_ERR_UNSUPPORTED: return "SS_ERR_UNSUPPORTED";
        case SS_ERR_WORKSPACE: return "SS_ERR_WORKSPACE";
        case SS_ERR_CUDA: return "SS_ERR_CUDA";
        case SS_ERR_TIMEOUT: return "SS_ERR_TIMEOUT";
        case SS_ERR_BOUNDS: return "SS_ERR_BOUNDS";
        default: return "SS_ERR_UNKNOWN";
    }
}

int ss_abi_version(void) { return SS_ABI_VERSION; }

size_t ss_affine_scan_workspace_bytes(int64_t n) { return ss::affine_workspace_bytes(n); }

ss_status ss_affine_scan(const float *a, const float *b, float *h, int64_t n, void *workspace,
                         size_t workspace_bytes, void *stream) {
    return affine_entry(a, b, h, n, workspace, workspace_bytes, stream, false);
}

ss_status ss_affine_scan_log_step(const float *a, const float *b, float *h, int64_t n,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    return affine_entry(a, b, h, n, workspace, workspace_bytes, stream, true);
}

ss_status ss_affine_scan_state(const float *a, const float *b, float *h, int64_t n,
                               const float *h0, void *workspace, size_t workspace_bytes,
                               void *stream) {
    return affine_entry(a, b, h, n, workspace, workspace_bytes, stream, false, h0);
}

size_t ss_affine_scan_host_workspace_bytes(int64_t n) { return ss::affine_host_workspace_bytes(n); }

ss_status ss_affine_scan_host(const float *a, const float *b, float *h, int64_t n,
                              void *workspace, size_t workspace_bytes, void *stream) {
    if (n < 0) return SS_ERR_INVALID;
    if (n == 0) return SS_OK;
    if (!a || !b || !h) return SS_ERR_INVALID;
    if (!aligned(a, 4) || !aligned(b, 4) || !aligned(h, 4)) return SS_ERR_INVALID;
    if (!workspace || workspace_bytes < ss::affine_host_workspace_bytes(n) ||
        !aligned(workspace, 256))
        return SS_ERR_WORKSPACE;
    return ss::affine_host_launch(a, b, h, n, workspace, workspace_bytes,
                                  static_cast<cudaStream_t>(stream), g_timeout_ns.load());
}

size_t ss_selective_scan_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N, int io_dtype,
                                         int bidir) {
    if (N < 1 || N > 16 || (io_dtype != SS_F32 && io_dtype != SS_BF16)) return 0;
    return ss::s6_workspace_bytes(B, L, D, N, io_dtype == SS_BF16, bidir != 0);
}

ss_status ss_selective_scan_fwd(const void *x, const void *delta, const void *Bt, const void *Ct,
                                const float *A, const float *Dskip, void *y, int64_t B, int64_t L,
                                int64_t D, int64_t N, int io_dtype, int delta_softplus,
                                void *workspace, size_t workspace_bytes, void *stream) {
    return s6_entry(x, delta, Bt, Ct, A, Dskip, y, B, L, D, N, io_dtype, delta_softplus, workspace,
                    workspace_bytes, stream, 0);
}

ss_status ss_selective_scan_bidir(const void *x, const void *delta, const void *Bt, const void *Ct,
                                  const float *A, const float *Dskip, void *y, int64_t B, int64_t L,
                                  int64_t D, int64_t N, int io_dtype, int delta_softplus,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    return s6_entry(x, delta, Bt, Ct, A, Dskip, y, B, L, D, N, io_dtype, delta_softplus, workspace,
                    workspace_bytes, stream, 1);
}

ss_status ss_selective_scan_fwd_state(const void *x, const void *delta, const void *Bt,
                                      const void *Ct, const float *A, const float *Dskip,
                                      const float *h0, void *y, float *h_last, int64_t B,
                                      int64_t L, int64_t D, int64_t N, int io_dtype,
                                      int delta_softplus, void *workspace, size_t workspace_bytes,
                                      void *stream) {
    return s6_entry(x, delta, Bt, Ct, A, Dskip, y, B, L, D, N, io_dtype, delta_softplus, workspace,
                    workspace_bytes, stream, 0, h0, h_last);
}

size_t ss_selective_scan_layer_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N,
                                               int io_dtype) {
    if (N < 1 || N > 16 || (io_dtype != SS_F32 && io_dtype != SS_BF16)) return 0;
    return ss::layer_workspace_bytes(B, L, D, N, io_dtype == SS_BF16);
}

ss_status ss_selective_scan_layer_fwd(const void *x, const void *W_proj, const float *b_delta,
                                      const float *A, const float *Dskip, void *y, int64_t B,
                                      int64_t L, int64_t D, int64_t N, int io_dtype,
                                      void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || L < 0 || D < 0 || N < 0) return SS_ERR_INVALID;
    if (io_dtype != SS_F32 && io_dtype != SS_BF16) return SS_ERR_INVALID;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    if (B == 0 || L == 0 || D == 0) return SS_OK;
    if (!x || !W_proj || !b_delta || !A || !y) return SS_ERR_INVALID;
    const uintptr_t es = io_dtype == SS_BF16 ? 2 : 4;
    if (!aligned(x, es) || !aligned(W_proj, es) || !aligned(y, es) || !aligned(b_delta, 4) ||
        !aligned(A, 4) || !aligned(Dskip, 4))
        return SS_ERR_INVALID;
    if (B > (1LL << 31) || L > (1LL << 40) || D > (1LL << 31) || B * L > (1LL << 48))
        return SS_ERR_UNSUPPORTED;
    return ss::layer_fwd_launch(x, W_proj, b_delta, A, Dskip, y, B, L, D, N,
                                io_dtype == SS_BF16, workspace, workspace_bytes,
                                static_cast<cudaStream_t>(stream), g_timeout_ns.load(),
                                take_skip_unit());
}

size_t ss_selective_scan_bwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N) {
    if (N < 1 || N > 16) return 0;
    return ss::s6_bwd_workspace_bytes(B, L, D, N);
}

ss_status ss_selective_scan_bwd(const void *x, const void *delta, const void *Bt, const void *Ct,
                                const float *A, const float *Dskip, const float *h0, const void *dy,
                                const float *dh_last, void *dx, void *ddelta, float *dA,
                                float *dBt, float *dCt, float *dDskip, float *dh0, int64_t B,
                                int64_t L, int64_t D, int64_t N, int io_dtype, int delta_softplus,
                                void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || L < 0 || D < 0 || N < 0) return SS_ERR_INVALID;
    if (io_dtype != SS_F32 && io_dtype != SS_BF16) return SS_ERR_INVALID;
    if (N < 1 || N > 16) return SS_ERR_UNSUPPORTED;
    if (B > (1LL << 31) || L > (1LL << 40) || D > (1LL << 31) || B * L > (1LL << 48))
        return SS_ERR_UNSUPPORTED;
    const uintptr_t es = io_dtype == SS_BF16 ? 2 : 4;
    const bool empty = B == 0 || L == 0 || D == 0;
    if (!A || !dA || (!empty && (!x || !delta || !Bt || !Ct || !dy || !dx || !ddelta)) ||
        (B * L > 0 && (!dBt || !dCt)))
        return SS_ERR_INVALID;
    if (!aligned(x, es) || !aligned(delta, es) || !aligned(Bt, es) || !aligned(Ct, es) ||
        !aligned(dy, es) || !aligned(dx, es) || !aligned(ddelta, es) || !aligned(A, 4) ||
        !aligned(Dskip, 4) || !aligned(h0, 4) || !aligned(dh_last, 4) || !aligned(dA, 4) ||
        !aligned(dBt, 4) || !aligned(dCt, 4) || !aligned(dDskip, 4) || !aligned(dh0, 4))
        return SS_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (empty) {
        // sums over nothing are zero; with no steps h_last is h0, so dh0 = dh_last
        bool ok = cudaMemsetAsync(dA, 0, (size_t)(D * N) * sizeof(float), s) == cudaSuccess;
        if (dDskip) ok &= cudaMemsetAsync(dDskip, 0, (size_t)D * sizeof(float), s) == cudaSuccess;
        if (B * L > 0) {
            ok &= cudaMemsetAsync(dBt, 0, (size_t)(B * L * N) * sizeof(float), s) == cudaSuccess;
            ok &= cudaMemsetAsync(dCt, 0, (size_t)(B * L * N) * sizeof(float), s) == cudaSuccess;
        }
        if (dh0 && B * D > 0) {
            const size_t bytes = (size_t)(B * D * N) * sizeof(float);
            ok &= (dh_last && L == 0
                       ? cudaMemcpyAsync(dh0, dh_last, bytes, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(dh0, 0, bytes, s)) == cudaSuccess;
        }
        return ok ? SS_OK : SS_ERR_CUDA;
    }
    ss::S6BwdArgs a;
    a.x = x;
    a.delta = delta;
    a.Bt = Bt;
    a.Ct = Ct;
    a.dy = dy;
    a.A = A;
    a.Dskip = Dskip;
    a.h0 = h0;
    a.dh_last = dh_last;
    a.dx = dx;
    a.ddelta = ddelta;
    a.dA = dA;
    a.dBt = dBt;
    a.dCt = dCt;
    a.dDskip = dDskip;
    a.dh0 = dh0;
    a.B = B;
    a.L = L;
    a.D = D;
    a.N = N;
    a.io_bf16 = io_dtype == SS_BF16;
    a.softplus = delta_softplus != 0;
    return ss::s6_bwd_launch(a, workspace, workspace_bytes, s);
}

ss_status ss_get_device_status(void *workspace, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SS_ERR_CUDA;
    if (!workspace) return SS_OK;
    ss::WsHeader *ws = static_cast<ss::WsHeader *>(workspace);
    unsigned err = 0;
    if (cudaMemcpy(&err, &ws->error, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SS_ERR_CUDA;
    if (err != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(&ws->error, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return SS_ERR_CUDA;
    }
    return static_cast<ss_status>(err);
}

void ss_testing_skip_publish_once(int64_t unit) { g_skip_unit.store(unit < 0 ? -1 : unit); }

void ss_testing_s6_plan(int kind, int a, int b, int c) { ss::s6_set_plan_override(kind, a, b, c); }

int ss_testing_proj_gemm(const void *x, const void *W, void *out, const float *bias,
                         int64_t n_bias, int64_t M, int64_t K, int64_t Nout, int64_t ld_out,
                         void *workspace, void *stream) {
    if (M < 0 || K < 0 || Nout < 0 || n_bias < 0) return SS_ERR_INVALID;
    if (M == 0 || Nout == 0) return SS_OK;
    if (!x || !W || !out || !workspace || !aligned(workspace, 256)) return SS_ERR_INVALID;
    return ss::proj_gemm_launch(x, W, out, bias, n_bias, M, K, Nout, ld_out, workspace,
                                static_cast<cudaStream_t>(stream), g_timeout_ns.load());
}

int ss_testing_proj_gemm_describe_plan(int64_t M, int64_t K, int64_t Nout, int64_t *out) {
    return ss::proj_gemm_describe_plan(M, K, Nout, out);
}

int ss_testing_s6_describe_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_dtype,
                                int bidir, int64_t *out) {
    if (!out || (io_dtype != SS_F32 && io_dtype != SS_BF16)) return -1;
    return ss::s6_describe_plan(B, L, D, N, io_dtype == SS_BF16, bidir != 0, out);
}

ss_status ss_set_spin_timeout_ns(uint64_t ns) {
    if (ns == 0) return SS_ERR_INVALID;
    g_timeout_ns.store(ns);
    return SS_OK;
}

}  // extern "C"
