// Selective-scan layer forward: the three input projections, then the scan.
//
// "POPCORNBENCH FW-GLM-5-1 l2_p30", the model's parameters and forward pass:
// delta = softplus(proj_delta(x)) with a bias, B_t = proj_B(x), C_t =
// proj_C(x), then the S6 recurrence. The three projections are one dense
// GEMM: x ((B*L) x D) times the stacked weights W_proj ((D + 2N) x D)
// transposed, into one (B*L) x ld workspace buffer whose row holds the
// pre-activation, B_t and C_t of one step; the scan reads the three column
// blocks in place at that row stride, with softplus fused in.
//  * bf16: the hand-written tensor-core GEMM (proj_gemm.cu) adds the delta
//    bias to the fp32 accumulator and rounds once to bf16, as a bf16 Linear
//    layer does; rows are padded to a multiple of 8 elements (16 bytes).
//  * fp32: a cuBLASLt fp32 GEMM (full fp32 products and sums; the tensor
//    cores have no fp32-exact mode) and the scan adds the bias in fp32.
#include <cublasLt.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr size_t kLtWorkspace = 32u << 20;  // cuBLASLt scratch per call

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

cublasLtHandle_t lt_handle() {
    static std::once_flag once;
    static cublasLtHandle_t h = nullptr;
    std::call_once(once, [] {
        if (cublasLtCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
    });
    return h;
}

// out (M x nout, row-major) = x (M x K, row-major) * W^T, W (nout x K,
// row-major: the Linear weight layout). In cuBLAS's column-major terms:
// out^T (nout x M) = op(W) * x^T with W viewed as K x nout, transposed.
ss_status gemm_xwT(const void *x, const void *W, void *out, int64_t M, int64_t K, int64_t nout,
                   bool bf16, void *lt_ws, cudaStream_t stream) {
    cublasLtHandle_t h = lt_handle();
    if (!h) return SS_ERR_CUDA;
    const cudaDataType_t t = bf16 ? CUDA_R_16BF : CUDA_R_32F;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    ss_status st = SS_ERR_CUDA;
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    const size_t wsb = kLtWorkspace;
    cublasLtMatmulHeuristicResult_t heur{};
    int found = 0;
    const float alpha = 1.0f, beta = 0.0f;
    if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) !=
            CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) !=
            CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&la, t, (uint64_t)K, (uint64_t)nout, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&lb, t, (uint64_t)K, (uint64_t)M, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&lc, t, (uint64_t)nout, (uint64_t)M, nout) !=
            CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb,
                                             sizeof(wsb)) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, lc, lc, pref, 1, &heur, &found) !=
            CUBLAS_STATUS_SUCCESS ||
        found < 1) {
        st = SS_ERR_UNSUPPORTED;
    } else if (cublasLtMatmul(h, op, &alpha, W, la, x, lb, &beta, out, lc, out, lc, &heur.algo,
                              lt_ws, wsb, stream) == CUBLAS_STATUS_SUCCESS) {
        st = SS_OK;
    }
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (lc) cublasLtMatrixLayoutDestroy(lc);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return st;
}

struct LayerPlan {
    size_t proj, lt, scan, total;  // section offsets, then total bytes
    int64_t ld;                    // row stride (elements) of the projections
};

LayerPlan layer_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16) {
    LayerPlan pl{};
    const size_t es = io_bf16 ? 2 : 4;
    const size_t M = (size_t)(B * L);
    pl.ld = io_bf16 ? (D + 2 * N + 7) / 8 * 8 : D + 2 * N;
    // the scan's section comes first, so the workspace starts with its
    // header (error word) even when the scan needs no further workspace
    pl.scan = 0;
    pl.proj = std::max<size_t>(kWsHeaderBytes, align256(s6_workspace_bytes(B, L, D, N, io_bf16, 0)));
    pl.lt = pl.proj + align256(M * (size_t)pl.ld * es);
    pl.total = pl.lt + (io_bf16 ? 0 : kLtWorkspace);
    return pl;
}

}  // namespace

size_t layer_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16) {
    if (B <= 0 || L <= 0 || D <= 0 || N <= 0) return 0;
    return layer_plan(B, L, D, N, io_bf16).total;
}

ss_status layer_fwd_launch(const void *x, const void *W_proj, const float *b_delta, const float *A,
                           const float *Dskip, void *y, int64_t B, int64_t L, int64_t D,
                           int64_t N, int io_bf16, void *workspace, size_t ws_bytes,
                           cudaStream_t stream, unsigned long long timeout_ns, long long skip_unit) {
    const LayerPlan pl = layer_plan(B, L, D, N, io_bf16);
    if (workspace == nullptr || ws_bytes < pl.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return SS_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    const size_t es = io_bf16 ? 2 : 4;
    const int64_t M = B * L;
    // rows [0, D) of W_proj: proj_delta; [D, D + N): proj_B; [D + N, D + 2N):
    // proj_C, so output row m is (pre-activation, B_t, C_t) of step m
    ss_status st;
    if (io_bf16) {
        if (!proj_gemm_supported(x, W_proj, ws + pl.proj, M, D, D + 2 * N, pl.ld))
            return SS_ERR_UNSUPPORTED;
        st = proj_gemm_launch(x, W_proj, ws + pl.proj, b_delta, D, M, D, D + 2 * N, pl.ld, ws,
                              stream, timeout_ns);
    } else {
        st = gemm_xwT(x, W_proj, ws + pl.proj, M, D, D + 2 * N, false, ws + pl.lt, stream);
    }
    if (st != SS_OK) return st;
    S6Args a;
    a.x = x;
    a.delta = ws + pl.proj;
    a.Bt = ws + pl.proj + (size_t)D * es;
    a.Ct = ws + pl.proj + (size_t)(D + N) * es;
    a.ld_delta = pl.ld;
    a.ld_bc = pl.ld;
    a.A = A;
    a.Dskip = Dskip;
    a.y = y;
    a.delta_bias = io_bf16 ? nullptr : b_delta;  // bf16: added in the GEMM epilogue
    a.h0 = nullptr;
    a.h_last = nullptr;
    a.B = B;
    a.L = L;
    a.D = D;
    a.N = N;
    a.io_bf16 = io_bf16;
    a.softplus = 1;
    a.bidir = 0;
    return s6_launch(a, ws + pl.scan, pl.proj - pl.scan, stream, timeout_ns, skip_unit);
}

}  // namespace ss
