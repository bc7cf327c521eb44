"""The C ABI library: loads without a GPU, exports what include/ss.h
declares, and rejects bad arguments synchronously (no launch, no GPU)."""
import ctypes
import os
import re

import pytest

import linear_recurrences_gb300 as ss
from linear_recurrences_gb300 import build as ssbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    ssbuild.build()
    return ss.lib()


def declared_functions():
    names = set()
    for f in os.listdir(INCLUDE):
        if f.endswith(".h"):
            text = open(os.path.join(INCLUDE, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ss_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("ss_affine_scan", "ss_selective_scan_fwd", "ss_selective_scan_bidir"):
        assert required in names
    assert set(names) == set(ss.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} not exported by libss.so"


def test_status_strings(L):
    assert ss.ss_status_string(ss.SS_OK) == "SS_OK"
    assert ss.ss_status_string(ss.SS_ERR_TIMEOUT) == "SS_ERR_TIMEOUT"
    assert ss.ss_status_string(99) == "SS_ERR_UNKNOWN"
    assert L.ss_abi_version() == 1


def test_affine_argument_errors(L):
    p = ctypes.c_void_p(256)  # never dereferenced: every call below fails validation
    assert L.ss_affine_scan(p, p, p, -1, p, 1 << 20, None) == ss.SS_ERR_INVALID
    assert L.ss_affine_scan(None, p, p, 10, p, 1 << 20, None) == ss.SS_ERR_INVALID
    assert L.ss_affine_scan(ctypes.c_void_p(258), p, p, 10, p, 1 << 20, None) == ss.SS_ERR_INVALID
    assert L.ss_affine_scan(p, p, p, 10, None, 0, None) == ss.SS_ERR_WORKSPACE
    assert L.ss_affine_scan(p, p, p, 10000, p, 64, None) == ss.SS_ERR_WORKSPACE
    assert L.ss_affine_scan(p, p, p, 0, None, 0, None) == ss.SS_OK  # empty: nothing to do


def test_affine_state_and_host_argument_errors(L):
    p = ctypes.c_void_p(256)
    h = ctypes.c_void_p(4096)
    inside = ctypes.c_void_p(4096 + 4 * 5)  # h0 at h[5]: the kernel would overwrite it
    assert L.ss_affine_scan_state(p, p, h, 10, inside, p, 1 << 20, None) == ss.SS_ERR_INVALID
    assert L.ss_affine_scan_state(p, p, h, 10, ctypes.c_void_p(258), p, 1 << 20, None) == \
        ss.SS_ERR_INVALID
    assert L.ss_affine_scan_state(p, p, h, -1, None, p, 1 << 20, None) == ss.SS_ERR_INVALID
    assert L.ss_affine_scan_state(p, p, h, 10, None, None, 0, None) == ss.SS_ERR_WORKSPACE
    assert L.ss_affine_scan_state(p, p, h, 0, None, None, 0, None) == ss.SS_OK
    assert L.ss_affine_scan_host(p, p, h, -1, p, 1 << 30, None) == ss.SS_ERR_INVALID
    assert L.ss_affine_scan_host(None, p, h, 10, p, 1 << 30, None) == ss.SS_ERR_INVALID
    assert L.ss_affine_scan_host(p, p, h, 10, p, 64, None) == ss.SS_ERR_WORKSPACE
    assert L.ss_affine_scan_host(p, p, h, 0, None, 0, None) == ss.SS_OK


def test_affine_host_workspace_size(L):
    """Scan workspace for one chunk (2^23 elements at most), then three slots
    of a, b and h for one chunk each, every section 256-byte aligned."""
    assert L.ss_affine_scan_host_workspace_bytes(0) == 0
    assert L.ss_affine_scan_host_workspace_bytes(1) == 512 + 9 * 256
    chunk = 1 << 23
    full = (256 + 32 * (chunk // 4096)) + 9 * 4 * chunk
    assert L.ss_affine_scan_host_workspace_bytes(chunk) == full
    assert L.ss_affine_scan_host_workspace_bytes(1 << 28) == full


def test_affine_workspace_size(L):
    assert L.ss_affine_scan_workspace_bytes(0) == 0
    assert L.ss_affine_scan_workspace_bytes(1) == 256 + 32
    assert L.ss_affine_scan_workspace_bytes(4096) == 256 + 32
    assert L.ss_affine_scan_workspace_bytes(4097) == 256 + 64
    assert L.ss_affine_scan_workspace_bytes(1 << 28) == 256 + 32 * 65536


def test_s6_argument_errors(L):
    p = ctypes.c_void_p(256)
    args = lambda B, L_, D, N, io=0, sp=0, ws=None, wsb=0: (
        p, p, p, p, p, None, p, B, L_, D, N, io, sp, ws, wsb, None)
    for fn in (L.ss_selective_scan_fwd, L.ss_selective_scan_bidir):
        assert fn(*args(2, 8, 4, 17)) == ss.SS_ERR_UNSUPPORTED
        assert fn(*args(2, 8, 4, 0)) == ss.SS_ERR_UNSUPPORTED
        assert fn(*args(-1, 8, 4, 16)) == ss.SS_ERR_INVALID
        assert fn(*args(2, 8, 4, 16, io=7)) == ss.SS_ERR_INVALID
        assert fn(*args(0, 8, 4, 16)) == ss.SS_OK
        assert fn(*args(2, 0, 4, 16)) == ss.SS_OK
        bad = (None, p, p, p, p, None, p, 2, 8, 4, 16, 0, 0, None, 0, None)
        assert fn(*bad) == ss.SS_ERR_INVALID
    assert L.ss_selective_scan_workspace_bytes(2, 8, 4, 17, 0, 0) == 0


def test_s6_state_argument_errors(L):
    p = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(258)  # not 4-byte aligned
    fn = L.ss_selective_scan_fwd_state
    args = lambda h0, hl, B=2, L_=8, D=4, N=16: (
        p, p, p, p, p, None, h0, p, hl, B, L_, D, N, 0, 0, None, 0, None)
    assert fn(*args(odd, p)) == ss.SS_ERR_INVALID
    assert fn(*args(p, odd)) == ss.SS_ERR_INVALID
    assert fn(*args(None, None, N=17)) == ss.SS_ERR_UNSUPPORTED
    assert fn(*args(p, p, L_=0)) == ss.SS_OK  # empty: nothing launched, nothing written
    assert fn(*args(p, p, B=-1)) == ss.SS_ERR_INVALID


def test_s6_bwd_argument_errors(L):
    p = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(258)
    fn = L.ss_selective_scan_bwd
    # x delta Bt Ct A Dskip h0 dy dh_last dx ddelta dA dBt dCt dDskip dh0
    args = lambda ptrs, B=2, L_=8, D=4, N=16, io=0: (*ptrs, B, L_, D, N, io, 0, p, 1 << 30, None)
    full = [p] * 16
    assert fn(*args(full, N=17)) == ss.SS_ERR_UNSUPPORTED
    assert fn(*args(full, io=5)) == ss.SS_ERR_INVALID
    assert fn(*args(full, B=-1)) == ss.SS_ERR_INVALID
    for i in (0, 1, 2, 3, 4, 7, 9, 10, 11, 12, 13):  # required pointers
        bad = list(full)
        bad[i] = None
        assert fn(*args(bad)) == ss.SS_ERR_INVALID, f"null argument {i} accepted"
    for i in range(16):
        bad = list(full)
        bad[i] = odd
        assert fn(*args(bad)) == ss.SS_ERR_INVALID, f"misaligned argument {i} accepted"
    assert fn(*(full + [2, 8, 4, 16, 0, 0, None, 0, None])) == ss.SS_ERR_WORKSPACE
    assert L.ss_selective_scan_bwd_workspace_bytes(2, 8, 4, 17) == 0
    assert L.ss_selective_scan_bwd_workspace_bytes(0, 8, 4, 16) == 0


def test_spin_timeout(L):
    assert L.ss_set_spin_timeout_ns(0) == ss.SS_ERR_INVALID
    assert L.ss_set_spin_timeout_ns(10**9) == ss.SS_OK


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "linear_recurrences_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"


def test_library_reads_no_environment():
    """Plans and workspace sizes depend on the call's arguments only: no
    source of the library reads an environment variable (a stray one could
    change a plan between a workspace-size query and the launch)."""
    csrc = os.path.join(ROOT, "linear_recurrences_gb300", "csrc")
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            text = open(os.path.join(csrc, f)).read()
            assert "getenv" not in text and "environ" not in text, f"{f} reads the environment"


def _chunked_plan(B, Lq, D, N, io, bidir):
    """(chunks per sequence, warps per CTA, timesteps per warp) the chunked
    kernel's planner takes for a shape (the time-parallel pass set aside)."""
    ss.ss_testing_s6_plan(1, 0, 0, 1)
    try:
        kind, p = ss.ss_testing_s6_describe_plan(B, Lq, D, N, io, bidir)
    finally:
        ss.ss_testing_s6_plan(0)
    assert kind == 0
    return p[3], p[1], p[2]


def test_forward_plans_fill_whole_waves(L):
    """The chunked planner's sub-chunk choice for the three S6 workloads on
    152 SMs (the values it falls back to without a GPU): 7 chunks of 4 x 80
    steps for fp32 (896 CTAs, 1.96 waves of 456), 8 of 4 x 128 for bf16, 27
    of 4 x 152 for the bidirectional workload (1296 CTAs, 2.84 waves)."""
    assert _chunked_plan(16, 2048, 256, 16, ss.SS_F32, 0) == (7, 4, 80)
    assert _chunked_plan(8, 4096, 1536, 16, ss.SS_BF16, 0) == (8, 4, 128)
    assert _chunked_plan(2, 16384, 768, 16, ss.SS_F32, 1) == (27, 4, 152)
    # within one wave the plan is left alone
    assert _chunked_plan(1, 1000, 96, 16, ss.SS_F32, 0)[0] == 8


def test_planner_paths(L):
    """Bidirectional shapes and forward shapes with few channels take the
    chunked kernel; the test override forces the time-parallel pass on
    forward shapes only."""  # noqa: D401
    assert ss.ss_testing_s6_describe_plan(2, 16384, 768, 16, ss.SS_F32, 1)[0] == 0
    assert ss.ss_testing_s6_describe_plan(1, 5000, 64, 16, ss.SS_F32, 0)[0] == 0
    # forward shapes with channels for two 32-channel CTAs per SM: the
    # wavefront single pass (13 steps x 4 slices); the fp32 workload has 128
    # such CTAs and stays chunked
    assert ss.ss_testing_s6_describe_plan(8, 4096, 1536, 16, ss.SS_BF16, 0) == \
        (2, (13, 4, 32, 79, 384, 52))
    assert ss.ss_testing_s6_describe_plan(16, 2048, 256, 16, ss.SS_F32, 0)[0] == 0
    ss.ss_testing_s6_plan(2, 4, 9, 2)
    try:
        k, p = ss.ss_testing_s6_describe_plan(1, 5000, 64, 16, ss.SS_F32, 0)
        assert k == 1 and p[:3] == (4, 9, 2)
        assert ss.ss_testing_s6_describe_plan(1, 5000, 64, 16, ss.SS_F32, 1)[0] == 0
    finally:
        ss.ss_testing_s6_plan(0)
    assert ss.ss_testing_s6_describe_plan(1, 10, 8, 17, ss.SS_F32, 0)[0] == -1


def test_time_parallel_workspace_size(L):
    """Forward workspace of a time-parallel plan: the chunked plan's section
    (for inputs whose rows turn out unaligned), then the packed B_t / C_t:
    per sequence and block, ceil(N / 8) slots of 2 matrices x 4 state pairs
    x 16 slices x 5 float4 (80-byte slice rows)."""
    B, Lq, D, N = 16, 2048, 256, 16
    nblk = (Lq + 143) // 144
    pack = B * nblk * 2 * (2 * 4 * 16 * 80)
    ss.ss_testing_s6_plan(1, 0, 0, 1)
    try:
        chunked = L.ss_selective_scan_workspace_bytes(B, Lq, D, N, ss.SS_F32, 0)
    finally:
        ss.ss_testing_s6_plan(0)
    ss.ss_testing_s6_plan(2, 2, 9, 4)
    try:
        total = L.ss_selective_scan_workspace_bytes(B, Lq, D, N, ss.SS_F32, 0)
    finally:
        ss.ss_testing_s6_plan(0)
    assert total == (chunked + 255) // 256 * 256 + pack


def _bwd_ranges(L, B, Lq, D, N):
    """Channel ranges of the backward plan, from its workspace size: six
    (B, K, D, N) sections, one (B, K, D), two (ranges, B, L, N)."""
    K = (Lq + 255) // 256
    al = lambda v: (v + 255) // 256 * 256
    fixed = 6 * al(B * K * D * N * 4) + al(B * K * D * 4)
    rest = L.ss_selective_scan_bwd_workspace_bytes(B, Lq, D, N) - fixed
    for sd in range(1, 1025):
        if rest == 2 * al(sd * B * Lq * N * 4):
            return sd
    raise AssertionError("workspace size matches no channel split")


def test_backward_plans_fill_whole_waves(L):
    """Channel ranges per (b, chunk) minimising waves x (channels + 16) at 2
    gradient CTAs per SM on 152 SMs: 2 for the fp32 workload, 7 for bf16."""
    assert _bwd_ranges(L, 16, 2048, 256, 16) == 2
    assert _bwd_ranges(L, 8, 4096, 1536, 16) == 7


def test_projection_gemm_plans(L):
    """The projection GEMM's planner (host only): the layer's shape takes
    7 N-tiles of 224 columns, 12 K-blocks of 128 columns in 3 stages and CTA
    pairs; over a sweep of shapes every plan covers the product with no
    empty tile, has at least two stages, fits in shared memory, and pairs
    CTAs exactly when there are two M-blocks or more."""
    assert ss.ss_testing_proj_gemm_describe_plan(32768, 1536, 1568) == \
        (224, 7, 128, 12, 3, 1, 896, 201728)
    for M in (1, 100, 128, 129, 256, 300, 32768, 1000003):
        for K in (8, 40, 64, 72, 128, 1536, 4096):
            for Nout in (8, 50, 224, 256, 257, 1568, 4096, 5000):
                BN, nt, kc, kb, stages, pair, units, smem = \
                    ss.ss_testing_proj_gemm_describe_plan(M, K, Nout)
                assert BN % 32 == 0 and 32 <= BN <= 256
                assert nt * BN >= Nout and (nt - 1) * BN < Nout
                assert kb * kc >= K and (kb - 1) * kc < K
                assert 2 <= stages <= 8
                assert smem <= 224 * 1024
                m_tiles = -(-M // 128)
                assert pair == (1 if m_tiles >= 2 else 0)
                assert units == (-(-m_tiles // 2) if pair else m_tiles) * nt
    assert ss.ss_testing_proj_gemm_describe_plan(0, 64, 64) is None
    assert ss.ss_testing_proj_gemm_describe_plan(64, -1, 64) is None


def test_projection_gemm_extent_limit(L):
    """Tile coordinates are 32-bit: extents up to 2^31 - 256 plan, larger ones
    are refused."""
    assert ss.ss_testing_proj_gemm_describe_plan(2**31 - 256, 64, 64) is not None
    assert ss.ss_testing_proj_gemm_describe_plan(2**31 - 255, 64, 64) is None
    assert ss.ss_testing_proj_gemm_describe_plan(64, 2**31 - 255, 64) is None
    assert ss.ss_testing_proj_gemm_describe_plan(64, 64, 2**31 - 255) is None
