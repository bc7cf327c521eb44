"""ss_affine_scan_noalloc, the affine scan for callers that cannot allocate
device memory (code running where cudaMalloc is not allowed or not safe,
such as inside an allocator or a plugin that must leave the device heap
alone). Its scratch is a static array inside the library instead of a
caller-provided workspace.

Called through the C ABI and checked on two calls in a row (so the second
call runs on scratch the first one left behind): bitwise against the regular
entry point (ss_affine_scan with a workspace; the same kernel on the same
tiles, so the results must be identical) and against the float64 oracle.
A look-back wait that runs out is reported by ss_affine_scan_noalloc_status.
This file is named to be collected last: if it fails, a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu

pytestmark = pytest.mark.gpu
TOL = 1e-4


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    torch = require_gpu()
    import linear_recurrences_gb300 as ss
    lib = ss.lib()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    for call, (n, seed) in enumerate([(1_000_003, 41), (ss.SS_AFFINE_NOALLOC_MAX_N, 42)]):
        a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=seed)
        ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
        ref = ss.ss_affine_scan(ta, tb)                      # regular entry point
        h = torch.full_like(ta, float("nan"))
        st = lib.ss_affine_scan_noalloc(_p(ta), _p(tb), _p(h), n, sh)
        assert st == ss.SS_OK, f"call {call}: {ss.ss_status_string(st)}"
        assert lib.ss_affine_scan_noalloc_status(sh) == ss.SS_OK, f"call {call}"
        got, want = h.cpu().numpy(), ref.cpu().numpy()
        assert np.array_equal(got, want), f"call {call}: differs from ss_affine_scan"
        assert rel_err(got, oracle.affine(a, b)) <= TOL, f"call {call}"


def test_noalloc_reports_a_wait_that_ran_out():
    """Tile 3 skips publishing for one call: the waits on it give up after a
    5 ms spin limit, the status call returns SS_ERR_TIMEOUT, and the next call
    is clean and exact again."""
    torch = require_gpu()
    import linear_recurrences_gb300 as ss
    lib = ss.lib()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    n = 50 * 4096 + 17
    a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=43)
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    h = torch.empty_like(ta)
    try:
        ss.ss_set_spin_timeout_ns(5_000_000)
        ss.ss_testing_skip_publish_once(3)
        assert lib.ss_affine_scan_noalloc(_p(ta), _p(tb), _p(h), n, sh) == ss.SS_OK
        assert lib.ss_affine_scan_noalloc_status(sh) == ss.SS_ERR_TIMEOUT
    finally:
        ss.ss_testing_skip_publish_once(-1)
        ss.ss_set_spin_timeout_ns(1_000_000_000)
    assert lib.ss_affine_scan_noalloc(_p(ta), _p(tb), _p(h), n, sh) == ss.SS_OK
    assert lib.ss_affine_scan_noalloc_status(sh) == ss.SS_OK
    assert np.array_equal(h.cpu().numpy(), ss.ss_affine_scan(ta, tb).cpu().numpy())


def test_noalloc_refuses_sizes_beyond_its_scratch():
    require_gpu()
    import linear_recurrences_gb300 as ss
    lib = ss.lib()
    p = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    assert lib.ss_affine_scan_noalloc(p, p, p, ss.SS_AFFINE_NOALLOC_MAX_N + 1, None) == \
        ss.SS_ERR_UNSUPPORTED
    assert lib.ss_affine_scan_noalloc(p, p, p, -1, None) == ss.SS_ERR_INVALID
    assert lib.ss_affine_scan_noalloc(p, p, p, 0, None) == ss.SS_OK
