"""ss_affine_scan_noalloc, the affine scan for callers that cannot allocate
device memory (code running where cudaMalloc is not allowed or not safe,
such as inside an allocator or a plugin that must leave the device heap
alone). Its scratch is a static array inside the library instead of a
caller-provided workspace.

Called through the C ABI and checked against the regular entry point
(ss_affine_scan with a workspace) on two calls in a row, so the second call
runs on scratch the first one left behind. This file is named to be
collected last: if it fails, a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

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
        torch.cuda.synchronize()
        got, want = h.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: unwritten outputs"
        assert rel_err(got, want) <= TOL, f"call {call}"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    require_gpu()
    import linear_recurrences_gb300 as ss
    lib = ss.lib()
    p = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    assert lib.ss_affine_scan_noalloc(p, p, p, ss.SS_AFFINE_NOALLOC_MAX_N + 1, None) == \
        ss.SS_ERR_UNSUPPORTED
    assert lib.ss_affine_scan_noalloc(p, p, p, -1, None) == ss.SS_ERR_INVALID
    assert lib.ss_affine_scan_noalloc(p, p, p, 0, None) == ss.SS_OK
