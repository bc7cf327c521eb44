"""GPU affine scan with log-step (Hillis-Steele) tiles vs the float64 oracle.

The comparison kernel runs the same staging, look-back and fix-up as the
production affine scan; only the scan inside each 4096-element tile differs.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu

pytestmark = pytest.mark.gpu
TOL = 1e-4
TILE = 4096


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m


def run(ss, torch, a, b):
    dev = torch.device("cuda:0")
    h = ss.ss_affine_scan_log_step(torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev))
    return h.cpu().numpy()


@pytest.mark.parametrize("n", [1, 2, 3, 5, 17, 31, 33, 129, 513, TILE - 1, TILE, TILE + 1,
                               3 * TILE + 7, 257 * TILE + 1])
def test_sizes(torch, ss, n):
    a, b = workloads.affine_inputs(n, 0.5, 1.0, seed=n + 1)
    assert rel_err(run(ss, torch, a, b), oracle.affine(a, b)) <= TOL


def test_ones_give_exact_prefix_sums(torch, ss):
    """a == 1, small integer b: every partial sum is an exact fp32 integer,
    so any association order gives the exact prefix sums."""
    n = 5 * TILE + 123
    g = np.random.Generator(np.random.PCG64(3))
    a = np.ones(n, np.float32)
    b = g.integers(-8, 9, n).astype(np.float32)
    assert np.array_equal(run(ss, torch, a, b), np.cumsum(b.astype(np.float64)))


def test_large_workload(torch, ss):
    w = workloads.AFFINE["affine_large"]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    assert rel_err(run(ss, torch, a, b), oracle.affine(a, b)) <= TOL


def test_deterministic(torch, ss):
    a, b = workloads.affine_inputs(300 * TILE + 5, 0.9, 1.0, seed=4)
    dev = torch.device("cuda:0")
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    first = ss.ss_affine_scan_log_step(ta, tb).clone()
    out = torch.empty_like(first)
    for _ in range(100):
        ss.ss_affine_scan_log_step(ta, tb, out)
        assert torch.equal(out, first)
