"""GPU affine scan vs the float64 oracle (parity, exactness, determinism)."""
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
    h = ss.ss_affine_scan(torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev))
    return h.cpu().numpy()


def test_workload_affine_small(torch, ss):
    w = workloads.AFFINE["affine_small"]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    assert rel_err(run(ss, torch, a, b), oracle.affine(a, b)) <= TOL


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 127, 128, 129, 511, 513, TILE - 1, TILE, TILE + 1,
                               3 * TILE + 7, 257 * TILE + 1, 1000 * TILE + 999])
def test_sizes(torch, ss, n):
    a, b = workloads.affine_inputs(n, 0.5, 1.0, seed=n)
    assert rel_err(run(ss, torch, a, b), oracle.affine(a, b)) <= TOL


def test_ones_give_exact_prefix_sums(torch, ss):
    n = 5 * TILE + 123
    g = np.random.Generator(np.random.PCG64(7))
    b = g.integers(-8, 9, size=n).astype(np.float32)
    h = run(ss, torch, np.ones(n, np.float32), b)
    assert np.array_equal(h.astype(np.float64), np.cumsum(b.astype(np.int64)).astype(np.float64))


def test_zeros_give_b(torch, ss):
    n = 3 * TILE + 5
    _, b = workloads.affine_inputs(n, 0.0, 1.0, seed=3)
    h = run(ss, torch, np.zeros(n, np.float32), b)
    assert np.array_equal(h, b)


@pytest.mark.parametrize("a0", [0.5, 0.9, 0.999])
def test_constant_a_geometric(torch, ss, a0):
    n = 4 * TILE + 9
    a32 = np.float32(a0)
    h = run(ss, torch, np.full(n, a32, np.float32), np.ones(n, np.float32))
    t = np.arange(n, dtype=np.float64)
    closed = (1.0 - float(a32) ** (t + 1)) / (1.0 - float(a32))
    assert rel_err(h, closed) <= TOL


def test_unaligned_pointers(torch, ss):
    """Inputs and output at a 4-byte offset take the plain-load / scalar-store path."""
    n = 2 * TILE + 50
    a, b = workloads.affine_inputs(n + 1, 0.5, 1.0, seed=11)
    dev = torch.device("cuda:0")
    ta = torch.from_numpy(a).to(dev)[1:]
    tb = torch.from_numpy(b).to(dev)[1:]
    out = torch.zeros(n + 1, device=dev)[1:]
    ss.ss_affine_scan(ta, tb, out)
    assert rel_err(out.cpu().numpy(), oracle.affine(a[1:].copy(), b[1:].copy())) <= TOL


def test_large_workload_full_compare(torch, ss):
    """affine_large (n = 2**28), in the configuration the benchmark times."""
    w = workloads.AFFINE["affine_large"]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    h = run(ss, torch, a, b)
    ref = oracle.affine(a, b)
    assert rel_err(h, ref) <= TOL


def test_determinism_1000_runs(torch, ss):
    w = workloads.AFFINE["affine_small"]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    dev = torch.device("cuda:0")
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    first = ss.ss_affine_scan(ta, tb).clone()
    out = torch.empty_like(first)
    for _ in range(1000):
        ss.ss_affine_scan(ta, tb, out)
        assert torch.equal(out, first)


def test_determinism_large_1000_runs(torch, ss):
    """affine_large (n = 2**28) in the benchmark's launch configuration: 1000
    calls, each bitwise equal to the first (the look-back order of the carries
    must not depend on which tile finishes first)."""
    w = workloads.AFFINE["affine_large"]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    dev = torch.device("cuda:0")
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    del a, b
    first = ss.ss_affine_scan(ta, tb).clone()
    out = torch.empty_like(first)
    for _ in range(1000):
        ss.ss_affine_scan(ta, tb, out)
        assert torch.equal(out, first)


def test_timeout_is_reported_not_hung(torch, ss):
    """Tile 5 skips publishing; tile 6's bounded wait runs out, the kernel
    finishes, the host reads SS_ERR_TIMEOUT, and the next call is clean."""
    n = 64 * TILE
    a, b = workloads.affine_inputs(n, 0.5, 1.0, seed=13)
    dev = torch.device("cuda:0")
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    ws = ss.new_workspace(ss.ss_affine_scan_workspace_bytes(n), dev)
    out = torch.empty_like(ta)
    try:
        ss.ss_set_spin_timeout_ns(5_000_000)
        ss.ss_testing_skip_publish_once(5)
        ss.ss_affine_scan(ta, tb, out, workspace=ws)
        assert ss.ss_get_device_status(ws) == ss.SS_ERR_TIMEOUT
    finally:
        ss.ss_testing_skip_publish_once(-1)
        ss.ss_set_spin_timeout_ns(1_000_000_000)
    ss.ss_affine_scan(ta, tb, out, workspace=ws)
    assert ss.ss_get_device_status(ws) == ss.SS_OK
    assert rel_err(out.cpu().numpy(), oracle.affine(a, b)) <= TOL
