"""GPU affine scan from an initial state, and over host buffers, vs the
float64 oracle."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu

pytestmark = pytest.mark.gpu
TOL = 1e-4
TILE = 4096
CHUNK = 1 << 23  # elements per chunk of the host pipeline


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m


def dev(torch, v):
    return torch.from_numpy(np.ascontiguousarray(v)).to("cuda:0")


@pytest.mark.parametrize("n", [1, 2, 33, TILE - 1, TILE, TILE + 1, 3 * TILE + 7, 257 * TILE + 1,
                               1000 * TILE + 999])
def test_state_sizes(torch, ss, n):
    a, b = workloads.affine_inputs(n, 0.5, 1.0, seed=n + 11)
    h0 = np.float32(np.random.Generator(np.random.PCG64(n)).normal(0.0, 4.0))
    h = ss.ss_affine_scan_state(dev(torch, a), dev(torch, b), dev(torch, np.array([h0])))
    assert rel_err(h.cpu().numpy(), oracle.affine(a, b, h0=float(h0))) <= TOL


def test_state_with_no_h0_is_the_plain_scan(torch, ss):
    a, b = workloads.affine_inputs(37 * TILE + 5, 0.9, 1.0, seed=5)
    ta, tb = dev(torch, a), dev(torch, b)
    h1 = ss.ss_affine_scan(ta, tb)
    h2 = ss.ss_affine_scan_state(ta, tb, None)
    assert torch.equal(h1, h2)


def test_state_decay_of_h0_alone(torch, ss):
    """b == 0: h[t] = h0 * prod a[0..t]; with a == 1/2 every value is exact."""
    n = 50 * TILE + 3
    a = np.full(n, 0.5, np.float32)
    a[100:] = 1.0  # 3 * 2^-100 stays a normal fp32 value; every step exact
    h = ss.ss_affine_scan_state(dev(torch, a), dev(torch, np.zeros(n, np.float32)),
                                dev(torch, np.array([3.0], np.float32)))
    assert np.array_equal(h.cpu().numpy().astype(np.float64),
                          oracle.affine(a, np.zeros(n, np.float32), h0=3.0))


def test_state_chained_segments(torch, ss):
    """A sequence scanned as segments, each from the previous segment's last
    output read on the device, matches the oracle on the whole sequence."""
    n = 400 * TILE + 17
    a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=21)
    ta, tb = dev(torch, a), dev(torch, b)
    h = torch.empty_like(ta)
    cuts = [0, 1, 5000, 5001, 70 * TILE, 70 * TILE + 1, 300 * TILE + 3, n]
    last = None
    for s, e in zip(cuts[:-1], cuts[1:]):
        ss.ss_affine_scan_state(ta[s:e], tb[s:e], last, h=h[s:e])
        last = h[e - 1:e].clone()
    assert rel_err(h.cpu().numpy(), oracle.affine(a, b)) <= TOL


def test_state_deterministic(torch, ss):
    a, b = workloads.affine_inputs(600 * TILE + 9, 0.9, 1.0, seed=31)
    ta, tb = dev(torch, a), dev(torch, b)
    h0 = dev(torch, np.array([-7.5], np.float32))
    ref = ss.ss_affine_scan_state(ta, tb, h0)
    for _ in range(20):
        assert torch.equal(ss.ss_affine_scan_state(ta, tb, h0), ref)


def test_state_h0_inside_h_is_rejected(torch, ss):
    ta = dev(torch, np.ones(100, np.float32))
    h = torch.empty_like(ta)
    with pytest.raises(ss.SSError):
        ss.ss_affine_scan_state(ta, ta, h[10:11], h=h)


def host(torch, v, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(v))
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("n", [1, TILE + 1, CHUNK - 1, CHUNK, CHUNK + 1, 3 * CHUNK + 12345,
                               7 * CHUNK + 5])
def test_host_sizes(torch, ss, n):
    a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=n % 1000 + 3)
    h = ss.ss_affine_scan_host(host(torch, a), host(torch, b))
    torch.cuda.current_stream().synchronize()
    assert rel_err(h.numpy(), oracle.affine(a, b)) <= TOL


def test_host_workload_affine_large(torch, ss):
    """The 2^28-element affine workload through host buffers; every 64th
    element against the oracle (all elements are computed by it anyway)."""
    w = workloads.AFFINE["affine_large"]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    h = ss.ss_affine_scan_host(host(torch, a), host(torch, b))
    torch.cuda.current_stream().synchronize()
    ref = oracle.affine(a, b)
    assert rel_err(h.numpy()[::64], ref[::64]) <= TOL
    assert np.isfinite(h.numpy()).all()


def test_host_pageable_buffers(torch, ss):
    """Pageable host memory works too (the driver stages the copies)."""
    n = 2 * CHUNK + 77
    a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=41)
    h = torch.empty(n, dtype=torch.float32)
    ss.ss_affine_scan_host(host(torch, a, False), host(torch, b, False), h=h)
    torch.cuda.current_stream().synchronize()
    assert rel_err(h.numpy(), oracle.affine(a, b)) <= TOL


def test_host_deterministic_and_reusable(torch, ss):
    n = 3 * CHUNK + 1
    a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=43)
    ta, tb = host(torch, a), host(torch, b)
    ws = ss.new_workspace(ss.ss_affine_scan_host_workspace_bytes(n), "cuda:0")
    h1 = ss.ss_affine_scan_host(ta, tb, workspace=ws)
    h2 = ss.ss_affine_scan_host(ta, tb, workspace=ws)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(h1, h2)
    assert ss.ss_get_device_status(ws) == ss.SS_OK


def test_host_orders_after_earlier_stream_work(torch, ss):
    """Inputs written by a copy queued earlier on the same stream are the
    ones the pipeline reads (it starts after the stream's queued work)."""
    n = CHUNK + 3
    a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=47)
    ta, tb = host(torch, np.zeros(n, np.float32)), host(torch, np.zeros(n, np.float32))
    src_a, src_b = dev(torch, a), dev(torch, b)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ta.copy_(src_a, non_blocking=True)
        tb.copy_(src_b, non_blocking=True)
        h = ss.ss_affine_scan_host(ta, tb, stream=s)
    s.synchronize()
    assert rel_err(h.numpy(), oracle.affine(a, b)) <= TOL
