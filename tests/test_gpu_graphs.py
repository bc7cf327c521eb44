"""The library's calls captured in CUDA graphs: replays give the results of
direct calls, bitwise, and leave the workspaces ready (no device error)."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m


def test_affine_scan_graph_replays(torch, ss):
    dev = torch.device("cuda:0")
    n = 37 * 4096 + 11
    a, b = workloads.affine_inputs(n, 0.9, 1.0, seed=51)
    ta, tb = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    h = torch.empty_like(ta)
    ws = ss.new_workspace(ss.ss_affine_scan_workspace_bytes(n), dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first call outside the capture (lazy init)
        ss.ss_affine_scan(ta, tb, h, workspace=ws, stream=s)
    s.synchronize()
    direct = h.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ss.ss_affine_scan(ta, tb, h, workspace=ws, stream=s)
    for _ in range(5):
        h.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(h, direct)
    assert ss.ss_get_device_status(ws) == ss.SS_OK
    assert rel_err(h.cpu().numpy(), oracle.affine(a, b)) <= 1e-4


def test_selective_scan_graph_replays(torch, ss):
    dev = torch.device("cuda:0")
    inp = workloads.s6_inputs(2, 700, 96, 16, io="f32", seed=53)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    args = (t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A), t(inp.Dskip))
    y = torch.empty_like(args[0])
    ws = ss.new_workspace(ss.ss_selective_scan_workspace_bytes(2, 700, 96, 16, ss.SS_F32), dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ss.ss_selective_scan_fwd(*args, y=y, workspace=ws, stream=s)
    s.synchronize()
    direct = y.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ss.ss_selective_scan_fwd(*args, y=y, workspace=ws, stream=s)
    for _ in range(5):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, direct)
    assert ss.ss_get_device_status(ws) == ss.SS_OK


def test_backward_graph_replays(torch, ss):
    dev = torch.device("cuda:0")
    inp = workloads.s6_inputs(2, 600, 40, 16, io="f32", delta="preact", seed=57)
    g0 = np.random.Generator(np.random.PCG64(58))
    dy = g0.standard_normal((2, 600, 40)).astype(np.float32)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    args = (t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A), t(inp.Dskip), t(dy))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ref = ss.ss_selective_scan_bwd(*args, delta_softplus=True, stream=s)
    s.synchronize()
    ref = {k: v.clone() for k, v in ref.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out = ss.ss_selective_scan_bwd(*args, delta_softplus=True, stream=s)
    for _ in range(3):
        for v in out.values():
            v.zero_()
        g.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(out[k], ref[k]), f"{k} differs on replay"
