"""GPU S6 forward from an initial state, with the final state returned, vs
the float64 oracle; and a sequence streamed in pieces."""
import os

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu, to_dev, to_host_f64

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 2e-2}
TOL_STATE = {"f32": 1e-4, "bf16": 1e-3}  # h_last is fp32 for both storage types
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m


@pytest.fixture
def plan_override(ss):
    """Forces a plan for one test through the library's test hook: (wt, tsub)
    for the chunked kernel, ("tp", G, T, W) for the time-parallel pass, None
    for the planner's own choice."""
    def set_(wt, tsub=0, *rest):
        if wt is None:
            ss.ss_testing_s6_plan(0)
        elif wt == "tp":
            ss.ss_testing_s6_plan(2, tsub, *rest)
        else:
            ss.ss_testing_s6_plan(1, wt, tsub, 1)
    yield set_
    ss.ss_testing_s6_plan(0)


def inputs(B, L, D, N, io="f32", softplus=False, seed=0):
    inp = workloads.s6_inputs(B, L, D, N, io=io, delta="preact" if softplus else "loguniform",
                              dskip="normal", seed=seed)
    g = np.random.Generator(np.random.PCG64(seed + 500))
    inp.A = (-g.uniform(0.1, 4.0, (D, N))).astype(np.float32)
    h0 = g.standard_normal((B, D, N)).astype(np.float32)
    return inp, h0


def gpu_state(ss, torch, inp, h0, softplus, t0=0, t1=None):
    """Runs steps [t0, t1) from h0 on a fresh workspace; returns (y, h_last)
    on the host and checks the device status word."""
    dev = torch.device("cuda:0")
    sl = lambda v: np.ascontiguousarray(v[:, t0:t1])
    t = lambda v: to_dev(v, dev, inp.io)
    x, dl, Bt, Ct = (t(sl(v)) for v in (inp.x, inp.delta, inp.Bt, inp.Ct))
    B, L, D = x.shape
    N = inp.A.shape[1]
    io = ss.SS_BF16 if inp.io == "bf16" else ss.SS_F32
    nbytes = ss.ss_selective_scan_workspace_bytes(B, L, D, N, io, False)
    ws = ss.new_workspace(nbytes, dev) if nbytes else None
    h0d = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, np.float32)).to(dev)
    y, hl = ss.ss_selective_scan_fwd_state(x, dl, Bt, Ct, to_dev(inp.A, dev), to_dev(inp.Dskip, dev),
                                           h0=h0d, delta_softplus=softplus, workspace=ws)
    if ws is not None:
        assert ss.ss_get_device_status(ws) == ss.SS_OK
    return to_host_f64(y), hl.double().cpu().numpy()


def oracle_state(inp, h0, softplus, t0=0, t1=None):
    sl = lambda v: np.ascontiguousarray(v[:, t0:t1])
    return oracle.s6_fwd_state(sl(inp.x_f32), sl(inp.delta_f32), sl(inp.Bt_f32), sl(inp.Ct_f32),
                               inp.A, inp.Dskip, h0=h0, softplus=softplus, threads=THREADS)


SHAPES = [(1, 1, 1, 1), (2, 5, 3, 4), (1, 40, 32, 16), (2, 100, 33, 16), (3, 257, 40, 3),
          (2, 600, 64, 16)]
# default, chunked, unsplit multi-warp, time-parallel (channels/warp, steps/lane, warps/CTA)
PLANS = [None, (1, 8), (2, 16), (4, 5), (2, 1024), ("tp", 2, 9, 4), ("tp", 4, 9, 2),
         ("tp", 8, 9, 2)]


@pytest.mark.parametrize("plan", PLANS,
                         ids=lambda p: "default" if p is None else "x".join(map(str, p)))
@pytest.mark.parametrize("io,softplus", [("f32", False), ("bf16", True)])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_state_parity(torch, ss, plan_override, shape, io, softplus, plan):
    inp, h0 = inputs(*shape, io=io, softplus=softplus, seed=sum(shape))
    plan_override(*(plan or (None, None)))
    y, hl = gpu_state(ss, torch, inp, h0, softplus)
    ry, rhl = oracle_state(inp, h0.astype(np.float64), softplus)
    assert rel_err(y, ry) <= TOL[io]
    assert rel_err(hl, rhl) <= TOL_STATE[io]


def test_no_initial_state_is_the_plain_forward(torch, ss):
    inp, _ = inputs(2, 300, 48, 16, seed=3)
    y, hl = gpu_state(ss, torch, inp, None, False)
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev)
    y2 = ss.ss_selective_scan_fwd(t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A),
                                  t(inp.Dskip))
    assert np.array_equal(y, to_host_f64(y2)), "h0 = None must match ss_selective_scan_fwd bitwise"
    ry, rhl = oracle_state(inp, None, False)
    assert rel_err(hl, rhl) <= TOL_STATE["f32"]


@pytest.mark.parametrize("io,softplus", [("f32", False), ("bf16", True)])
def test_streamed_in_pieces(torch, ss, plan_override, io, softplus):
    """[0, L) run as three calls, each starting from the previous call's
    final state, matches the oracle's single run."""
    inp, h0 = inputs(2, 900, 70, 16, io=io, softplus=softplus, seed=11)
    cuts = [0, 1, 433, 900]
    ys, h = [], h0
    for i, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        plan_override(*[(None, None), (1, 8), ("tp", 4, 9, 2)][i])
        y, h = gpu_state(ss, torch, inp, h, softplus, a, b)
        ys.append(y)
    ry, rhl = oracle_state(inp, h0.astype(np.float64), softplus)
    assert rel_err(np.concatenate(ys, axis=1), ry) <= TOL[io]
    assert rel_err(h, rhl) <= TOL_STATE[io]


def test_state_workload_full(torch, ss):
    """The fp32 S6 workload (B16 L2048 D256 N16) in the default plan, from a
    random h0: every y and every final state compared."""
    w = workloads.S6["s6_fp32"]
    inp = workloads.s6_workload_inputs(w)
    h0 = np.random.Generator(np.random.PCG64(7)).standard_normal((w.B, w.D, w.N)).astype(np.float32)
    y, hl = gpu_state(ss, torch, inp, h0, w.softplus)
    ry, rhl = oracle_state(inp, h0.astype(np.float64), w.softplus)
    assert rel_err(y, ry) <= TOL["f32"]
    assert rel_err(hl, rhl) <= TOL_STATE["f32"]


def test_state_workload_bf16_first_batch(torch, ss):
    """The bf16 S6 workload (B8 L4096 D1536 N16, softplus) from a random h0, in
    the benchmark's configuration; batch element 0 (which depends on nothing
    else) compared in full, y and h_last."""
    w = workloads.S6["s6_bf16"]
    inp = workloads.s6_workload_inputs(w)
    h0 = np.random.Generator(np.random.PCG64(7)).standard_normal((w.B, w.D, w.N)).astype(np.float32)
    y, hl = gpu_state(ss, torch, inp, h0, w.softplus)
    one = lambda v: np.ascontiguousarray(v[:1])
    ry, rhl = oracle.s6_fwd_state(one(inp.x_f32), one(inp.delta_f32), one(inp.Bt_f32),
                                  one(inp.Ct_f32), inp.A, inp.Dskip, h0=h0[:1].astype(np.float64),
                                  softplus=True, threads=THREADS)
    assert rel_err(y[:1], ry) <= TOL["bf16"]
    assert rel_err(hl[:1], rhl) <= TOL_STATE["bf16"]
