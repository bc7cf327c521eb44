"""GPU S6 forward and bidirectional scans vs the float64 oracle."""
import os

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu, to_dev, to_host_f64

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 2e-2}
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
    """Forces the chunked kernel with (warps per CTA, timesteps per warp, lanes
    per channel) for one test, through the library's test hook."""
    def set_(wt, tsub, lpc=1):
        ss.ss_testing_s6_plan(1, wt, tsub, lpc)
    yield set_
    ss.ss_testing_s6_plan(0)


def gpu_run(ss, torch, inp, softplus, bidir):
    """Runs the scan on a fresh workspace and checks that the device reported
    no error (a look-back that ran out of time would otherwise only show up
    as wrong numbers)."""
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev, inp.io)
    fn = ss.ss_selective_scan_bidir if bidir else ss.ss_selective_scan_fwd
    B, L, D = inp.x.shape
    N = inp.Bt.shape[-1]
    io = ss.SS_BF16 if inp.io == "bf16" else ss.SS_F32
    nbytes = ss.ss_selective_scan_workspace_bytes(B, L, D, N, io, bidir)
    ws = ss.new_workspace(nbytes, dev) if nbytes else None
    y = fn(t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A), t(inp.Dskip),
           delta_softplus=softplus, workspace=ws)
    if ws is not None:
        assert ss.ss_get_device_status(ws) == ss.SS_OK
    return to_host_f64(y)


def oracle_run(inp, softplus, bidir):
    f = oracle.s6_bidir if bidir else oracle.s6_fwd
    return f(inp.x_f32, inp.delta_f32, inp.Bt_f32, inp.Ct_f32, inp.A, inp.Dskip,
             softplus=softplus, threads=THREADS)


def small(B, L, D, N, io="f32", softplus=False, seed=0, A_random=True):
    inp = workloads.s6_inputs(B, L, D, N, io=io, delta="preact" if softplus else "loguniform",
                              dskip="normal", seed=seed)
    if A_random:  # d- and n-dependent A so a transposed index cannot hide
        g = np.random.Generator(np.random.PCG64(seed + 100))
        inp.A = (-g.uniform(0.1, 4.0, (D, N))).astype(np.float32)
    return inp


SHAPES = [
    # (B, L, D, N)
    (1, 1, 1, 1),
    (2, 2, 3, 4),
    (1, 33, 32, 16),
    (2, 64, 33, 16),
    (3, 100, 64, 8),
    (2, 257, 40, 3),
    (1, 1000, 96, 16),
    (4, 513, 31, 5),
]


@pytest.mark.parametrize("bidir", [False, True], ids=["fwd", "bidir"])
@pytest.mark.parametrize("io,softplus", [("f32", False), ("f32", True), ("bf16", True), ("bf16", False)])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(torch, ss, shape, io, softplus, bidir):
    inp = small(*shape, io=io, softplus=softplus, seed=sum(shape))
    y = gpu_run(ss, torch, inp, softplus, bidir)
    ref = oracle_run(inp, softplus, bidir)
    assert rel_err(y, ref) <= TOL[io]


@pytest.mark.parametrize("bidir", [False, True], ids=["fwd", "bidir"])
@pytest.mark.parametrize("wt,tsub", [(1, 3), (1, 7), (2, 8), (3, 5), (4, 4), (4, 33), (4, 64)])
def test_chunk_splits(torch, ss, plan_override, wt, tsub, bidir):
    """Forces many chunks and sub-chunks so the look-back, the look-forward
    and the in-CTA folds run across ragged boundaries."""
    plan_override(wt, tsub)
    inp = small(2, 777, 70, 16, seed=wt * 100 + tsub)
    y = gpu_run(ss, torch, inp, False, bidir)
    assert rel_err(y, oracle_run(inp, False, bidir)) <= TOL["f32"]


@pytest.mark.parametrize("bidir", [False, True], ids=["fwd", "bidir"])
def test_more_chunks_than_one_lookback_window(torch, ss, plan_override, bidir):
    """300 chunks: walks reach past the 128 chunks a look-back examines at
    once, in both directions, and the two directions must not wait on each
    other."""
    plan_override(1, 2)
    inp = small(1, 600, 40, 16, seed=77)
    y = gpu_run(ss, torch, inp, False, bidir)
    assert rel_err(y, oracle_run(inp, False, bidir)) <= TOL["f32"]


def test_forward_with_one_step_chunks(torch, ss, plan_override):
    """777 chunks of one timestep each: the look-back walks several windows."""
    plan_override(1, 1)
    inp = small(2, 777, 70, 16, seed=101)
    y = gpu_run(ss, torch, inp, False, False)
    assert rel_err(y, oracle_run(inp, False, False)) <= TOL["f32"]


def test_bidir_refuses_more_chunks_than_fit(torch, ss, plan_override):
    """Every chunk of a bidirectional sequence must be resident at once; a
    plan that cannot be is refused up front instead of risking a stall."""
    plan_override(1, 1)
    inp = small(1, 20000, 32, 16, seed=3)
    with pytest.raises(ss.SSError) as e:
        gpu_run(ss, torch, inp, False, True)
    assert e.value.status == ss.SS_ERR_UNSUPPORTED


def test_chunked_bf16_softplus(torch, ss, plan_override):
    plan_override(4, 16)
    inp = small(3, 1500, 48, 16, io="bf16", softplus=True, seed=5)
    for bidir in (False, True):
        y = gpu_run(ss, torch, inp, True, bidir)
        assert rel_err(y, oracle_run(inp, True, bidir)) <= TOL["bf16"]


def test_null_dskip(torch, ss):
    inp = small(2, 50, 16, 16, seed=9)
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev)
    y = ss.ss_selective_scan_fwd(t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A), None)
    ref = oracle.s6_fwd(inp.x_f32, inp.delta_f32, inp.Bt_f32, inp.Ct_f32, inp.A, None)
    assert rel_err(to_host_f64(y), ref) <= TOL["f32"]


# ---------------------------------------------------------------- workloads
def _sample_channels(B, D, count, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    chans = np.unique(np.concatenate([[0, B * D - 1, D - 1, D], g.integers(0, B * D, count)]))
    return chans[chans < B * D]


@pytest.mark.parametrize("name", ["s6_fp32", "s6_bf16", "s6_bidir"])
def test_workload(torch, ss, name):
    """Each S6 workload at full size, in the benchmark's launch configuration
    (the library's own plan choice): every output element of every channel
    against the oracle."""
    w = workloads.S6[name]
    inp = workloads.s6_workload_inputs(w)
    y = gpu_run(ss, torch, inp, w.softplus, w.bidir)
    ref = oracle_run(inp, w.softplus, w.bidir)
    assert y.shape == ref.shape
    assert rel_err(y, ref) <= TOL[w.io]


@pytest.mark.parametrize("name", ["s6_fp32", "s6_bf16", "s6_bidir"])
def test_workload_determinism_1000_runs(torch, ss, name):
    w = workloads.S6[name]
    inp = workloads.s6_workload_inputs(w)
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev, inp.io)
    args = (t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A), t(inp.Dskip))
    fn = ss.ss_selective_scan_bidir if w.bidir else ss.ss_selective_scan_fwd
    first = fn(*args, delta_softplus=w.softplus).clone()
    out = torch.empty_like(first)
    for _ in range(1000):
        fn(*args, delta_softplus=w.softplus, y=out)
        assert torch.equal(out, first)


@pytest.mark.parametrize("bidir", [False, True], ids=["fwd", "bidir"])
def test_timeout_is_reported_not_hung(torch, ss, plan_override, bidir):
    """One chunk skips publishing; the bounded waits on it run out, the host
    reads SS_ERR_TIMEOUT, and the next call on the same workspace is clean."""
    plan_override(2, 16)
    inp = small(2, 640, 64, 16, seed=21)
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev)
    args = (t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A), t(inp.Dskip))
    fn = ss.ss_selective_scan_bidir if bidir else ss.ss_selective_scan_fwd
    B, L, D, N = 2, 640, 64, 16
    ws = ss.new_workspace(ss.ss_selective_scan_workspace_bytes(B, L, D, N, ss.SS_F32, bidir), dev)
    out = torch.empty_like(args[0])
    try:
        ss.ss_set_spin_timeout_ns(5_000_000)
        ss.ss_testing_skip_publish_once(7)
        fn(*args, y=out, workspace=ws)
        assert ss.ss_get_device_status(ws) == ss.SS_ERR_TIMEOUT
    finally:
        ss.ss_testing_skip_publish_once(-1)
        ss.ss_set_spin_timeout_ns(1_000_000_000)
    fn(*args, y=out, workspace=ws)
    assert ss.ss_get_device_status(ws) == ss.SS_OK
    assert rel_err(to_host_f64(out), oracle_run(inp, False, bidir)) <= TOL["f32"]


@pytest.mark.parametrize("lpc", [1, 2, 4])
@pytest.mark.parametrize("bidir", [False, True], ids=["fwd", "bidir"])
@pytest.mark.parametrize("io,softplus", [("f32", False), ("bf16", True)])
def test_both_lane_layouts(torch, ss, plan_override, lpc, bidir, io, softplus):
    """The chunked kernel with 16 states per lane, or 8 / 4 states on each of
    two / four lanes per channel: under its planner's own split of L and a
    forced split of 2 warps x 24 steps."""
    for wt_tsub in ((0, 0), (2, 24)):
        plan_override(*wt_tsub, lpc)
        inp = small(2, 333, 70, 16, io=io, softplus=softplus, seed=7 + lpc)
        y = gpu_run(ss, torch, inp, softplus, bidir)
        assert rel_err(y, oracle_run(inp, softplus, bidir)) <= TOL[io]


@pytest.mark.parametrize("bidir", [False, True], ids=["fwd", "bidir"])
@pytest.mark.parametrize("io,softplus", [("f32", False), ("bf16", True)])
def test_register_path_long_sequence(torch, ss, plan_override, bidir, io, softplus):
    """The chunked kernel's register path: one warp per 32 channels runs all
    of a 3000-step sequence (one chunk, one warp per CTA), forced by plan."""
    L = 3000
    plan_override(1, L)
    B, D, N = 2, 70, 16
    kind, prm = ss.ss_testing_s6_describe_plan(B, L, D, N, ss.SS_BF16 if io == "bf16" else ss.SS_F32,
                                               bidir)
    assert kind == 0 and prm[1] == 1 and prm[3] == 1  # one warp per CTA, one chunk
    inp = small(B, L, D, N, io=io, softplus=softplus, seed=31)
    y = gpu_run(ss, torch, inp, softplus, bidir)
    assert rel_err(y, oracle_run(inp, softplus, bidir)) <= TOL[io]


def test_register_path_chosen_for_many_channels(torch, ss):
    """A bidirectional shape with B*D large enough to fill the chip with one
    warp per 32 channels takes the register path by itself (L = 1024, 80,000
    channels); sampled channels against the oracle."""
    B, L, D, N = 1, 1024, 80000, 16
    kind, prm = ss.ss_testing_s6_describe_plan(B, L, D, N, ss.SS_F32, True)
    assert kind == 0 and prm[1] == 1 and prm[3] == 1
    inp = workloads.s6_inputs(B, L, D, N, io="f32", delta="loguniform", dskip="normal", seed=41)
    y = gpu_run(ss, torch, inp, False, True)
    chans = _sample_channels(B, D, 200, seed=2)
    ref = oracle.s6_channels(inp.x_f32, inp.delta_f32, inp.Bt_f32, inp.Ct_f32, inp.A, inp.Dskip,
                             chans, softplus=False, bidir=True, threads=THREADS)
    got = np.stack([y[c // D, :, c % D] for c in chans])
    assert rel_err(got, ref) <= TOL["f32"]
