"""GPU wavefront single-pass S6 forward (every built launch shape) vs the
float64 oracle, element by element."""
import os

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu, to_dev, to_host_f64

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 2e-2}
TOL_STATE = {"f32": 1e-4, "bf16": 1e-3}
THREADS = os.cpu_count() or 1

# (steps per warp slice T, slices per CTA S); a block is S * T steps of 32 channels
VARIANTS = [(9, 4), (11, 4), (13, 4), (15, 4), (9, 2), (13, 2)]


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m


@pytest.fixture
def ws_plan(ss):
    def set_(T, S):
        ss.ss_testing_s6_plan(3, T, S)
    yield set_
    ss.ss_testing_s6_plan(0)


def inputs(B, L, D, N, io, softplus, seed):
    inp = workloads.s6_inputs(B, L, D, N, io=io, delta="preact" if softplus else "loguniform",
                              dskip="normal", seed=seed)
    g = np.random.Generator(np.random.PCG64(seed + 100))
    inp.A = (-g.uniform(0.1, 4.0, (D, N))).astype(np.float32)  # d- and n-dependent
    return inp


def run(ss, torch, inp, softplus, h0=None):
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev, inp.io)
    B, L, D = inp.x.shape
    N = inp.A.shape[1]
    io = ss.SS_BF16 if inp.io == "bf16" else ss.SS_F32
    ws = ss.new_workspace(ss.ss_selective_scan_workspace_bytes(B, L, D, N, io, False), dev)
    h0d = None if h0 is None else torch.from_numpy(h0).to(dev)
    y, hl = ss.ss_selective_scan_fwd_state(t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct),
                                           to_dev(inp.A, dev), to_dev(inp.Dskip, dev), h0=h0d,
                                           delta_softplus=softplus, workspace=ws)
    assert ss.ss_get_device_status(ws) == ss.SS_OK
    return to_host_f64(y), hl.double().cpu().numpy()


def check(ss, torch, inp, softplus, with_h0, seed):
    B, L, D = inp.x.shape
    N = inp.A.shape[1]
    h0 = None
    if with_h0:
        h0 = np.random.Generator(np.random.PCG64(seed + 7)).standard_normal((B, D, N))
        h0 = h0.astype(np.float32)
    y, hl = run(ss, torch, inp, softplus, h0)
    ry, rhl = oracle.s6_fwd_state(inp.x_f32, inp.delta_f32, inp.Bt_f32, inp.Ct_f32, inp.A,
                                  inp.Dskip, h0=None if h0 is None else h0.astype(np.float64),
                                  softplus=softplus, threads=THREADS)
    assert rel_err(y, ry) <= TOL[inp.io]
    assert rel_err(hl, rhl) <= TOL_STATE[inp.io]


# one step; a ragged single block; several blocks with a ragged tail;
# channels not filling the CTA's 32; odd N; N = 1; more than one CTA
SHAPES = [(1, 1, 8, 16), (2, 37, 16, 16), (2, 700, 40, 16), (3, 333, 24, 5), (1, 1000, 8, 1),
          (2, 290, 64, 13), (1, 2000, 96, 16)]


@pytest.mark.parametrize("io,softplus", [("f32", False), ("f32", True), ("bf16", True),
                                         ("bf16", False)])
@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "T{}S{}".format(*v))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_variant_parity(torch, ss, ws_plan, shape, variant, io, softplus):
    B, L, D, N = shape
    es = 2 if io == "bf16" else 4
    if (D * es) % 16:
        pytest.skip("rows of x must be a multiple of 16 bytes for the tile copies")
    ws_plan(*variant)
    kind, prm = ss.ss_testing_s6_describe_plan(B, L, D, N, ss.SS_BF16 if io == "bf16" else ss.SS_F32)
    assert kind == 2 and prm[:2] == variant
    seed = sum(shape) + 10 * variant[0] + variant[1]
    inp = inputs(*shape, io=io, softplus=softplus, seed=seed)
    check(ss, torch, inp, softplus, with_h0=(seed % 2 == 0), seed=seed)


@pytest.mark.parametrize("name", ["s6_fp32", "s6_bf16"])
def test_workload_every_element(torch, ss, ws_plan, name):
    """The fp32 and bf16 forward workloads at full size through the wavefront
    pass: every output element against the oracle."""
    ws_plan(13, 4)
    w = workloads.S6[name]
    io = ss.SS_BF16 if w.io == "bf16" else ss.SS_F32
    kind, prm = ss.ss_testing_s6_describe_plan(w.B, w.L, w.D, w.N, io)
    assert kind == 2 and prm[:2] == (13, 4)
    inp = workloads.s6_workload_inputs(w)
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev, inp.io)
    y = ss.ss_selective_scan_fwd(t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A),
                                 t(inp.Dskip), delta_softplus=w.softplus)
    ref = oracle.s6_fwd(inp.x_f32, inp.delta_f32, inp.Bt_f32, inp.Ct_f32, inp.A, inp.Dskip,
                        softplus=w.softplus, threads=THREADS)
    assert rel_err(to_host_f64(y), ref) <= TOL[w.io]


def test_unaligned_rows_fall_back(torch, ss, ws_plan):
    """D = 37 fp32 rows are not 16-byte multiples: the call takes the chunked
    kernel and stays correct."""
    ws_plan(11, 4)
    inp = inputs(2, 300, 37, 16, "f32", False, seed=5)
    check(ss, torch, inp, False, with_h0=True, seed=5)


def test_determinism_small(torch, ss, ws_plan):
    """Repeated calls are bitwise identical."""
    ws_plan(11, 4)
    inp = inputs(2, 1500, 64, 16, "f32", True, seed=3)
    a, _ = run(ss, torch, inp, True)
    for _ in range(20):
        b, _ = run(ss, torch, inp, True)
        assert np.array_equal(a, b)
