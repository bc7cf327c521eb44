"""GPU S6 backward pass vs the float64 oracle's reverse-mode derivative."""
import os

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu, to_dev, to_host_f64

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
NAMES = ("dx", "ddelta", "dA", "dBt", "dCt", "dDskip", "dh0")
# element-wise: max_i |g_i - ref_i| / max(1, |ref_i|) over each tensor;
# dx and ddelta are stored in the storage type, the rest in fp32. ddelta and
# dA are cancelling sums (ddelta over the 2N terms dh.(A a h) < 0 and
# dh.(B x) of either sign, dA over all B*L steps), so their fp32 rounding error
# scales with the sum of the terms' magnitudes, a few times |result|: each
# gets 5x the fp32 bound of the others.
TOL = {"f32": {**{k: 1e-4 for k in NAMES}, "ddelta": 5e-4, "dA": 5e-4},
       "bf16": {**{k: 1e-3 for k in NAMES}, "dx": 2e-2, "ddelta": 2e-2}}


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m




def case(B, L, D, N, io="f32", softplus=False, state=True, seed=0):
    inp = workloads.s6_inputs(B, L, D, N, io=io, delta="preact" if softplus else "loguniform",
                              dskip="normal", seed=seed)
    g = np.random.Generator(np.random.PCG64(seed + 900))
    inp.A = (-g.uniform(0.1, 4.0, (D, N))).astype(np.float32)
    dy = g.standard_normal((B, L, D)).astype(np.float32)
    if io == "bf16":
        dy_store = workloads.f32_to_bf16_bits(dy)
        dy = workloads.bf16_bits_to_f32(dy_store)
    else:
        dy_store = dy
    h0 = g.standard_normal((B, D, N)).astype(np.float32) if state else None
    dhl = g.standard_normal((B, D, N)).astype(np.float32) if state else None
    return inp, dy, dy_store, h0, dhl


def gpu_bwd(ss, torch, inp, dy_store, h0, dhl, softplus):
    dev = torch.device("cuda:0")
    t = lambda v: to_dev(v, dev, inp.io)
    f = lambda v: None if v is None else to_dev(v, dev)
    out = ss.ss_selective_scan_bwd(t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), f(inp.A),
                                   f(inp.Dskip), t(dy_store), h0=f(h0), dh_last=f(dhl),
                                   delta_softplus=softplus)
    return {k: to_host_f64(v) for k, v in out.items()}


def oracle_bwd(inp, dy, h0, dhl, softplus):
    return oracle.s6_bwd(inp.x_f32, inp.delta_f32, inp.Bt_f32, inp.Ct_f32, inp.A, inp.Dskip, dy,
                         h0=h0, dh_last=dhl, softplus=softplus, threads=THREADS)


def check(got, ref, io, skip_dh0=False):
    for k in NAMES:
        if skip_dh0 and k == "dh0":
            continue
        assert got[k].shape == ref[k].shape, k
        err = rel_err(got[k], ref[k])
        assert err <= TOL[io][k], f"{k}: {err:.3g} > {TOL[io][k]}"


# D = 12, 20: 16-byte rows, so full 8-channel blocks take the vector row
# staging and the last, partial block the per-channel path
SHAPES = [(1, 1, 1, 1), (2, 7, 3, 4), (1, 256, 8, 16), (2, 300, 13, 16), (3, 600, 40, 5),
          (1, 1000, 33, 16), (2, 513, 64, 3), (2, 257, 20, 16), (1, 300, 12, 8)]


@pytest.mark.parametrize("state", [False, True], ids=["zero_state", "with_state"])
@pytest.mark.parametrize("io,softplus", [("f32", False), ("f32", True), ("bf16", True)])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bwd_parity(torch, ss, shape, io, softplus, state):
    inp, dy, dys, h0, dhl = case(*shape, io=io, softplus=softplus, state=state, seed=sum(shape))
    got = gpu_bwd(ss, torch, inp, dys, h0, dhl, softplus)
    ref = oracle_bwd(inp, dy, h0, dhl, softplus)
    check(got, ref, io)


def test_bwd_deterministic(torch, ss):
    inp, dy, dys, h0, dhl = case(2, 700, 72, 16, softplus=True, seed=5)
    first = gpu_bwd(ss, torch, inp, dys, h0, dhl, True)
    for _ in range(20):
        again = gpu_bwd(ss, torch, inp, dys, h0, dhl, True)
        for k in NAMES:
            assert np.array_equal(again[k], first[k]), f"{k} differs between runs"


def test_bwd_empty_sequence(torch, ss):
    """L == 0: no steps, so h_last is h0 and dh0 = dh_last; every sum is 0."""
    dev = torch.device("cuda:0")
    B, D, N = 2, 5, 4
    z = torch.zeros((B, 0, D), device=dev)
    zb = torch.zeros((B, 0, N), device=dev)
    A = -torch.ones((D, N), device=dev)
    dhl = torch.randn((B, D, N), device=dev)
    out = ss.ss_selective_scan_bwd(z, z, zb, zb, A, torch.ones(D, device=dev), z,
                                   h0=torch.randn((B, D, N), device=dev), dh_last=dhl)
    assert torch.equal(out["dh0"], dhl)
    assert not out["dA"].any() and not out["dDskip"].any()


def test_bwd_workload_fp32(torch, ss):
    """The fp32 S6 workload (B16 L2048 D256 N16), every gradient compared."""
    w = workloads.S6["s6_fp32"]
    inp = workloads.s6_workload_inputs(w)
    g = np.random.Generator(np.random.PCG64(17))
    dy = g.standard_normal((w.B, w.L, w.D)).astype(np.float32)
    got = gpu_bwd(ss, torch, inp, dy, None, None, w.softplus)
    ref = oracle_bwd(inp, dy, None, None, w.softplus)
    check(got, ref, "f32")


def test_bwd_workload_bf16(torch, ss):
    """The bf16 S6 workload (B8 L4096 D1536 N16, softplus) in the benchmark's
    configuration, every gradient compared."""
    w = workloads.S6["s6_bf16"]
    inp = workloads.s6_workload_inputs(w)
    g = np.random.Generator(np.random.PCG64(17))
    dys = workloads.f32_to_bf16_bits(g.standard_normal((w.B, w.L, w.D)).astype(np.float32))
    got = gpu_bwd(ss, torch, inp, dys, None, None, w.softplus)
    ref = oracle_bwd(inp, workloads.bf16_bits_to_f32(dys), None, None, w.softplus)
    check(got, ref, "bf16")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_unaligned_rows_match_aligned(torch, ss, io):
    """Inputs 4 (fp32) or 2 (bf16) bytes off a 16-byte boundary take the
    per-element row staging; the gradients are bitwise those of the vector
    path on aligned copies of the same values."""
    inp, dy, dys, h0, dhl = case(2, 300, 24, 16, io=io, softplus=True, seed=29)
    dev = torch.device("cuda:0")
    dt = torch.bfloat16 if io == "bf16" else torch.float32

    def shifted(v):
        src = to_dev(v, dev, io)
        buf = torch.empty(src.numel() + 8, dtype=dt, device=dev)
        out = buf[1:1 + src.numel()].view(src.shape)
        out.copy_(src)
        return out

    f = lambda v: to_dev(v, dev)
    args = [inp.x, inp.delta, inp.Bt, inp.Ct]
    aligned = ss.ss_selective_scan_bwd(*[to_dev(v, dev, io) for v in args], f(inp.A),
                                       f(inp.Dskip), to_dev(dys, dev, io), h0=f(h0),
                                       dh_last=f(dhl), delta_softplus=True)
    moved = ss.ss_selective_scan_bwd(*[shifted(v) for v in args], f(inp.A), f(inp.Dskip),
                                     shifted(dys), h0=f(h0), dh_last=f(dhl), delta_softplus=True)
    assert moved["dx"].data_ptr() % 16 == 0  # outputs are the binding's own
    for k in NAMES:
        assert torch.equal(aligned[k], moved[k]), f"{k} differs between the staging paths"
