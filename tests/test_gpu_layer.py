"""GPU selective-scan layer forward (projections + scan) vs the float64 oracle."""
import os

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import rel_err, require_gpu, to_dev, to_host_f64

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m


def layer_case(B, L, D, N, io="f32", seed=0):
    """workloads.layer_inputs: x ~ N(0,1); W ~ N(0, 1/D); b_delta ~ N(-4, 1)
    (small steps, as in the bf16 workload). For bf16 the values lie on the
    grid on which every projection sum is exact in fp32, so the GEMM and the
    oracle round the same pre-activations to bf16."""
    return workloads.layer_inputs(B, L, D, N, io=io, seed=seed)


def gpu_layer(ss, torch, io, x, W, b, A, Ds):
    dev = torch.device("cuda:0")
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    t = lambda v: torch.from_numpy(v).to(dev).to(dt)
    f = lambda v: torch.from_numpy(v).to(dev)
    B, L, D = x.shape
    N = A.shape[1]
    io_dtype = ss.SS_BF16 if io == "bf16" else ss.SS_F32
    ws = ss.new_workspace(ss.ss_selective_scan_layer_workspace_bytes(B, L, D, N, io_dtype), dev)
    y = ss.ss_selective_scan_layer_fwd(t(x), t(W), f(b), f(A), f(Ds), workspace=ws)
    assert ss.ss_get_device_status(ws) == ss.SS_OK
    return to_host_f64(y)


SHAPES = [(1, 1, 8, 1), (2, 33, 16, 4), (2, 300, 64, 16), (1, 1000, 96, 16), (3, 129, 40, 5)]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_layer_parity(torch, ss, shape, io):
    x, W, b, A, Ds = layer_case(*shape, io=io, seed=sum(shape))
    y = gpu_layer(ss, torch, io, x, W, b, A, Ds)
    ref = oracle.layer_fwd(x, W, b, A, Ds, io=io, threads=THREADS)
    assert rel_err(y, ref) <= TOL[io]


def test_layer_matches_scan_on_its_projections(torch, ss):
    """The layer equals the plain scan run on the projections and the
    biased pre-activation, computed here with torch in fp32."""
    dev = torch.device("cuda:0")
    x, W, b, A, Ds = layer_case(2, 500, 48, 16, seed=9)
    tx, tW = torch.from_numpy(x).to(dev), torch.from_numpy(W).to(dev)
    D, N = 48, 16
    y = gpu_layer(ss, torch, "f32", x, W, b, A, Ds)
    P = tx @ tW.T
    pre = (P[..., :D] + torch.from_numpy(b).to(dev)).contiguous()
    ys = ss.ss_selective_scan_fwd(tx, pre, P[..., D:D + N].contiguous(),
                                  P[..., D + N:].contiguous(), torch.from_numpy(A).to(dev),
                                  torch.from_numpy(Ds).to(dev), delta_softplus=True)
    assert rel_err(y, to_host_f64(ys)) <= 1e-4


def test_layer_workload_bf16(torch, ss):
    """The layer on the bf16 workload's shape (B8 L4096 D1536 N16), every
    output of every batch element against the oracle."""
    B, L, D, N = 8, 4096, 1536, 16
    x, W, b, A, Ds = layer_case(B, L, D, N, io="bf16", seed=23)
    y = gpu_layer(ss, torch, "bf16", x, W, b, A, Ds)
    ref = oracle.layer_fwd(x, W, b, A, Ds, io="bf16", threads=THREADS)
    assert rel_err(y, ref) <= TOL["bf16"]


def test_layer_bf16_refuses_unaligned_rows(torch, ss):
    """bf16 rows of D = 12 elements are not 16-byte multiples: the tensor-core
    projection cannot tile them and the call reports SS_ERR_UNSUPPORTED."""
    dev = torch.device("cuda:0")
    B, L, D, N = 1, 8, 12, 2
    x = torch.zeros((B, L, D), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((D + 2 * N, D), dtype=torch.bfloat16, device=dev)
    f = lambda *sh: torch.zeros(sh, dtype=torch.float32, device=dev)
    with pytest.raises(ss.SSError) as e:
        ss.ss_selective_scan_layer_fwd(x, W, f(D), f(D, N), f(D))
    assert e.value.status == ss.SS_ERR_UNSUPPORTED
