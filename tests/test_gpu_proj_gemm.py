"""The layer's projection GEMM (tcgen05 tensor cores, bias in the epilogue)
alone, bit for bit against the oracle's projections.

Inputs follow the layer's exact-sum recipe (workloads.layer_inputs with
io="bf16"): every projection sum is exact in fp32 in any order, so the GPU
and the float64 oracle round the same value to bf16 and must agree exactly.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


@pytest.fixture(scope="module")
def ss():
    import linear_recurrences_gb300 as m
    return m


def gemm_case(M, K, Nout, n_bias, seed):
    """x (M, K) ~ N(0, 1), W (Nout, K) ~ N(0, 1/K), bias (n_bias,) ~ N(-4, 1),
    on the exact-sum grid."""
    g = workloads.generator(seed)
    x = g.standard_normal((M, K))
    W = g.standard_normal((Nout, K)) / np.sqrt(max(K, 1))
    b = g.normal(-4.0, 1.0, n_bias)
    x, W, b = workloads.exact_sum_grid(x, W, b)
    return x.astype(np.float32), W.astype(np.float32), b.astype(np.float32)


def run(ss, torch, x, W, bias, ld_out=None, sentinel=None):
    dev = torch.device("cuda:0")
    tb = lambda v: torch.from_numpy(np.ascontiguousarray(v)).to(dev).to(torch.bfloat16)
    M, Nout = x.shape[0], W.shape[0]
    ld = ld_out or (Nout + 7) // 8 * 8  # rows of 16-byte multiples
    out = torch.zeros((M, ld), dtype=torch.bfloat16, device=dev)
    if sentinel is not None:
        out.fill_(sentinel)
    ws = ss.new_workspace(256, dev)
    bt = torch.from_numpy(bias).to(dev) if bias is not None and bias.size else None
    ss.ss_testing_proj_gemm(tb(x), tb(W), bias=bt, out=out, ld_out=ld, workspace=ws)
    assert ss.ss_get_device_status(ws) == ss.SS_OK
    return out.float().cpu().numpy().astype(np.float64)[:, :ld_out or Nout]


# (M, K, Nout, n_bias): one tile; ragged M, K (< and > one 64-wide K-block)
# and N; two N tiles; the layer's K and N (D = 1536, N = 16)
SHAPES = [(128, 64, 32, 32), (300, 72, 50, 40), (64, 8, 16, 0), (4096, 256, 288, 256),
          (1000, 1536, 1568, 1536), (513, 200, 520, 7)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_bit_exact(torch, ss, shape):
    M, K, Nout, nb = shape
    x, W, bias = gemm_case(M, K, Nout, nb, seed=sum(shape))
    got = run(ss, torch, x, W, bias)
    ref = oracle.projections(x, W, bias if nb else None, io="bf16")
    assert np.array_equal(got, ref), f"{np.sum(got != ref)} of {got.size} differ"


def test_gemm_padded_rows_untouched(torch, ss):
    """Row stride 64 for 50 columns: the columns from the next 16-byte
    boundary on (56..63) keep their values; the tile stores may write 50..55."""
    x, W, bias = gemm_case(200, 64, 50, 20, seed=3)
    got = run(ss, torch, x, W, bias, ld_out=64, sentinel=7.0)
    ref = oracle.projections(x, W, bias, io="bf16")
    assert np.array_equal(got[:, :50], ref)
    assert np.all(got[:, 56:] == 7.0)


def test_gemm_layer_workload_size(torch, ss):
    """The bf16 layer workload's projections at full size (M = B*L = 32768,
    K = D = 1536, Nout = D + 2N = 1568), bias on the first D columns."""
    x, W, bias = gemm_case(32768, 1536, 1568, 1536, seed=11)
    got = run(ss, torch, x, W, bias)
    ref = oracle.projections(x, W, bias, io="bf16")
    assert np.array_equal(got, ref), f"{np.sum(got != ref)} of {got.size} differ"


def test_gemm_deterministic(torch, ss):
    x, W, bias = gemm_case(2048, 512, 544, 512, seed=5)
    first = run(ss, torch, x, W, bias)
    for _ in range(5):
        assert np.array_equal(run(ss, torch, x, W, bias), first)


def test_gemm_refuses_unaligned_layouts(torch, ss):
    dev = torch.device("cuda:0")
    x = torch.zeros((64, 12), dtype=torch.bfloat16, device=dev)   # K = 12: rows not 16 B
    W = torch.zeros((16, 12), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ss.SSError):
        ss.ss_testing_proj_gemm(x, W)
