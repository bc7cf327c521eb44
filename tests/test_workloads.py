"""Host checks of the seeded input generators (no GPU): the exact-sum grid
that lets the projection GEMM be compared bit for bit, and the layer
inputs' shapes and storage types."""
import numpy as np
import pytest

import workloads



@pytest.mark.parametrize("M,K,Nout,nb", [(257, 1536, 96, 64), (64, 72, 50, 40), (33, 8, 16, 0)])
def test_exact_sum_grid_makes_fp32_sums_exact(M, K, Nout, nb):
    """On the grid, x W^T + b in float32 (one summation order, numpy's) and
    in float64 agree exactly, and x, W are bf16 values."""
    g = workloads.generator(M + K)
    x, W, b = workloads.exact_sum_grid(g.standard_normal((M, K)),
                                       g.standard_normal((Nout, K)) / np.sqrt(K),
                                       g.normal(-4.0, 1.0, nb))
    p64 = x @ W.T
    p64[:, :nb] += b
    p32 = x.astype(np.float32) @ W.astype(np.float32).T
    p32[:, :nb] += b.astype(np.float32)
    assert np.array_equal(p64, p32.astype(np.float64))
    assert np.abs(p64).max() < 16.0
    for v in (x, W):
        v32 = v.astype(np.float32)
        assert np.array_equal(workloads.bf16_bits_to_f32(workloads.f32_to_bf16_bits(v32)), v32)


def test_exact_sum_grid_holds_in_reversed_order():
    """The same sums accumulated term by term in the reverse order (another
    fp32 order) give the same values."""
    g = workloads.generator(5)
    x, W, _ = workloads.exact_sum_grid(g.standard_normal((4, 512)),
                                       g.standard_normal((3, 512)) / np.sqrt(512), np.zeros(0))
    x32, W32 = x.astype(np.float32), W.astype(np.float32)
    for i in range(4):
        for j in range(3):
            acc = np.float32(0.0)
            for k in range(511, -1, -1):
                acc = np.float32(acc + x32[i, k] * W32[j, k])
            assert float(acc) == float(x[i] @ W[j])


def test_layer_inputs_shapes_and_grid():
    x, W, b, A, Ds = workloads.layer_inputs(2, 7, 24, 4, io="bf16", seed=1)
    assert x.shape == (2, 7, 24) and W.shape == (32, 24) and b.shape == (24,)
    assert A.shape == (24, 4) and Ds.shape == (24,) and (A < 0).all()
    assert all(v.dtype == np.float32 for v in (x, W, b, A, Ds))
    assert np.array_equal(np.round(x * 32) / 32, x)
    xf, Wf, _, _, _ = workloads.layer_inputs(2, 7, 24, 4, io="f32", seed=1)
    assert not np.array_equal(xf, x)  # the fp32 recipe stays off the grid
