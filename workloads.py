"""Seeded synthetic inputs for the selective-scan workloads.

This module is shared by the tests, the benchmark and the CPU oracle's
callers. It draws random numbers and packs them into the storage types the
kernels read (fp32, or bf16 bit patterns). It contains no step of the
recurrence itself: no scan, no discretisation, no readout.

Draws use numpy's PCG64 generator, in float64, in a fixed order per
workload (a then b; x, delta, Bt, Ct, Dskip), then cast to the storage
type. A[d, n] is not random: it is -(n + 1) in every S6 workload.

The workload shapes and distributions follow the five configurations of the
selective-scan problem:
  affine_small  n = 65,536,  a ~ U(0.5, 1), b ~ N(0, 1)
  affine_large  n = 2**28,   a ~ U(0.9, 1), b ~ N(0, 1)
  s6_fp32       B16 L2048 D256 N16 fp32, x ~ N(0,1), delta log-uniform in
                [1e-3, 1e-1], Bt, Ct ~ N(0,1), Dskip = 1
  s6_bf16       B8 L4096 D1536 N16, x, delta, Bt, Ct stored as bf16,
                delta pre-activation ~ N(-4, 1) (softplus applied in-kernel),
                Dskip ~ N(0,1) fp32, y stored as bf16
  s6_bidir      B2 L16384 D768 N16 fp32, distributions as s6_fp32
"""
from __future__ import annotations

import dataclasses

import numpy as np

SEED = 0


def generator(seed: int = SEED) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- bf16 packing
def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16. NaN stays NaN (quiet bit forced).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    nan = np.isnan(x)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- affine scan
@dataclasses.dataclass(frozen=True)
class AffineWorkload:
    name: str
    n: int
    a_lo: float
    a_hi: float


AFFINE = {
    "affine_small": AffineWorkload("affine_small", 65_536, 0.5, 1.0),
    "affine_large": AffineWorkload("affine_large", 1 << 28, 0.9, 1.0),
}


def affine_inputs(n: int, a_lo: float, a_hi: float, seed: int = SEED):
    """(a, b) as float32 arrays of length n: a ~ U(a_lo, a_hi), b ~ N(0, 1)."""
    g = generator(seed)
    a = g.uniform(a_lo, a_hi, size=n).astype(np.float32)
    b = g.standard_normal(size=n).astype(np.float32)
    return a, b


# ---------------------------------------------------------------- S6
@dataclasses.dataclass(frozen=True)
class S6Workload:
    name: str
    B: int
    L: int
    D: int
    N: int
    io: str              # "f32" or "bf16"
    delta: str           # "loguniform" (positive step) or "preact" (softplus input)
    dskip: str           # "one" or "normal"
    softplus: bool
    bidir: bool

    @property
    def elements(self) -> int:
        return self.B * self.L * self.D


S6 = {
    "s6_fp32": S6Workload("s6_fp32", 16, 2048, 256, 16, "f32", "loguniform", "one", False, False),
    "s6_bf16": S6Workload("s6_bf16", 8, 4096, 1536, 16, "bf16", "preact", "normal", True, False),
    "s6_bidir": S6Workload("s6_bidir", 2, 16384, 768, 16, "f32", "loguniform", "one", False, True),
}


@dataclasses.dataclass
class S6Inputs:
    """Storage-typed inputs plus their exact float32 values.

    `x`, `delta`, `Bt`, `Ct` are float32 arrays (io == "f32") or uint16 bf16
    bit patterns (io == "bf16"); `*_f32` hold the exact float32 value of what
    is stored. A and Dskip are always float32.
    """
    io: str
    x: np.ndarray
    delta: np.ndarray
    Bt: np.ndarray
    Ct: np.ndarray
    A: np.ndarray
    Dskip: np.ndarray
    x_f32: np.ndarray
    delta_f32: np.ndarray
    Bt_f32: np.ndarray
    Ct_f32: np.ndarray


def s6_inputs(B: int, L: int, D: int, N: int, *, io: str = "f32",
              delta: str = "loguniform", dskip: str = "one",
              seed: int = SEED) -> S6Inputs:
    """Seeded S6 inputs in the layouts x, delta: (B, L, D); Bt, Ct: (B, L, N);
    A: (D, N); Dskip: (D,)."""
    g = generator(seed)
    x = g.standard_normal(size=(B, L, D))
    if delta == "loguniform":
        dl = 10.0 ** g.uniform(-3.0, -1.0, size=(B, L, D))
    elif delta == "preact":
        dl = g.normal(-4.0, 1.0, size=(B, L, D))
    else:
        raise ValueError(delta)
    Bt = g.standard_normal(size=(B, L, N))
    Ct = g.standard_normal(size=(B, L, N))
    if dskip == "one":
        Ds = np.ones(D)
    elif dskip == "normal":
        Ds = g.standard_normal(size=D)
    elif dskip == "zero":
        Ds = np.zeros(D)
    else:
        raise ValueError(dskip)
    A = -np.broadcast_to(np.arange(1, N + 1, dtype=np.float64), (D, N))

    def store(v):
        v32 = np.ascontiguousarray(v, dtype=np.float32)
        if io == "f32":
            return v32, v32
        if io == "bf16":
            bits = f32_to_bf16_bits(v32)
            return bits, bf16_bits_to_f32(bits)
        raise ValueError(io)

    xs, x32 = store(x)
    ds, d32 = store(dl)
    bs, b32 = store(Bt)
    cs, c32 = store(Ct)
    return S6Inputs(io, xs, ds, bs, cs,
                    np.ascontiguousarray(A, dtype=np.float32),
                    np.ascontiguousarray(Ds, dtype=np.float32),
                    x32, d32, b32, c32)


def s6_workload_inputs(w: S6Workload, seed: int = SEED) -> S6Inputs:
    return s6_inputs(w.B, w.L, w.D, w.N, io=w.io, delta=w.delta,
                     dskip=w.dskip, seed=seed)


# ---------------------------------------------------------------- layer
def layer_inputs(B: int, L: int, D: int, N: int, *, io: str = "f32", seed: int = SEED):
    """Inputs of the selective-scan layer (projections, then the scan):
    x (B, L, D), W_proj (D + 2N, D) in Linear layout (rows: proj_delta,
    proj_B, proj_C), b_delta (D,), A (D, N), Dskip (D,), all float32 arrays
    holding the values the kernels see. x ~ N(0, 1), W ~ N(0, 1/D) (unit-
    variance projections), b_delta ~ N(-4, 1) (softplus gives small steps, as
    in the bf16 workload), A ~ -U(0.1, 4), Dskip ~ N(0, 1).

    io == "bf16" puts every value on a grid on which a projection sum is
    exact in fp32 whatever the order of its terms: x on multiples of 2^-5
    inside (-4, 4); W rounded to bf16 with magnitudes below 2^-8 set to 0 (so
    every product is a multiple of 2^-20); b_delta on multiples of 2^-20. The
    projections stay far below 16 in magnitude, so the fp32 sums are exact and
    the one rounding to bf16 sees the same value on every side."""
    g = generator(seed)
    x = g.standard_normal((B, L, D))
    W = g.standard_normal((D + 2 * N, D)) / np.sqrt(D)
    b = g.normal(-4.0, 1.0, D)
    A = -g.uniform(0.1, 4.0, (D, N))
    Ds = g.standard_normal(D)
    if io == "bf16":
        x, W, b = exact_sum_grid(x, W, b)
    f = lambda v: np.ascontiguousarray(v, dtype=np.float32)
    return f(x), f(W), f(b), f(A), f(Ds)


def exact_sum_grid(x, W, b):
    """Puts GEMM operands on the grid on which x W^T + b is exact in fp32 in
    any summation order (for |x W^T + b| < 16): x on multiples of 2^-5 inside
    (-4, 4), W rounded to bf16 with magnitudes below 2^-8 set to 0 (every
    product a multiple of 2^-20), b on multiples of 2^-20. x and W are then
    bf16 values. Returns float64 arrays."""
    x = np.clip(np.round(np.asarray(x, np.float64) * 32.0), -127, 127) / 32.0
    W = bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(W, np.float32))).astype(np.float64)
    W[np.abs(W) < 2.0 ** -8] = 0.0
    b = np.round(np.asarray(b, np.float64) * 2.0 ** 20) / 2.0 ** 20
    return x, W, b
