"""Float64 CPU oracle for the selective-scan hot path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The CUDA library and its Python
binding never import it; the two share no code. The arithmetic lives in
``oracle.c`` (plain sequential loops in double precision); this module only
builds that file with gcc and marshals numpy arrays to it.

Inputs are the exact values the GPU is given: float32 arrays, or bf16 bit
patterns widened exactly to float32 by ``workloads.bf16_bits_to_f32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-pthread"]


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile ``src`` to the shared library ``out`` with gcc (no fast-math,
    no FMA contraction). Returns the path of the library."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    f = ctypes.POINTER(ctypes.c_float)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_affine_f64.argtypes = [f, f, dp, i64]
    lib.oracle_affine_f64.restype = None
    lib.oracle_affine_state_f64.argtypes = [f, f, ctypes.c_double, dp, i64]
    lib.oracle_affine_state_f64.restype = None
    lib.oracle_softplus_f64.argtypes = [ctypes.c_double]
    lib.oracle_softplus_f64.restype = ctypes.c_double
    s6 = [f, f, f, f, f, f, dp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int]
    lib.oracle_s6_fwd_f64.argtypes = s6
    lib.oracle_s6_fwd_f64.restype = ctypes.c_int
    lib.oracle_s6_bidir_f64.argtypes = s6
    lib.oracle_s6_bidir_f64.restype = ctypes.c_int
    lib.oracle_s6_fwd_state_f64.argtypes = [f, f, f, f, f, f, dp, dp, dp, i64, i64, i64, i64,
                                            ctypes.c_int, ctypes.c_int]
    lib.oracle_s6_fwd_state_f64.restype = ctypes.c_int
    lib.oracle_s6_bwd_f64.argtypes = [f, f, f, f, f, f, dp, f, dp, i64, i64, i64, i64,
                                      ctypes.c_int, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
    lib.oracle_s6_bwd_f64.restype = ctypes.c_int
    lib.oracle_s6_channels_f64.argtypes = [
        f, f, f, f, f, f, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
        ctypes.POINTER(ctypes.c_int64), i64, dp, ctypes.c_int]
    lib.oracle_s6_channels_f64.restype = ctypes.c_int
    return lib


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle inputs are float32 (got {a.dtype})")
    return a


def _p(a, t=ctypes.c_float):
    return a.ctypes.data_as(ctypes.POINTER(t))


# ---------------------------------------------------------------- affine
def affine(a, b, lib: ctypes.CDLL | None = None, h0: float | None = None) -> np.ndarray:
    """h[t] = a[t]*h[t-1] + b[t], in float64, from h[-1] = 0, or from h[-1] =
    h0 (a scan continued from an earlier segment's last state)."""
    lib = lib or load()
    a, b = _f32(a), _f32(b)
    if a.shape != b.shape or a.ndim != 1:
        raise ValueError("a and b must be 1-D of equal length")
    h = np.empty(a.shape[0], dtype=np.float64)
    if h0 is None:
        lib.oracle_affine_f64(_p(a), _p(b), _p(h, ctypes.c_double), a.shape[0])
    else:
        lib.oracle_affine_state_f64(_p(a), _p(b), float(h0), _p(h, ctypes.c_double), a.shape[0])
    return h


def softplus(v: float, lib: ctypes.CDLL | None = None) -> float:
    return (lib or load()).oracle_softplus_f64(float(v))


# ---------------------------------------------------------------- S6
def _s6_args(x, delta, Bt, Ct, A, Dskip):
    x, delta, Bt, Ct, A = map(_f32, (x, delta, Bt, Ct, A))
    B, L, D = x.shape
    N = A.shape[1]
    if delta.shape != (B, L, D) or Bt.shape != (B, L, N) or Ct.shape != (B, L, N):
        raise ValueError("shape mismatch")
    if A.shape != (D, N):
        raise ValueError("A must be (D, N)")
    Dskip = np.zeros(D, np.float32) if Dskip is None else _f32(Dskip)
    if Dskip.shape != (D,):
        raise ValueError("Dskip must be (D,)")
    return x, delta, Bt, Ct, A, Dskip, B, L, D, N


def s6_fwd(x, delta, Bt, Ct, A, Dskip=None, softplus=False, threads=1,
           lib: ctypes.CDLL | None = None) -> np.ndarray:
    """S6 selective-scan forward, y (B, L, D) float64."""
    lib = lib or load()
    x, delta, Bt, Ct, A, Dskip, B, L, D, N = _s6_args(x, delta, Bt, Ct, A, Dskip)
    y = np.zeros((B, L, D), dtype=np.float64)
    rc = lib.oracle_s6_fwd_f64(_p(x), _p(delta), _p(Bt), _p(Ct), _p(A), _p(Dskip),
                               _p(y, ctypes.c_double), B, L, D, N,
                               int(bool(softplus)), int(threads))
    if rc:
        raise RuntimeError(f"oracle_s6_fwd_f64 failed ({rc})")
    return y


def s6_fwd_state(x, delta, Bt, Ct, A, Dskip=None, h0=None, softplus=False, threads=1,
                 lib: ctypes.CDLL | None = None):
    """S6 forward from the state h0 ((B, D, N), zeros if None); returns
    (y (B, L, D), h_last (B, D, N)) in float64."""
    lib = lib or load()
    x, delta, Bt, Ct, A, Dskip, B, L, D, N = _s6_args(x, delta, Bt, Ct, A, Dskip)
    h0p = None
    if h0 is not None:
        h0 = np.ascontiguousarray(h0, dtype=np.float64)
        if h0.shape != (B, D, N):
            raise ValueError("h0 must be (B, D, N)")
        h0p = _p(h0, ctypes.c_double)
    y = np.zeros((B, L, D), dtype=np.float64)
    h_last = np.zeros((B, D, N), dtype=np.float64)
    rc = lib.oracle_s6_fwd_state_f64(_p(x), _p(delta), _p(Bt), _p(Ct), _p(A), _p(Dskip), h0p,
                                     _p(y, ctypes.c_double), _p(h_last, ctypes.c_double),
                                     B, L, D, N, int(bool(softplus)), int(threads))
    if rc:
        raise RuntimeError(f"oracle_s6_fwd_state_f64 failed ({rc})")
    return y, h_last


def s6_bidir(x, delta, Bt, Ct, A, Dskip=None, softplus=False, threads=1,
             lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Forward plus reverse recurrence over shared dA, dBx; y (B, L, D)."""
    lib = lib or load()
    x, delta, Bt, Ct, A, Dskip, B, L, D, N = _s6_args(x, delta, Bt, Ct, A, Dskip)
    y = np.zeros((B, L, D), dtype=np.float64)
    rc = lib.oracle_s6_bidir_f64(_p(x), _p(delta), _p(Bt), _p(Ct), _p(A), _p(Dskip),
                                 _p(y, ctypes.c_double), B, L, D, N,
                                 int(bool(softplus)), int(threads))
    if rc:
        raise RuntimeError(f"oracle_s6_bidir_f64 failed ({rc})")
    return y


def s6_channels(x, delta, Bt, Ct, A, Dskip, chans, softplus=False, bidir=False,
                threads=1, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """y for the listed channels c = b*D + d only, as (len(chans), L)."""
    lib = lib or load()
    x, delta, Bt, Ct, A, Dskip, B, L, D, N = _s6_args(x, delta, Bt, Ct, A, Dskip)
    ch = np.ascontiguousarray(chans, dtype=np.int64)
    out = np.zeros((ch.shape[0], L), dtype=np.float64)
    rc = lib.oracle_s6_channels_f64(
        _p(x), _p(delta), _p(Bt), _p(Ct), _p(A), _p(Dskip), B, L, D, N,
        int(bool(softplus)), int(bool(bidir)), _p(ch, ctypes.c_int64),
        ch.shape[0], _p(out, ctypes.c_double), int(threads))
    if rc:
        raise RuntimeError(f"oracle_s6_channels_f64 failed ({rc})")
    return out


def s6_bwd(x, delta, Bt, Ct, A, Dskip, dy, h0=None, dh_last=None, softplus=False, threads=1,
           lib: ctypes.CDLL | None = None) -> dict:
    """Gradients of sum(dy * y) + sum(dh_last * h_last) for the S6 forward
    from h0, in float64: dict with dx, ddelta (B, L, D), dA (D, N),
    dBt, dCt (B, L, N), dDskip (D,), dh0 (B, D, N)."""
    lib = lib or load()
    x, delta, Bt, Ct, A, Dskip, B, L, D, N = _s6_args(x, delta, Bt, Ct, A, Dskip)
    dy = _f32(dy)
    if dy.shape != (B, L, D):
        raise ValueError("dy must be (B, L, D)")

    def state(v, name):
        if v is None:
            return None
        v = np.ascontiguousarray(v, dtype=np.float64)
        if v.shape != (B, D, N):
            raise ValueError(f"{name} must be (B, D, N)")
        return v
    h0, dh_last = state(h0, "h0"), state(dh_last, "dh_last")
    out = {"dx": np.zeros((B, L, D)), "ddelta": np.zeros((B, L, D)), "dA": np.zeros((D, N)),
           "dBt": np.zeros((B, L, N)), "dCt": np.zeros((B, L, N)), "dDskip": np.zeros(D),
           "dh0": np.zeros((B, D, N))}
    dp = lambda v: None if v is None else _p(v, ctypes.c_double)
    rc = lib.oracle_s6_bwd_f64(_p(x), _p(delta), _p(Bt), _p(Ct), _p(A), _p(Dskip), dp(h0), _p(dy),
                               dp(dh_last), B, L, D, N, int(bool(softplus)),
                               *(dp(out[k]) for k in ("dx", "ddelta", "dA", "dBt", "dCt",
                                                      "dDskip", "dh0")), int(threads))
    if rc:
        raise RuntimeError(f"oracle_s6_bwd_f64 failed ({rc})")
    return out


# ---------------------------------------------------------------- layer
def _round_bf16(v):
    """float64 values rounded once to bfloat16 (8 significant bits), to
    nearest with ties to even; returned as float64."""
    m, e = np.frexp(np.asarray(v, dtype=np.float64))  # v = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def projections(x2d, W_proj, bias, io="f32") -> np.ndarray:
    """x2d (M, K) times W_proj (n_out, K) transposed, plus bias (n_bias <=
    n_out values) on the first n_bias columns: a float64 product of the exact
    input values, the bias added before the single rounding to the storage
    type (float32, or bfloat16 with io == "bf16"), as a Linear layer with a
    bias returns it. Returns (M, n_out) float64 holding the rounded values."""
    x2d = np.ascontiguousarray(x2d, dtype=np.float32).astype(np.float64)
    W = np.ascontiguousarray(W_proj, dtype=np.float32).astype(np.float64)
    P = x2d @ W.T
    if bias is not None:
        b = np.ascontiguousarray(bias, dtype=np.float32).astype(np.float64)
        P[:, :b.shape[0]] += b
    if io == "bf16":
        return _round_bf16(P)
    return P.astype(np.float32).astype(np.float64)


def layer_fwd(x, W_proj, b_delta, A, Dskip, io="f32", threads=1,
              lib: ctypes.CDLL | None = None):
    """The selective-scan layer's forward pass ("POPCORNBENCH FW-GLM-5-1
    l2_p30", the model's parameters and forward pass): the three input
    projections, then the scan. W_proj is (D + 2N, D), PyTorch Linear layout:
    rows [0, D) proj_delta, [D, D + N) proj_B, [D + N, D + 2N) proj_C.
        delta = softplus(x W_delta^T + b_delta),  B_t = x W_B^T,  C_t = x W_C^T
    The projections are float64 matrix products of the exact input values,
    the delta bias added to the pre-activation before any rounding (a Linear
    layer adds its bias to the accumulated product); the results enter the
    float64 scan loop rounded once to float32 (the loop's input type), or,
    with io == "bf16", rounded once to bfloat16, as a Linear layer in that
    storage type returns them. Returns y (B, L, D) float64."""
    x = _f32(x)
    W = np.ascontiguousarray(W_proj, dtype=np.float32)
    B, L, D = x.shape
    N = (W.shape[0] - D) // 2
    if W.shape != (D + 2 * N, D) or N < 1:
        raise ValueError("W_proj must be (D + 2N, D)")
    if np.shape(b_delta) != (D,):
        raise ValueError("b_delta must be (D,)")
    P = projections(x.reshape(B * L, D), W, b_delta, io)               # (B*L, D + 2N)
    pre = P[:, :D].reshape(B, L, D).astype(np.float32)
    Bt = P[:, D:D + N].reshape(B, L, N).astype(np.float32)
    Ct = P[:, D + N:].reshape(B, L, N).astype(np.float32)
    return s6_fwd(x, pre, Bt, Ct, A, Dskip, softplus=True, threads=threads, lib=lib)
