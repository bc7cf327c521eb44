"""Checks that pin the float64 oracle to facts fixed outside the oracle.

Each check takes a loaded oracle library (ctypes handle) and raises
AssertionError on a mismatch. The same checks run against the real oracle
(tests/test_oracle_pins.py, all must pass) and against copies of oracle.c
with a planted mistake (tests/test_oracle_mutants.py, at least one must
fail), so a dropped term, a wrong sign or index, or a swapped operand in
the oracle cannot go unnoticed.

What pins what:
  affine  a == 1 with integer b: the exact integer prefix sum.
          a == 0: h == b exactly.
          constant a, b == 1: geometric closed form (1 - a^(t+1)) / (1 - a).
          constant a, general b: explicit power sum with math.fsum.
          random dyadic inputs, n <= 8: every bracketing of the affine-pair
          combine (a, b) o (a', b') = (a a', a' b + b') in exact rational
          arithmetic equals the oracle exactly; the operand-swapped combine
          does not.
          impulse response: b = e_j gives products of a.
  S6      explicit O(L^2) solution of the linear recurrence (matrix form),
          with math.fsum, for forward and bidirectional outputs.
          A == 0: prefix-sum closed form.  Ct == 0 or delta == 0: y == D x.
          L == 1: one-step closed form.  softplus: ln 2 at 0, the identity
          sp(v) - sp(-v) = v, threshold reading v > 20 -> v.
          time-reversal involution of the bidirectional output; bidir equals
          forward plus flipped forward of flipped inputs; linearity in x;
          channel permutation equivariance; batch independence.
  state   forward from an initial state h0: the matrix form plus h0's decay
          term, and the final state's matrix form; x == 0: pure decay of h0
          in closed form; a run split at any step and resumed from the first
          part's final state equals the unsplit run exactly.
"""
from __future__ import annotations

import itertools
import math
from fractions import Fraction

import numpy as np

import oracle


# ---------------------------------------------------------------- helpers
def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _dyadic(g, n, lo, hi, bits):
    """Random multiples of 2**-bits in [lo, hi], exactly representable."""
    k = g.integers(int(lo * 2 ** bits), int(hi * 2 ** bits) + 1, size=n)
    return (k / 2.0 ** bits).astype(np.float32)


def _combine(p, q):
    """(a, b) o (a', b') = (a a', a' b + b'): p earlier, q later."""
    return (p[0] * q[0], q[0] * p[1] + q[1])


def _swapped(p, q):
    return (p[0] * q[0], p[0] * q[1] + p[1])


def _all_folds(items, comb):
    """Every full bracketing of a non-empty sequence under `comb`."""
    if len(items) == 1:
        return [items[0]]
    out = []
    for k in range(1, len(items)):
        for left in _all_folds(items[:k], comb):
            for right in _all_folds(items[k:], comb):
                out.append(comb(left, right))
    return out


def _rel(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(x - ref) / np.maximum(1.0, np.abs(ref)))) if x.size else 0.0


# ---------------------------------------------------------------- affine pins
def pin_affine_ones_integer(lib):
    g = _rng(1)
    n = 4096
    b = g.integers(-8, 9, size=n).astype(np.float32)
    a = np.ones(n, np.float32)
    h = oracle.affine(a, b, lib=lib)
    exact = np.cumsum(b.astype(np.int64))
    assert np.array_equal(h, exact.astype(np.float64)), "a==1 must give the exact prefix sum"


def pin_affine_zero(lib):
    g = _rng(2)
    b = g.standard_normal(1000).astype(np.float32)
    h = oracle.affine(np.zeros_like(b), b, lib=lib)
    assert np.array_equal(h, b.astype(np.float64)), "a==0 must give h==b"


def pin_affine_geometric(lib):
    for a0 in (0.5, 0.9, 0.99):
        a32 = np.float32(a0)
        n = 300
        h = oracle.affine(np.full(n, a32, np.float32), np.ones(n, np.float32), lib=lib)
        av = float(a32)
        t = np.arange(n)
        closed = (1.0 - av ** (t + 1)) / (1.0 - av)
        assert _rel(h, closed) < 1e-12, f"geometric closed form, a={a0}"


def pin_affine_power_sum(lib):
    g = _rng(3)
    n = 64
    a32 = np.float32(0.875)
    b = g.standard_normal(n).astype(np.float32)
    h = oracle.affine(np.full(n, a32, np.float32), b, lib=lib)
    av = float(a32)
    ref = [math.fsum(av ** (t - j) * float(b[j]) for j in range(t + 1)) for t in range(n)]
    assert _rel(h, ref) < 1e-12, "power-sum closed form"


def pin_affine_bracketings(lib):
    g = _rng(4)
    for n in range(1, 8):
        for _ in range(3):
            a = _dyadic(g, n, -1.0, 1.0, 3)
            b = _dyadic(g, n, -2.0, 2.0, 3)
            h = oracle.affine(a, b, lib=lib)
            pairs = [(Fraction(float(x)), Fraction(float(y))) for x, y in zip(a, b)]
            for t in range(n):
                for res in _all_folds(pairs[: t + 1], _combine):
                    # h[t] is the b-part of the prefix composition (h[-1] = 0)
                    assert Fraction(h[t]) == res[1], "bracketing disagrees with oracle"


def pin_affine_swapped_combine_is_caught(lib):
    """The suite must catch an operand-order error: the swapped combine gives
    a different value on a random instance, so a scan built on it would fail
    pin_affine_bracketings."""
    g = _rng(5)
    a = _dyadic(g, 6, -1.0, 1.0, 3)
    b = _dyadic(g, 6, -2.0, 2.0, 3)
    h = oracle.affine(a, b, lib=lib)
    pairs = [(Fraction(float(x)), Fraction(float(y))) for x, y in zip(a, b)]
    good = _all_folds(pairs, _combine)
    bad = _all_folds(pairs, _swapped)
    assert all(r[1] == Fraction(h[-1]) for r in good)
    assert any(r[1] != Fraction(h[-1]) for r in bad), "swapped combine went unnoticed"


def pin_affine_impulse(lib):
    g = _rng(6)
    n, j = 40, 7
    a = _dyadic(g, n, 0.5, 1.0, 4)
    b = np.zeros(n, np.float32)
    b[j] = 1.0
    h = oracle.affine(a, b, lib=lib)
    for t in range(n):
        ref = 0.0 if t < j else math.prod(float(v) for v in a[j + 1: t + 1])
        assert abs(h[t] - ref) <= 1e-15 * max(1.0, abs(ref)), "impulse response"


def pin_affine_edges(lib):
    assert oracle.affine(np.zeros(0, np.float32), np.zeros(0, np.float32), lib=lib).shape == (0,)
    h = oracle.affine(np.array([0.75], np.float32), np.array([-2.5], np.float32), lib=lib)
    assert h[0] == -2.5


def pin_affine_state_prepend(lib):
    """Starting from h0 is the plain scan of the sequence with one element
    (a = 0, b = h0) put in front: exact, since the arithmetic is the same."""
    g = _rng(7)
    for n in (1, 5, 33):
        a = _dyadic(g, n, -1.0, 1.0, 4)
        b = _dyadic(g, n, -2.0, 2.0, 4)
        h0 = float(_dyadic(g, 1, -4.0, 4.0, 4)[0])
        h = oracle.affine(a, b, lib=lib, h0=h0)
        longer = oracle.affine(np.concatenate([np.zeros(1, np.float32), a]),
                               np.concatenate([np.array([h0], np.float32), b]), lib=lib)
        assert np.array_equal(h, longer[1:]), "h0 start differs from a prepended element"


def pin_affine_state_closed_form(lib):
    """a == c, b == 1 from h0: h[t] = c^(t+1) h0 + (1 - c^(t+1)) / (1 - c)."""
    c, h0, n = 0.75, -3.0, 200
    h = oracle.affine(np.full(n, c, np.float32), np.ones(n, np.float32), lib=lib, h0=h0)
    t = np.arange(n)
    closed = c ** (t + 1) * h0 + (1.0 - c ** (t + 1)) / (1.0 - c)
    assert _rel(h, closed) < 1e-12, "closed form from h0"
    # c = 1/2: every power is exact, so the decay of h0 must be too
    h = oracle.affine(np.full(n, 0.5, np.float32), np.zeros(n, np.float32), lib=lib, h0=h0)
    assert np.array_equal(h, 0.5 ** (t + 1) * h0), "pure decay of h0"


def pin_affine_state_split(lib):
    """Scanning [0, k) and then [k, n) from the first part's last state is the
    same loop as scanning [0, n) in one go: bitwise equal."""
    g = _rng(8)
    n = 1000
    a = g.uniform(0.9, 1.0, n).astype(np.float32)
    b = g.standard_normal(n).astype(np.float32)
    whole = oracle.affine(a, b, lib=lib)
    for k in (1, 17, 500, 999):
        first = oracle.affine(a[:k], b[:k], lib=lib)
        second = oracle.affine(a[k:], b[k:], lib=lib, h0=first[-1])
        assert np.array_equal(np.concatenate([first, second]), whole), f"split at {k}"


AFFINE_PINS = [pin_affine_ones_integer, pin_affine_zero, pin_affine_geometric,
               pin_affine_power_sum, pin_affine_bracketings,
               pin_affine_swapped_combine_is_caught, pin_affine_impulse,
               pin_affine_edges, pin_affine_state_prepend, pin_affine_state_closed_form,
               pin_affine_state_split]


# ---------------------------------------------------------------- S6 pins
def _small_s6(seed, B=2, L=9, D=3, N=4, softplus=False, A_zero=False):
    g = _rng(seed)
    x = g.standard_normal((B, L, D)).astype(np.float32)
    if softplus:
        dl = g.normal(-1.0, 1.5, (B, L, D)).astype(np.float32)
    else:
        dl = (10.0 ** g.uniform(-2, 0, (B, L, D))).astype(np.float32)
    Bt = g.standard_normal((B, L, N)).astype(np.float32)
    Ct = g.standard_normal((B, L, N)).astype(np.float32)
    # A depends on d and n, so a transposed index shows up
    A = (np.zeros((D, N)) if A_zero else -g.uniform(0.2, 3.0, (D, N))).astype(np.float32)
    Ds = g.standard_normal(D).astype(np.float32)
    return x, dl, Bt, Ct, A, Ds


def _sp(v):
    return v if v > 20.0 else math.log1p(math.exp(v))


def _matrix_form(x, dl, Bt, Ct, A, Ds, softplus, bidir):
    """y[b,t,d] = sum_{j<=t} sum_n C[t,n] exp(A[d,n] sum_{i=j+1..t} delta_i)
                  delta_j B[j,n] x_j + D x_t   (+ the mirror sum over j>=t)."""
    B, L, D = x.shape
    N = A.shape[1]
    y = np.zeros((B, L, D))
    for b in range(B):
        for d in range(D):
            dd = [(_sp(float(dl[b, t, d])) if softplus else float(dl[b, t, d])) for t in range(L)]
            for t in range(L):
                terms = []
                for j in range(t + 1):
                    s = math.fsum(dd[j + 1: t + 1])
                    for n in range(N):
                        terms.append(float(Ct[b, t, n]) * math.exp(float(A[d, n]) * s)
                                     * dd[j] * float(Bt[b, j, n]) * float(x[b, j, d]))
                if bidir:
                    for j in range(t, L):
                        s = math.fsum(dd[t:j])
                        for n in range(N):
                            terms.append(float(Ct[b, t, n]) * math.exp(float(A[d, n]) * s)
                                         * dd[j] * float(Bt[b, j, n]) * float(x[b, j, d]))
                    terms.append(float(Ds[d]) * float(x[b, t, d]))
                terms.append(float(Ds[d]) * float(x[b, t, d]))
                y[b, t, d] = math.fsum(terms)
    return y


def pin_s6_matrix_form(lib):
    for seed, sp in ((10, False), (11, True)):
        args = _small_s6(seed, softplus=sp)
        y = oracle.s6_fwd(*args, softplus=sp, lib=lib)
        ref = _matrix_form(*args, softplus=sp, bidir=False)
        assert _rel(y, ref) < 1e-12, f"forward matrix form (softplus={sp})"


def pin_s6_bidir_matrix_form(lib):
    for seed, sp in ((12, False), (13, True)):
        args = _small_s6(seed, L=8, softplus=sp)
        y = oracle.s6_bidir(*args, softplus=sp, lib=lib)
        ref = _matrix_form(*args, softplus=sp, bidir=True)
        assert _rel(y, ref) < 1e-12, f"bidirectional matrix form (softplus={sp})"


def pin_s6_A_zero(lib):
    x, dl, Bt, Ct, A, Ds = _small_s6(14, L=50, A_zero=True)
    y = oracle.s6_fwd(x, dl, Bt, Ct, A, Ds, lib=lib)
    # dA = 1: h[t, n] = sum_{j<=t} delta_j B[j, n] x_j
    u = dl.astype(np.float64) * x.astype(np.float64)                 # (B, L, D)
    h = np.cumsum(u[:, :, :, None] * Bt.astype(np.float64)[:, :, None, :], axis=1)
    ref = np.einsum("bldn,bln->bld", h, Ct.astype(np.float64)) + x * Ds.astype(np.float64)
    assert _rel(y, ref) < 1e-12, "A == 0 prefix-sum closed form"


def pin_s6_C_zero_and_delta_zero(lib):
    x, dl, Bt, Ct, A, Ds = _small_s6(15, L=20)
    ref = x.astype(np.float64) * Ds.astype(np.float64)
    y = oracle.s6_fwd(x, dl, Bt, np.zeros_like(Ct), A, Ds, lib=lib)
    assert np.array_equal(y, ref), "Ct == 0 must give y == D x"
    y = oracle.s6_fwd(x, np.zeros_like(dl), Bt, Ct, A, Ds, lib=lib)
    assert np.array_equal(y, ref), "delta == 0 must give y == D x"
    y = oracle.s6_bidir(x, np.zeros_like(dl), Bt, Ct, A, Ds, lib=lib)
    assert np.array_equal(y, 2.0 * ref), "bidir with delta == 0 gives 2 D x"


def pin_s6_one_step(lib):
    x, dl, Bt, Ct, A, Ds = _small_s6(16, L=1, N=5)
    y = oracle.s6_fwd(x, dl, Bt, Ct, A, Ds, lib=lib)
    B, _, D = x.shape
    for b in range(B):
        for d in range(D):
            ref = math.fsum(float(Ct[b, 0, n]) * float(dl[b, 0, d]) * float(Bt[b, 0, n])
                            * float(x[b, 0, d]) for n in range(5)) + float(Ds[d]) * float(x[b, 0, d])
            assert abs(y[b, 0, d] - ref) <= 1e-14 * max(1.0, abs(ref)), "one-step closed form"


def pin_softplus(lib):
    sp = lambda v: oracle.softplus(v, lib=lib)
    assert abs(sp(0.0) - math.log(2.0)) < 1e-16
    for v in (-30.0, -5.0, -0.3, 0.7, 4.0, 19.5):
        assert abs(sp(v) - sp(-v) - v) < 1e-14 * max(1.0, abs(v)), "sp(v) - sp(-v) = v"
    assert sp(25.0) == 25.0 and sp(20.5) == 20.5, "threshold reading: v > 20 returns v"
    assert abs(sp(-40.0) - math.exp(-40.0)) < 1e-30
    assert abs(sp(1.0) - 1.3132616875182228) < 1e-15


def pin_s6_reversal(lib):
    args = _small_s6(17, L=30)
    x, dl, Bt, Ct, A, Ds = args
    y = oracle.s6_bidir(*args, lib=lib)
    fl = lambda v: np.ascontiguousarray(v[:, ::-1])
    yr = oracle.s6_bidir(fl(x), fl(dl), fl(Bt), fl(Ct), A, Ds, lib=lib)
    assert np.array_equal(fl(yr), y), "bidir(flip(inputs)) == flip(bidir(inputs))"
    yf = oracle.s6_fwd(*args, lib=lib)
    yb = fl(oracle.s6_fwd(fl(x), fl(dl), fl(Bt), fl(Ct), A, Ds, lib=lib))
    assert np.array_equal(y, yf + yb), "bidir == fwd + flip(fwd(flip))"


def pin_s6_linear_in_x(lib):
    x, dl, Bt, Ct, A, Ds = _small_s6(18, L=25)
    x2 = _rng(19).standard_normal(x.shape).astype(np.float32)
    for f in (oracle.s6_fwd, oracle.s6_bidir):
        y1 = f(x, dl, Bt, Ct, A, Ds, lib=lib)
        y2 = f(x2, dl, Bt, Ct, A, Ds, lib=lib)
        y12 = f((x.astype(np.float64) + x2).astype(np.float32), dl, Bt, Ct, A, Ds, lib=lib)
        # x + x2 is rounded to fp32; compare against the rounded-sum response
        assert _rel(y12, y1 + y2) < 1e-6, "linearity in x"


def pin_s6_channel_structure(lib):
    x, dl, Bt, Ct, A, Ds = _small_s6(20, B=3, L=12, D=5)
    y = oracle.s6_fwd(x, dl, Bt, Ct, A, Ds, lib=lib)
    perm = np.array([3, 0, 4, 1, 2])
    yp = oracle.s6_fwd(np.ascontiguousarray(x[:, :, perm]), np.ascontiguousarray(dl[:, :, perm]),
                       Bt, Ct, np.ascontiguousarray(A[perm]), np.ascontiguousarray(Ds[perm]), lib=lib)
    assert np.array_equal(yp, y[:, :, perm]), "channel permutation equivariance"
    y0 = oracle.s6_fwd(x[:1], dl[:1], Bt[:1], Ct[:1], A, Ds, lib=lib)
    assert np.array_equal(y0, y[:1]), "batch elements are independent"
    ch = np.array([0, 7, 14, 3])
    yc = oracle.s6_channels(x, dl, Bt, Ct, A, Ds, ch, lib=lib)
    for i, c in enumerate(ch):
        assert np.array_equal(yc[i], y[c // 5, :, c % 5]), "channel sampler agrees"


def _state_matrix_form(x, dl, Bt, Ct, A, Ds, h0):
    """The forward matrix form plus the initial state's response
    y[t] += sum_n C[t,n] exp(A[d,n] sum_{i<=t} delta_i) h0[n], and the final
    state h_last[n] = sum_j exp(A[d,n] sum_{i=j+1..L-1} delta_i) delta_j B[j,n]
    x_j + exp(A[d,n] sum_i delta_i) h0[n]."""
    y = _matrix_form(x, dl, Bt, Ct, A, Ds, softplus=False, bidir=False)
    B, L, D = x.shape
    N = A.shape[1]
    hl = np.zeros((B, D, N))
    for b in range(B):
        for d in range(D):
            dd = [float(dl[b, t, d]) for t in range(L)]
            for t in range(L):
                s = math.fsum(dd[: t + 1])
                y[b, t, d] += math.fsum(float(Ct[b, t, n]) * math.exp(float(A[d, n]) * s)
                                        * float(h0[b, d, n]) for n in range(N))
            for n in range(N):
                terms = [math.exp(float(A[d, n]) * math.fsum(dd[j + 1:])) * dd[j]
                         * float(Bt[b, j, n]) * float(x[b, j, d]) for j in range(L)]
                terms.append(math.exp(float(A[d, n]) * math.fsum(dd)) * float(h0[b, d, n]))
                hl[b, d, n] = math.fsum(terms)
    return y, hl


def pin_s6_state_matrix_form(lib):
    args = _small_s6(21, L=10)
    h0 = _rng(22).standard_normal((2, 3, 4))
    y, hl = oracle.s6_fwd_state(*args, h0=h0, lib=lib)
    ry, rhl = _state_matrix_form(*args, h0)
    assert _rel(y, ry) < 1e-12, "forward from h0: matrix form"
    assert _rel(hl, rhl) < 1e-12, "final state: matrix form"


def pin_s6_state_x_zero(lib):
    x, dl, Bt, Ct, A, Ds = _small_s6(23, L=40)
    h0 = _rng(24).standard_normal((2, 3, 4))
    y, hl = oracle.s6_fwd_state(np.zeros_like(x), dl, Bt, Ct, A, Ds, h0=h0, lib=lib)
    # no input: h[t, n] = exp(A[d, n] * sum_{i<=t} delta_i) * h0[n]
    S = np.cumsum(dl.astype(np.float64), axis=1)                       # (B, L, D)
    h = np.exp(S[:, :, :, None] * A.astype(np.float64)[None, None]) * h0[:, None]
    assert _rel(y, np.einsum("bldn,bln->bld", h, Ct.astype(np.float64))) < 1e-12, \
        "x == 0: decay of h0"
    assert _rel(hl, h[:, -1]) < 1e-12, "x == 0: final state"


def pin_s6_state_split(lib):
    args = _small_s6(25, L=31)
    x, dl, Bt, Ct, A, Ds = args
    h0 = _rng(26).standard_normal((2, 3, 4))
    y, hl = oracle.s6_fwd_state(*args, h0=h0, lib=lib)
    cut = lambda v, a, b: np.ascontiguousarray(v[:, a:b])
    for L1 in (1, 12, 30):
        y1, h1 = oracle.s6_fwd_state(cut(x, 0, L1), cut(dl, 0, L1), cut(Bt, 0, L1),
                                     cut(Ct, 0, L1), A, Ds, h0=h0, lib=lib)
        y2, h2 = oracle.s6_fwd_state(cut(x, L1, 31), cut(dl, L1, 31), cut(Bt, L1, 31),
                                     cut(Ct, L1, 31), A, Ds, h0=h1, lib=lib)
        assert np.array_equal(np.concatenate([y1, y2], axis=1), y), "split run == one run"
        assert np.array_equal(h2, hl), "split run's final state == one run's"
    y0, _ = oracle.s6_fwd_state(*args, lib=lib)
    assert np.array_equal(y0, oracle.s6_fwd(*args, lib=lib)), "h0 = None is the zero state"


S6_PINS = [pin_s6_matrix_form, pin_s6_bidir_matrix_form, pin_s6_A_zero,
           pin_s6_C_zero_and_delta_zero, pin_s6_one_step, pin_softplus,
           pin_s6_reversal, pin_s6_linear_in_x, pin_s6_channel_structure,
           pin_s6_state_matrix_form, pin_s6_state_x_zero, pin_s6_state_split]

ALL_PINS = AFFINE_PINS + S6_PINS


# ---------------------------------------------------------------- backward pins
def _dyadic_s6(seed, B=2, L=5, D=3, N=4, softplus=False):
    """Inputs that are multiples of 2**-6 (delta: 2**-8) in small ranges, so
    that moving any of them by 2**-14 is exact in float32."""
    g = _rng(seed)
    dy = lambda *sh: _dyadic(g, int(np.prod(sh)), -2.0, 2.0, 6).reshape(sh)
    x, Bt, Ct, dyv = dy(B, L, D), dy(B, L, N), dy(B, L, N), dy(B, L, D)
    if softplus:
        dl = _dyadic(g, B * L * D, -3.0, 2.0, 6).reshape(B, L, D)
    else:
        dl = _dyadic(g, B * L * D, 2.0 ** -6, 1.0, 8).reshape(B, L, D)
    A = _dyadic(g, D * N, -3.0, -0.25, 6).reshape(D, N)
    Ds = _dyadic(g, D, -1.0, 1.0, 6)
    h0 = g.integers(-64, 65, (B, D, N)) / 32.0
    dhl = g.integers(-64, 65, (B, D, N)) / 32.0
    return [x, dl, Bt, Ct, A, Ds], h0, dyv, dhl


def _loss(lib, args, h0, dyv, dhl, softplus):
    y, hl = oracle.s6_fwd_state(*args, h0=h0, softplus=softplus, lib=lib)
    return math.fsum((y * dyv.astype(np.float64)).ravel()) + math.fsum((hl * dhl).ravel())


def _check_fd(lib, seed, softplus):
    args, h0, dyv, dhl = _dyadic_s6(seed, softplus=softplus)
    gr = oracle.s6_bwd(*args, dyv, h0=h0, dh_last=dhl, softplus=softplus, lib=lib)
    eps = 2.0 ** -14
    names = ["dx", "ddelta", "dBt", "dCt", "dA", "dDskip"]
    for k, name in enumerate(names):
        src = {0: 0, 1: 1, 2: 2, 3: 3, 4: 4, 5: 5}[k]
        for idx in np.ndindex(args[src].shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[src][idx] += np.float32(eps)
            minus[src][idx] -= np.float32(eps)
            assert plus[src][idx] - minus[src][idx] == np.float32(2 * eps), "exact perturbation"
            fd = (_loss(lib, plus, h0, dyv, dhl, softplus)
                  - _loss(lib, minus, h0, dyv, dhl, softplus)) / (2 * eps)
            an = gr[name][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), f"{name}{idx}: fd {fd} vs {an}"
    for idx in np.ndindex(h0.shape):
        hp, hm = h0.copy(), h0.copy()
        hp[idx] += eps
        hm[idx] -= eps
        fd = (_loss(lib, args, hp, dyv, dhl, softplus)
              - _loss(lib, args, hm, dyv, dhl, softplus)) / (2 * eps)
        an = gr["dh0"][idx]
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), f"dh0{idx}: fd {fd} vs {an}"


def pin_bwd_finite_differences(lib):
    _check_fd(lib, 30, softplus=False)


def pin_bwd_finite_differences_softplus(lib):
    _check_fd(lib, 31, softplus=True)


def pin_bwd_euler_and_skip(lib):
    """y and h_last are linear in x (h0 = 0), in Bt, in Ct and in h0 (x = 0),
    so sum(v * dL/dv) recovers the matching part of the loss exactly; and
    dDskip[d] = sum over (b, t) of dy * x."""
    args, h0, dyv, dhl = _dyadic_s6(32, L=7)
    x, dl, Bt, Ct, A, Ds = args
    f64 = lambda v: v.astype(np.float64)
    y, hl = oracle.s6_fwd_state(*args, lib=lib)
    gr = oracle.s6_bwd(*args, dyv, dh_last=dhl, lib=lib)
    loss = math.fsum((y * f64(dyv)).ravel()) + math.fsum((hl * dhl).ravel())
    skip = math.fsum((f64(x) * f64(Ds) * f64(dyv)).ravel())
    chk = lambda a, b, what: abs(a - b) <= 1e-12 * max(1.0, abs(b))
    assert chk(math.fsum((f64(x) * gr["dx"]).ravel()), loss, "x"), "Euler identity in x"
    assert chk(math.fsum((f64(Bt) * gr["dBt"]).ravel()), loss - skip, "B"), "Euler identity in Bt"
    assert chk(math.fsum((f64(Ct) * gr["dCt"]).ravel()),
               math.fsum((y * f64(dyv)).ravel()) - skip, "C"), "Euler identity in Ct"
    assert np.allclose(gr["dDskip"], (f64(dyv) * f64(x)).sum(axis=(0, 1)), rtol=0, atol=1e-13), \
        "dDskip closed form"
    z = np.zeros_like(x)
    y0, hl0 = oracle.s6_fwd_state(z, dl, Bt, Ct, A, Ds, h0=h0, lib=lib)
    g0 = oracle.s6_bwd(z, dl, Bt, Ct, A, Ds, dyv, h0=h0, dh_last=dhl, lib=lib)
    loss0 = math.fsum((y0 * f64(dyv)).ravel()) + math.fsum((hl0 * dhl).ravel())
    assert chk(math.fsum((h0 * g0["dh0"]).ravel()), loss0, "h0"), "Euler identity in h0"


# ---------------------------------------------------------------- layer pins
def pin_layer_wiring(lib):
    """Zero projections give y = D x; selector weights make B_t, C_t slices of
    x and delta a constant, which must equal the scan run on those inputs
    directly; a transposed or swapped weight block fails."""
    g = _rng(40)
    B, L, D, N = 2, 9, 6, 3
    x = _dyadic(g, B * L * D, -2.0, 2.0, 6).reshape(B, L, D)
    A = -g.uniform(0.2, 2.0, (D, N)).astype(np.float32)
    Ds = g.standard_normal(D).astype(np.float32)
    bd = g.uniform(-2.0, 1.0, D).astype(np.float32)
    W = np.zeros((D + 2 * N, D), np.float32)
    y = oracle.layer_fwd(x, W, bd, A, Ds, lib=lib)
    assert np.array_equal(y, x.astype(np.float64) * Ds.astype(np.float64)), "zero projections"
    # B_t = x[..., [1, 4, 2]], C_t = x[..., [5, 0, 3]], delta = softplus(bd)
    for n, (cb, cc) in enumerate(((1, 5), (4, 0), (2, 3))):
        W[D + n, cb] = 1.0
        W[D + N + n, cc] = 1.0
    y = oracle.layer_fwd(x, W, bd, A, Ds, lib=lib)
    pre = np.broadcast_to(bd, (B, L, D)).copy()
    ref = oracle.s6_fwd(x, pre, np.ascontiguousarray(x[..., [1, 4, 2]]),
                        np.ascontiguousarray(x[..., [5, 0, 3]]), A, Ds, softplus=True, lib=lib)
    assert np.array_equal(y, ref), "selector projections"
    # proj_delta acts on x: W_delta = diag(1/4) gives delta = softplus(x/4 + bd)
    W[:D, :D] = np.eye(D, dtype=np.float32) / 4
    y = oracle.layer_fwd(x, W, bd, A, Ds, lib=lib)
    pre = (x.astype(np.float64) / 4 + bd).astype(np.float32)
    ref = oracle.s6_fwd(x, pre, np.ascontiguousarray(x[..., [1, 4, 2]]),
                        np.ascontiguousarray(x[..., [5, 0, 3]]), A, Ds, softplus=True, lib=lib)
    assert np.array_equal(y, ref), "delta projection and bias"


def pin_bf16_rounding(lib):
    """The bfloat16 rounding the layer oracle applies: values with at most 8
    significant bits are unchanged; halfway cases go to the even neighbour;
    otherwise the nearer neighbour."""
    r = oracle._round_bf16
    exact = np.array([1.0, -3.0, 0.75, 255.0, 2.0 ** -20 * 129, 1.5e-3 * 0 + 0.5])
    assert np.array_equal(r(exact), exact)
    # 1 + 2**-8 lies halfway between 1 and 1 + 2**-7: ties to even gives 1
    assert r(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert r(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2 * 2.0 ** -7  # tie, to even
    assert r(np.array([1.0 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1.0 + 2.0 ** -7
    assert r(np.array([-(1.0 + 2.0 ** -8 + 2.0 ** -30)]))[0] == -(1.0 + 2.0 ** -7)


def pin_layer_bf16_bias_before_rounding(lib):
    """Hand-worked bf16 layer step where the place of the bias decides the
    result. D = 2, N = 1, one step, x = (1, 1), W_delta row 0 = (1, 2^-8),
    row 1 = 0, W_B = W_C = (1, 0), b_delta = (2^-8, 0), A = -1, D = 0:
    proj_delta(x)_0 = 1 + 2^-8 and, with the bias, 1 + 2^-7, which bfloat16
    holds exactly; B_t = C_t = 1. A Linear layer adds the bias before its one
    rounding, so delta_0 = softplus(1 + 2^-7) and y_0 = delta_0 * B x_0 * C
    = softplus(1 + 2^-7); rounding first would give bf16(1 + 2^-8) = 1 (a
    tie, to even) and softplus(1 + 2^-8). Channel 1: y_1 = softplus(0) = ln 2.
    In float32 the same weights give the unrounded value."""
    x = np.array([[[1.0, 1.0]]], np.float32)
    W = np.array([[1.0, 2.0 ** -8], [0.0, 0.0], [1.0, 0.0], [1.0, 0.0]], np.float32)
    bd = np.array([2.0 ** -8, 0.0], np.float32)
    A = np.array([[-1.0], [-1.0]], np.float32)
    Ds = np.zeros(2, np.float32)
    sp = lambda v: math.log1p(math.exp(v))
    y = oracle.layer_fwd(x, W, bd, A, Ds, io="bf16", lib=lib)
    assert abs(y[0, 0, 0] - sp(1.0 + 2.0 ** -7)) <= 1e-12, "bf16: bias before the rounding"
    assert abs(y[0, 0, 1] - math.log(2.0)) <= 1e-12, "bf16: zero pre-activation"
    y = oracle.layer_fwd(x, W, bd, A, Ds, io="f32", lib=lib)
    assert abs(y[0, 0, 0] - sp(1.0 + 2.0 ** -7)) <= 1e-12, "f32: 1 + 2^-7 is exact too"


BWD_PINS = [pin_bwd_finite_differences, pin_bwd_finite_differences_softplus,
            pin_bwd_euler_and_skip, pin_layer_wiring, pin_bf16_rounding,
            pin_layer_bf16_bias_before_rounding]
ALL_PINS = ALL_PINS + BWD_PINS


def failures(lib) -> list[str]:
    """Names of the pins that fail (or crash) for this oracle library."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception as e:  # noqa: BLE001 - any failure counts
            bad.append(f"{pin.__name__}: {type(e).__name__}: {e}")
    return bad
