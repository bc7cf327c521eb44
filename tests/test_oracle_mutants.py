"""Plants one mistake at a time in a copy of the oracle and checks that the
pins catch it (CPU only). The real oracle.c is never modified: each mutant is
a rewritten copy compiled into a temporary directory."""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text to find, replacement, occurrence: 1 = first only, 0 = all)
MUTANTS = [
    ("affine_swapped_operands",
     "state = (double)a[t] * state + (double)b[t];",
     "state = (double)b[t] * state + (double)a[t];", 1),
    ("affine_index_off_by_one",
     "state = (double)a[t] * state",
     "state = (double)a[t > 0 ? t - 1 : 0] * state", 1),
    ("affine_store_before_update",
     "state = (double)a[t] * state + (double)b[t];\n        h[t] = state;",
     "h[t] = state;\n        state = (double)a[t] * state + (double)b[t];", 1),
    ("affine_h0_ignored",
     "double state = h0;", "double state = 0.0;", 1),
    ("affine_h0_added_after_first_step",
     "double state = h0;\n    for (int64_t t = 0; t < n; ++t) {\n        state = (double)a[t] * state + (double)b[t];",
     "double state = 0.0;\n    for (int64_t t = 0; t < n; ++t) {\n        state = (double)a[t] * state + (double)b[t] + (t == 0 ? h0 : 0.0);", 1),
    ("s6_dropped_skip_term",
     "y[t * ystride] = acc + xv * Dd;", "y[t * ystride] = acc;", 1),
    ("s6_exp_sign",
     "exp(dl * (double)j->A[d * N + n])", "exp(-dl * (double)j->A[d * N + n])", 1),
    ("s6_A_transposed",
     "j->A[d * N + n]", "j->A[n * D + d]", 0),
    ("s6_B_index_shifted",
     "const int64_t bi = (b * L + t) * N;       /* B_t[b, t, :] */",
     "const int64_t bi = (b * L + (t > 0 ? t - 1 : 0)) * N;", 1),
    ("s6_readout_uses_B",
     "acc += h[n] * (double)j->Ct[bi + n];", "acc += h[n] * (double)j->Bt[bi + n];", 1),
    ("s6_softplus_skipped",
     "if (j->softplus)\n            dl = oracle_softplus_f64(dl);", "", 1),
    ("s6_softplus_formula",
     "return log1p(exp(v));", "return log(exp(v));", 1),
    ("s6_x_dropped_from_input",
     "const double x_db = xv * dB;", "const double x_db = dB;", 1),
    ("s6_readout_before_update",
     "h[n] = dA * h[n] + x_db;\n            acc += h[n] * (double)j->Ct[bi + n];",
     "acc += h[n] * (double)j->Ct[bi + n];\n            h[n] = dA * h[n] + x_db;", 1),
    ("bidir_reverse_runs_forward",
     "for (int64_t t = L - 1; t >= 0; --t)", "for (int64_t t = 0; t < L; ++t)", 1),
    ("bidir_reverse_drops_skip_term",
     "y[t * ystride] += acc + xv * Dd;", "y[t * ystride] += acc;", 1),
    ("state_h0_ignored",
     "h[n] = j->h0 ? j->h0[(b * D + d) * N + n] : 0.0;", "h[n] = 0.0;", 1),
    ("state_h0_index_transposed",
     "h[n] = j->h0 ? j->h0[(b * D + d) * N + n] : 0.0;",
     "h[n] = j->h0 ? j->h0[(b * N + n) * D + d] : 0.0;", 1),
    ("state_hlast_is_h0",
     "j->hlast[(b * D + d) * N + n] = h[n];",
     "j->hlast[(b * D + d) * N + n] = j->h0 ? j->h0[(b * D + d) * N + n] : 0.0;", 1),
    ("bwd_hprev_is_h_t",
     "const double ht = hs[(t + 1) * N + n], hprev = hs[t * N + n];",
     "const double ht = hs[(t + 1) * N + n], hprev = hs[(t + 1) * N + n];", 1),
    ("bwd_ddelta_drops_A",
     "gdl += lam * (Bv * xv + hprev * dA * An);", "gdl += lam * (Bv * xv + hprev * dA);", 1),
    ("bwd_sigmoid_sign",
     "gdl / (1.0 + exp(-v))", "gdl / (1.0 + exp(v))", 1),
    ("bwd_dB_drops_delta",
     "j->dBt[bi + n] += lam * dl * xv;", "j->dBt[bi + n] += lam * xv;", 1),
    ("bwd_adjoint_not_decayed",
     "g[n] = lam * dA;", "g[n] = lam;", 1),
    ("bwd_dC_uses_adjoint",
     "j->dCt[bi + n] += gy * ht;", "j->dCt[bi + n] += lam * ht;", 1),
    ("bidir_reverse_state_not_reset",
     "    /* reverse: t = L-1 .. 0, h_rev[t] = dA[t]*h_rev[t+1] + dBx[t] */\n"
     "    for (int64_t n = 0; n < N; ++n)\n        h[n] = 0.0;\n",
     "    /* reverse: t = L-1 .. 0, h_rev[t] = dA[t]*h_rev[t+1] + dBx[t] */\n", 1),
]


@pytest.mark.parametrize("name,find,repl,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, find, repl, occ, tmp_path):
    text = open(SRC).read()
    assert find in text, f"mutation anchor for {name} not found in oracle.c"
    mutated = text.replace(find, repl) if occ == 0 else text.replace(find, repl, occ)
    assert mutated != text
    src = tmp_path / "oracle_mutant.c"
    src.write_text(mutated)
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "libmutant.so"), force=True))
    bad = oracle_pins.failures(lib)
    assert bad, f"planted mistake '{name}' passed every pin"
