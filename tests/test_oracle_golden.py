"""The oracle against small examples worked by hand (tests/golden/)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_affine_hand_examples(oracle_lib):
    for case in _load("affine_hand.json")["cases"]:
        h = oracle.affine(np.array(case["a"], np.float32), np.array(case["b"], np.float32),
                          lib=oracle_lib)
        np.testing.assert_allclose(h, case["h"], rtol=0, atol=1e-15)


def test_s6_hand_examples(oracle_lib):
    for case in _load("s6_hand.json")["cases"]:
        L = len(case["x"])
        x = np.array(case["x"], np.float32).reshape(1, L, 1)
        dl = np.array(case["delta"], np.float32).reshape(1, L, 1)
        Bt = np.array(case["Bt"], np.float32).reshape(1, L, 1)
        Ct = np.array(case["Ct"], np.float32).reshape(1, L, 1)
        A = np.array(case["A"], np.float32)
        Ds = np.array(case["Dskip"], np.float32)
        y = oracle.s6_fwd(x, dl, Bt, Ct, A, Ds, lib=oracle_lib)
        np.testing.assert_allclose(y.reshape(L), case["y_fwd"], rtol=1e-15, atol=1e-15)
        if "y_bidir" in case:
            y = oracle.s6_bidir(x, dl, Bt, Ct, A, Ds, lib=oracle_lib)
            np.testing.assert_allclose(y.reshape(L), case["y_bidir"], rtol=1e-15, atol=1e-15)


def test_affine_from_state_hand_examples(oracle_lib):
    for case in _load("affine_hand.json")["cases_from_state"]:
        h = oracle.affine(np.array(case["a"], np.float32), np.array(case["b"], np.float32),
                          lib=oracle_lib, h0=case["h0"])
        np.testing.assert_allclose(h, case["h"], rtol=0, atol=1e-15)


def test_s6_backward_hand_examples(oracle_lib):
    for case in _load("s6_bwd_hand.json")["cases"]:
        L = len(case["x"])
        col = lambda k: np.array(case[k], np.float32).reshape(1, L, 1)
        A = np.array([[case["A"]]], np.float32)
        Ds = np.array([case["Dskip"]], np.float32)
        h0 = np.array([[[case["h0"]]]], np.float32)
        dhl = np.array([[[case["dh_last"]]]], np.float32)
        y, _ = oracle.s6_fwd_state(col("x"), col("delta"), col("Bt"), col("Ct"), A, Ds, h0=h0,
                                   lib=oracle_lib)
        np.testing.assert_allclose(y.reshape(L), case["y"], rtol=case["tol"], atol=case["tol"])
        g = oracle.s6_bwd(col("x"), col("delta"), col("Bt"), col("Ct"), A, Ds, col("dy"), h0=h0,
                          dh_last=dhl, lib=oracle_lib)
        for k in ("dx", "ddelta", "dBt", "dCt"):
            np.testing.assert_allclose(g[k].reshape(L), case[k], rtol=case["tol"],
                                       atol=case["tol"], err_msg=k)
        for k in ("dA", "dDskip", "dh0"):
            np.testing.assert_allclose(float(np.ravel(g[k])[0]), case[k], rtol=case["tol"],
                                       atol=case["tol"], err_msg=k)
