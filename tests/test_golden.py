"""The oracle still reproduces the frozen regression fixtures (CPU only)."""
import json
import os

import numpy as np

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def test_fwd_bwd_fixture():
    g = _load("oracle_fwd_bwd_b1_t8_d4_w4.json")
    B, T, D, W = g["shape"]
    x = np.array(g["x"]).reshape(B, T, D)
    dy = np.array(g["dy"]).reshape(B, T, D)
    w = np.array(g["w"]).reshape(D, W)
    b = np.array(g["bias"])
    y = oracle.fwd(x, w, b)
    dx, dw, db = oracle.bwd(x, dy, w, b)
    np.testing.assert_allclose(y.ravel(), g["y"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dx.ravel(), g["dx"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dw.ravel(), g["dw"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(db.ravel(), g["dbias"], rtol=0, atol=1e-15)


def test_decode_fixture():
    g = _load("oracle_decode_s6_n3_d4_w4.json")
    S, N, D, W = g["shape"]
    st = np.array(g["state_bits"], np.uint16).reshape(S, D, W - 1)
    x = np.array(g["x_bits"], np.uint16).reshape(N, D)
    status, y, new = oracle.update(x, st, np.array(g["state_indices"], np.int32),
                                   np.array(g["w"]).reshape(D, W), np.array(g["bias"]))
    assert status == 0
    np.testing.assert_allclose(y.ravel(), g["y"], rtol=0, atol=1e-15)
    assert np.array_equal(new.ravel(), np.array(g["new_state_bits"], np.uint16))
