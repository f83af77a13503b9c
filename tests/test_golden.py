"""Oracle against the stored fixtures under tests/golden/."""

import json
import os

import numpy as np

import oracle
from layer_rnn_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_closed_form_fixtures():
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        mode, T = case["mode"], case["T"]
        H = len(case["h0"])
        G = oracle.GATES[mode]
        p = [dict(W_ih=np.zeros((G * H, 2)), W_hh=np.zeros((G * H, H)),
                  b_ih=np.zeros(G * H), b_hh=np.zeros(G * H))]
        x = np.random.default_rng(0).standard_normal((T, 1, 2))
        h0 = np.array(case["h0"]).reshape(1, 1, H)
        c0 = np.array(case["c0"]).reshape(1, 1, H) if "c0" in case else None
        y, hy, cy, _ = oracle.forward(mode, x, h0, c0, p, 1, False)
        np.testing.assert_allclose(hy.ravel(), case["expect_hy"], rtol=1e-15, atol=0)
        if "expect_cy" in case:
            np.testing.assert_allclose(cy.ravel(), case["expect_cy"], rtol=1e-15, atol=0)


def test_tiny_lstm_regression_fixture():
    with open(os.path.join(GOLDEN, "tiny_lstm_oracle.json")) as f:
        doc = json.load(f)
    cfg = wl.WORKLOADS["tiny_lstm"]
    inp = wl.make_inputs(cfg)
    out = oracle.run_flat(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"],
                          inp["x"], inp["h0"], inp["c0"], inp["w"], inp["dy"],
                          inp["dhy"], inp["dcy"])
    for k, v in doc["outputs"].items():
        np.testing.assert_allclose(out[k].ravel(), v, rtol=1e-13, atol=1e-15, err_msg=k)
