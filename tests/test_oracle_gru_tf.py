"""Pins for the oracle's TensorFlow-flavour GRU (mode "gru_tf": the reset gate
scales h before the candidate's recurrent matmul), against things other than
its own code:

* with the reset gate saturated at 1 the two flavours are the same function,
  so "gru_tf" must reproduce the PyTorch-flavour oracle (itself pinned against
  PyTorch's nn.GRU) in every output and gradient;
* on the first step from a zero state with b_hn = 0 both flavours give
  n = tanh(W_in x + b_in);
* central finite differences of the loss (also with variable lengths);
* on generic inputs the flavours differ;
* one step with two units evaluated exactly outside the oracle (literal
  expected values), and the unrolled scalar graph of tests/scalar_graph.py,
  which differentiates the TensorFlow equation node by node -- both tell
  W_hn (r * h) from r * (W_hn h).
"""

import numpy as np
import pytest

import oracle
from layer_rnn_gb300 import workloads as wl


def _case(L, bidir, T, N, I, H, seed, h0_std=0.3):
    cfg = wl.make_config("gru", L, bidir, T, N, I, H, "f32", h0_std, seed)
    inp = wl.make_inputs(cfg)
    inp["w"] = inp["w"] * 2.0
    return cfg, inp


def _run(mode, cfg, inp, w=None, lengths=None):
    return oracle.run_flat(mode, cfg["L"], cfg["bidir"], cfg["I"], cfg["H"], inp["x"],
                           inp["h0"], None, inp["w"] if w is None else w, inp["dy"],
                           inp["dhy"], None, lengths=lengths)


@pytest.mark.parametrize("L,bidir", [(1, False), (2, True), (3, False)])
def test_saturated_reset_gate_makes_the_flavours_agree(L, bidir):
    cfg, inp = _case(L, bidir, 5, 3, 4, 3, 91)
    H = cfg["H"]
    params = oracle.unflatten_weights(inp["w"], "gru", L, bidir, cfg["I"], H)
    for p in params:
        p["b_ih"][:H] = 80.0  # r = sigmoid(80 + ...) = 1 in float64
    w = oracle.flatten_weights(params, "gru", L, bidir, cfg["I"], H)
    a = _run("gru", cfg, inp, w)
    b = _run("gru_tf", cfg, inp, w)
    for k in ("y", "hy", "dx", "dh0", "dW"):
        np.testing.assert_allclose(b[k], a[k], rtol=1e-12, atol=1e-13, err_msg=k)


def test_first_step_from_zero_state_without_b_hn():
    cfg, inp = _case(1, True, 1, 4, 3, 5, 93, h0_std=0.0)
    H = cfg["H"]
    params = oracle.unflatten_weights(inp["w"], "gru", 1, True, cfg["I"], H)
    for p in params:
        p["b_hh"][2 * H:] = 0.0
    w = oracle.flatten_weights(params, "gru", 1, True, cfg["I"], H)
    a = _run("gru", cfg, inp, w)
    b = _run("gru_tf", cfg, inp, w)
    np.testing.assert_allclose(b["y"], a["y"], rtol=1e-14, atol=1e-15)
    # and the value itself: h' = (1 - z) * tanh(W_in x + b_in) from h = 0
    x = inp["x"][0]
    for d in range(2):
        p = params[d]
        gi = x @ p["W_ih"].T + p["b_ih"]
        z = oracle.sigmoid(gi[:, H:2 * H] + p["b_hh"][H:2 * H])
        np.testing.assert_allclose(b["y"][0, :, d * H:(d + 1) * H],
                                   (1 - z) * np.tanh(gi[:, 2 * H:]), rtol=1e-14, atol=1e-15)


def test_flavours_differ_on_generic_inputs():
    cfg, inp = _case(1, False, 3, 2, 3, 3, 95)
    a = _run("gru", cfg, inp)
    b = _run("gru_tf", cfg, inp)
    assert np.abs(a["y"] - b["y"]).max() > 1e-3


@pytest.mark.parametrize("L,bidir,lengths", [(1, False, None), (2, True, None),
                                             (1, True, [3, 1])])
def test_gru_tf_gradients_match_finite_differences(L, bidir, lengths):
    cfg, inp = _case(L, bidir, 3, 2, 2, 2, 97)
    out = _run("gru_tf", cfg, inp, lengths=lengths)
    params_of = lambda w: oracle.unflatten_weights(w, "gru_tf", L, bidir, cfg["I"], cfg["H"])

    def loss_of(d):
        y, hy, cy, _ = oracle.forward("gru_tf", d["x"], d["h0"], None, params_of(d["w"]), L,
                                      bidir, lengths)
        return oracle.loss(y, hy, cy, d["dy"], d["dhy"], None)

    grads = dict(x=out["dx"], h0=out["dh0"], w=out["dW"])
    eps = 1e-6
    for name, g in grads.items():
        base = inp[name]
        num = np.zeros(base.size)
        for e in range(base.size):
            plus, minus = dict(inp), dict(inp)
            bp, bm = base.copy().ravel(), base.copy().ravel()
            bp[e] += eps
            bm[e] -= eps
            plus[name], minus[name] = bp.reshape(base.shape), bm.reshape(base.shape)
            num[e] = (loss_of(plus) - loss_of(minus)) / (2 * eps)
        scale = max(1.0, np.abs(num).max())
        np.testing.assert_allclose(g.ravel(), num, rtol=0, atol=2e-7 * scale,
                                   err_msg="gradient of %s" % name)


def test_one_step_by_hand_two_units():
    """One TensorFlow-flavour step ("rnn training example?", the TensorFlow GRU
    equations: n = tanh(W_in x + b_in + W_hn (r * h) + b_hn)) with H = 2, a
    full (non-diagonal) W_hn, both reset gates strictly between 0 and 1, h != 0
    and b_hn != 0.  The expected values are that equation evaluated exactly
    (rational inputs, 25 significant digits) outside the oracle and written
    here as literals.  At H = 1 the product would be a scalar and could not
    tell W_hn (r * h) from r * (W_hn h); here the two differ in the second
    decimal."""
    x = 0.7
    h = [-0.4, 0.6]
    W_ih = np.array([0.3, -0.2, 0.5, 0.1, -0.3, 0.4]).reshape(6, 1)  # r0 r1 z0 z1 n0 n1
    W_hh = np.array([[-0.6, 0.4], [0.2, 0.5],      # W_hr
                     [-0.3, 0.25], [0.1, -0.4],    # W_hz
                     [0.7, -0.9], [0.5, 0.8]])     # W_hn
    b_ih = np.array([0.05, -0.1, 0.2, 0.0, -0.25, 0.15])
    b_hh = np.array([0.1, 0.3, -0.2, 0.15, 0.4, -0.3])
    p = [dict(W_ih=W_ih, W_hh=W_hh, b_ih=b_ih, b_hh=b_hh)]
    y, hy, _, cache = oracle.forward("gru_tf", np.array([[[x]]]), np.array([[h]]), None, p, 1,
                                     False)
    rec = cache["tapes"][0][0]  # layer 0, direction 0, step 0
    r_exact = [0.6984652160025387754745268, 0.5695462239392290158986344]
    z_exact = [0.6502185485738270628302611, 0.4850044983805899277070476]
    n_exact = [-0.5102925359619838186435149, 0.2577428642137648597495013]
    h_exact = [-0.4385782833102560749224672, 0.4237391146729452878227584]
    np.testing.assert_allclose(y[0, 0], h_exact, rtol=0, atol=1e-15)
    np.testing.assert_allclose(hy[0, 0], h_exact, rtol=0, atol=1e-15)
    np.testing.assert_allclose(rec["r"][0], r_exact, rtol=0, atol=1e-15)
    np.testing.assert_allclose(rec["z"][0], z_exact, rtol=0, atol=1e-15)
    np.testing.assert_allclose(rec["n"][0], n_exact, rtol=0, atol=1e-15)
    # the candidates of the other placements of r differ by far more than the
    # tolerance: r * (W_hn h + b_hn) (PyTorch flavour) and r * (W_hn h) + b_hn
    for wrong in ([-0.6371464663287032615489948, 0.3957580063783218927540946],
                  [-0.5599370473363979272877778, 0.2816496370598662883406038]):
        assert np.abs(np.array(wrong) - np.array(n_exact)).max() > 1e-2
