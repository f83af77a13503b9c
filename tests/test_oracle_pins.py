"""Pins for the float64 oracle against things other than itself.

* closed forms that follow from the cell equations at special points;
* saturated gates;
* a naive unrolled scalar graph with generic autodiff (``scalar_graph``);
* central finite differences of the loss;
* PyTorch's own CPU float64 nn.LSTM / nn.GRU / nn.RNN (PyTorch's GRU is the
  flavour "rnn training example?" (oneDNN issue #218) names as the reference);
* structural invariants (bidirection as time reversal, stacking as chaining);
* a negative test against the TensorFlow GRU variant quoted on the same page.
"""

import math

import numpy as np
import pytest

import oracle
from layer_rnn_gb300 import workloads as wl
from tests import scalar_graph


def _small(mode, L=1, bidir=False, T=3, N=2, I=3, H=2, seed=7, h0_std=0.3):
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, "f32", h0_std, seed)
    inp = wl.make_inputs(cfg)
    # widen the weights so the nonlinearities are exercised away from zero
    inp["w"] = inp["w"] * 2.0
    return cfg, inp


def _params(cfg, w):
    return oracle.unflatten_weights(w, cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"])


def _run(cfg, inp):
    return oracle.run_flat(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"],
                           inp["x"], inp["h0"], inp["c0"], inp["w"], inp["dy"],
                           inp["dhy"], inp["dcy"])


# ----------------------------------------------------------------------------
# closed forms at zero weights
# ----------------------------------------------------------------------------

def _zero_weight_case(mode, T=6, N=3, I=4, H=5, bidir=False):
    cfg = wl.make_config(mode, 1, bidir, T, N, I, H, "f32", 0.7, 11)
    inp = wl.make_inputs(cfg)
    inp["w"] = np.zeros_like(inp["w"])
    return cfg, inp


def test_gru_zero_weights_halves_state():
    # r = z = 1/2 and n = tanh(0) = 0, so h' = h / 2 and h_T = 2^-T h0 exactly
    cfg, inp = _zero_weight_case("gru")
    out = _run(cfg, inp)
    h0 = inp["h0"][0]
    for t in range(cfg["T"]):
        assert np.array_equal(out["y"][t], h0 * 2.0 ** -(t + 1))
    assert np.array_equal(out["hy"][0], h0 * 2.0 ** -cfg["T"])


def test_gru_zero_weights_backward_closed_form():
    # with h_t = 2^-(t+1) h0, d loss / d h0 = sum_t 2^-(t+1) dy_t + 2^-T dhy
    cfg, inp = _zero_weight_case("gru")
    out = _run(cfg, inp)
    T = cfg["T"]
    expect = sum(inp["dy"][t] * 2.0 ** -(t + 1) for t in range(T)) + inp["dhy"][0] * 2.0 ** -T
    np.testing.assert_allclose(out["dh0"][0], expect, rtol=1e-14, atol=1e-15)
    # W_ih = 0 means x has no influence
    assert np.all(out["dx"] == 0)


def test_lstm_zero_weights_closed_form():
    # i = f = o = 1/2, g = 0: c_t = 2^-(t+1) c0 and h_t = tanh(c_t) / 2
    cfg, inp = _zero_weight_case("lstm")
    out = _run(cfg, inp)
    c0 = inp["c0"][0]
    T = cfg["T"]
    for t in range(T):
        c_t = c0 * 2.0 ** -(t + 1)
        np.testing.assert_allclose(out["y"][t], 0.5 * np.tanh(c_t), rtol=1e-15, atol=0)
    assert np.array_equal(out["cy"][0], c0 * 2.0 ** -T)
    # derivative of that trajectory: d h_t / d c0 = (1 - tanh(c_t)^2) 2^-(t+2)
    dc0 = inp["dcy"][0] * 2.0 ** -T
    for t in range(T):
        c_t = c0 * 2.0 ** -(t + 1)
        dc0 = dc0 + inp["dy"][t] * (1 - np.tanh(c_t) ** 2) * 2.0 ** -(t + 2)
    dc0 = dc0 + inp["dhy"][0] * (1 - np.tanh(c0 * 2.0 ** -T) ** 2) * 2.0 ** -(T + 1)
    np.testing.assert_allclose(out["dc0"][0], dc0, rtol=1e-13, atol=1e-15)
    # h0 has no path to the loss when W_hh = 0
    assert np.all(out["dh0"] == 0)


def test_rnn_zero_weights_is_zero():
    cfg, inp = _zero_weight_case("rnn_tanh")
    out = _run(cfg, inp)
    assert np.all(out["y"] == 0) and np.all(out["hy"] == 0)
    # d tanh / d a at a = 0 is 1: db_ih = db_hh = sum over t, n of dy (+ dhy at t = T-1)
    p = _params(cfg, out["dW"])[0]
    expect = inp["dy"][:, :, :].sum(axis=(0, 1)) + inp["dhy"][0].sum(axis=0)
    np.testing.assert_allclose(p["b_ih"], expect, rtol=1e-13)
    np.testing.assert_allclose(p["b_hh"], expect, rtol=1e-13)


def test_zero_weight_reverse_direction():
    # the backward direction starts at t = T-1: y_bwd[t] = 2^-(T-t) h0
    cfg, inp = _zero_weight_case("gru", bidir=True)
    out = _run(cfg, inp)
    T, H = cfg["T"], cfg["H"]
    h0b = inp["h0"][1]
    for t in range(T):
        assert np.array_equal(out["y"][t][:, H:], h0b * 2.0 ** -(T - t))
    assert np.array_equal(out["hy"][1], h0b * 2.0 ** -T)


# ----------------------------------------------------------------------------
# saturated gates
# ----------------------------------------------------------------------------

def test_gru_saturated_update_gate_keeps_state():
    cfg, inp = _small("gru", T=5, H=3)
    p = _params(cfg, inp["w"])
    H = cfg["H"]
    p[0]["b_ih"][H:2 * H] = 40.0     # z = sigmoid(>= 40 - small) ~ 1
    w = oracle.flatten_weights(p, "gru", 1, False, cfg["I"], H)
    out = oracle.run_flat("gru", 1, False, cfg["I"], H, inp["x"], inp["h0"], None, w,
                          inp["dy"], inp["dhy"], None)
    np.testing.assert_allclose(out["hy"][0], inp["h0"][0], atol=1e-15)


def test_lstm_saturated_gates_keep_cell():
    cfg, inp = _small("lstm", T=5, H=3)
    p = _params(cfg, inp["w"])
    H = cfg["H"]
    p[0]["b_ih"][0:H] = -40.0        # i ~ 0
    p[0]["b_ih"][H:2 * H] = 40.0     # f ~ 1
    w = oracle.flatten_weights(p, "lstm", 1, False, cfg["I"], H)
    out = oracle.run_flat("lstm", 1, False, cfg["I"], H, inp["x"], inp["h0"], inp["c0"], w,
                          inp["dy"], inp["dhy"], inp["dcy"])
    np.testing.assert_allclose(out["cy"][0], inp["c0"][0], atol=1e-15)


def test_single_scalar_step_by_hand():
    # T = N = I = H = 1: every gate written out with math.* on scalars
    x, h, c = 0.7, -0.4, 0.25
    wi = [0.3, -0.2, 0.5, 0.1]
    wh = [-0.6, 0.4, 0.2, -0.3]
    bi = [0.05, -0.1, 0.2, 0.0]
    bh = [0.1, 0.3, -0.2, 0.15]
    sg = lambda a: 1.0 / (1.0 + math.exp(-a))
    a = [wi[k] * x + bi[k] + wh[k] * h + bh[k] for k in range(4)]
    c1 = sg(a[1]) * c + sg(a[0]) * math.tanh(a[2])
    h1 = sg(a[3]) * math.tanh(c1)
    p = [dict(W_ih=np.array(wi).reshape(4, 1), W_hh=np.array(wh).reshape(4, 1),
              b_ih=np.array(bi), b_hh=np.array(bh))]
    y, hy, cy, _ = oracle.forward("lstm", np.array([[[x]]]), np.array([[[h]]]),
                                  np.array([[[c]]]), p, 1, False)
    assert abs(y[0, 0, 0] - h1) < 1e-15 and abs(cy[0, 0, 0] - c1) < 1e-15
    # GRU with the first three gate rows
    r = sg(wi[0] * x + bi[0] + wh[0] * h + bh[0])
    z = sg(wi[1] * x + bi[1] + wh[1] * h + bh[1])
    n = math.tanh(wi[2] * x + bi[2] + r * (wh[2] * h + bh[2]))
    hg = n + z * (h - n)
    pg = [dict(W_ih=np.array(wi[:3]).reshape(3, 1), W_hh=np.array(wh[:3]).reshape(3, 1),
               b_ih=np.array(bi[:3]), b_hh=np.array(bh[:3]))]
    y, hy, _, _ = oracle.forward("gru", np.array([[[x]]]), np.array([[[h]]]), None, pg, 1, False)
    assert abs(y[0, 0, 0] - hg) < 1e-15
    # tanh RNN with the first gate row
    hr = math.tanh(wi[0] * x + bi[0] + wh[0] * h + bh[0])
    pr = [dict(W_ih=np.array(wi[:1]).reshape(1, 1), W_hh=np.array(wh[:1]).reshape(1, 1),
               b_ih=np.array(bi[:1]), b_hh=np.array(bh[:1]))]
    y, _, _, _ = oracle.forward("rnn_tanh", np.array([[[x]]]), np.array([[[h]]]), None, pr, 1, False)
    assert abs(y[0, 0, 0] - hr) < 1e-15


# ----------------------------------------------------------------------------
# unrolled scalar graph with generic autodiff
# ----------------------------------------------------------------------------

UNROLLED_CASES = [
    ("lstm", 1, False), ("gru", 1, False), ("rnn_tanh", 1, False),
    ("lstm", 2, True), ("gru", 2, True), ("rnn_tanh", 2, True),
    ("gru_tf", 1, False), ("gru_tf", 2, True),
]


@pytest.mark.parametrize("mode,L,bidir", UNROLLED_CASES)
def test_oracle_matches_unrolled_graph(mode, L, bidir):
    cfg, inp = _small(mode, L, bidir)
    out = _run(cfg, inp)
    params = _params(cfg, inp["w"])
    ref = scalar_graph.run(mode, L, bidir, inp["x"], inp["h0"], inp["c0"], params,
                           inp["dy"], inp["dhy"], inp["dcy"])
    tol = dict(rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out["y"], np.array(ref["y"]), **tol)
    np.testing.assert_allclose(out["hy"], np.array(ref["hy"]), **tol)
    np.testing.assert_allclose(out["dx"], np.array(ref["dx"]), **tol)
    np.testing.assert_allclose(out["dh0"], np.array(ref["dh0"]), **tol)
    if mode == "lstm":
        np.testing.assert_allclose(out["cy"], np.array(ref["cy"]), **tol)
        np.testing.assert_allclose(out["dc0"], np.array(ref["dc0"]), **tol)
    dp = _params(cfg, out["dW"])
    for k in range(len(dp)):
        for name in ("W_ih", "W_hh", "b_ih", "b_hh"):
            np.testing.assert_allclose(dp[k][name], np.array(ref["dparams"][k][name]), **tol)


# ----------------------------------------------------------------------------
# central finite differences of the loss
# ----------------------------------------------------------------------------

def _loss_of(cfg, inp):
    params = _params(cfg, inp["w"])
    y, hy, cy, _ = oracle.forward(cfg["mode"], inp["x"], inp["h0"], inp["c0"], params,
                                  cfg["L"], cfg["bidir"])
    return oracle.loss(y, hy, cy, inp["dy"], inp["dhy"], inp["dcy"])


FD_CASES = [("lstm", 1, False), ("gru", 1, False), ("rnn_tanh", 1, False),
            ("lstm", 2, True), ("gru", 2, True)]


@pytest.mark.parametrize("mode,L,bidir", FD_CASES)
def test_oracle_gradients_match_finite_differences(mode, L, bidir):
    cfg, inp = _small(mode, L, bidir, T=3, N=2, I=2, H=2, seed=21)
    out = _run(cfg, inp)
    grads = dict(x=out["dx"], h0=out["dh0"], w=out["dW"])
    if mode == "lstm":
        grads["c0"] = out["dc0"]
    eps = 1e-6
    for name, g in grads.items():
        base = inp[name]
        num = np.zeros(base.size)
        for e in range(base.size):
            plus = dict(inp)
            minus = dict(inp)
            bp = base.copy().ravel()
            bm = base.copy().ravel()
            bp[e] += eps
            bm[e] -= eps
            plus[name] = bp.reshape(base.shape)
            minus[name] = bm.reshape(base.shape)
            num[e] = (_loss_of(cfg, plus) - _loss_of(cfg, minus)) / (2 * eps)
        scale = max(1.0, np.abs(num).max())
        np.testing.assert_allclose(g.ravel(), num, rtol=0, atol=2e-7 * scale,
                                   err_msg="gradient of %s" % name)


# ----------------------------------------------------------------------------
# PyTorch float64 CPU modules (independent implementation)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode,L,bidir", [("lstm", 1, False), ("gru", 1, False),
                                          ("rnn_tanh", 1, False), ("lstm", 2, True),
                                          ("gru", 3, True), ("rnn_tanh", 2, True)])
def test_oracle_matches_torch_modules(mode, L, bidir):
    torch = pytest.importorskip("torch")
    cfg, inp = _small(mode, L, bidir, T=4, N=3, I=5, H=4, seed=31)
    out = _run(cfg, inp)
    params = _params(cfg, inp["w"])
    kw = dict(input_size=cfg["I"], hidden_size=cfg["H"], num_layers=L,
              bidirectional=bidir, bias=True)
    if mode == "lstm":
        m = torch.nn.LSTM(**kw)
    elif mode == "gru":
        m = torch.nn.GRU(**kw)
    else:
        m = torch.nn.RNN(nonlinearity="tanh", **kw)
    m = m.double()
    D = 2 if bidir else 1
    with torch.no_grad():
        for l in range(L):
            for d in range(D):
                sfx = "_l%d%s" % (l, "_reverse" if d == 1 else "")
                p = params[l * D + d]
                getattr(m, "weight_ih" + sfx).copy_(torch.from_numpy(p["W_ih"]))
                getattr(m, "weight_hh" + sfx).copy_(torch.from_numpy(p["W_hh"]))
                getattr(m, "bias_ih" + sfx).copy_(torch.from_numpy(p["b_ih"]))
                getattr(m, "bias_hh" + sfx).copy_(torch.from_numpy(p["b_hh"]))
    x = torch.from_numpy(inp["x"]).requires_grad_(True)
    h0 = torch.from_numpy(inp["h0"]).requires_grad_(True)
    if mode == "lstm":
        c0 = torch.from_numpy(inp["c0"]).requires_grad_(True)
        y, (hy, cy) = m(x, (h0, c0))
        loss = (y * torch.from_numpy(inp["dy"])).sum() + (hy * torch.from_numpy(inp["dhy"])).sum() \
            + (cy * torch.from_numpy(inp["dcy"])).sum()
    else:
        y, hy = m(x, h0)
        loss = (y * torch.from_numpy(inp["dy"])).sum() + (hy * torch.from_numpy(inp["dhy"])).sum()
    loss.backward()
    tol = dict(rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["y"], y.detach().numpy(), **tol)
    np.testing.assert_allclose(out["hy"], hy.detach().numpy(), **tol)
    np.testing.assert_allclose(out["dx"], x.grad.numpy(), **tol)
    np.testing.assert_allclose(out["dh0"], h0.grad.numpy(), **tol)
    if mode == "lstm":
        np.testing.assert_allclose(out["cy"], cy.detach().numpy(), **tol)
        np.testing.assert_allclose(out["dc0"], c0.grad.numpy(), **tol)
    dp = _params(cfg, out["dW"])
    for l in range(L):
        for d in range(D):
            sfx = "_l%d%s" % (l, "_reverse" if d == 1 else "")
            for name, tname in (("W_ih", "weight_ih"), ("W_hh", "weight_hh"),
                                ("b_ih", "bias_ih"), ("b_hh", "bias_hh")):
                np.testing.assert_allclose(dp[l * D + d][name],
                                           getattr(m, tname + sfx).grad.numpy(), **tol)


# ----------------------------------------------------------------------------
# structural invariants and the GRU flavour
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["lstm", "gru", "rnn_tanh"])
def test_backward_direction_is_time_reversed_forward(mode):
    cfg, inp = _small(mode, 1, True, T=5, N=2, I=3, H=3)
    params = _params(cfg, inp["w"])
    y, hy, cy, _ = oracle.forward(mode, inp["x"], inp["h0"], inp["c0"], params, 1, True)
    H = cfg["H"]
    c0 = inp["c0"][1:2] if inp["c0"] is not None else None
    yr, hyr, cyr, _ = oracle.forward(mode, inp["x"][::-1], inp["h0"][1:2], c0,
                                     [params[1]], 1, False)
    np.testing.assert_allclose(y[:, :, H:], yr[::-1], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(hy[1], hyr[0], rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("mode", ["lstm", "gru"])
def test_stack_is_chain_of_single_layers(mode):
    cfg, inp = _small(mode, 2, True, T=4, N=2, I=3, H=3)
    params = _params(cfg, inp["w"])
    y, hy, cy, _ = oracle.forward(mode, inp["x"], inp["h0"], inp["c0"], params, 2, True)
    c0 = inp["c0"]
    y1, _, _, _ = oracle.forward(mode, inp["x"], inp["h0"][0:2],
                                 c0[0:2] if c0 is not None else None, params[0:2], 1, True)
    y2, hy2, _, _ = oracle.forward(mode, y1, inp["h0"][2:4],
                                   c0[2:4] if c0 is not None else None, params[2:4], 1, True)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(hy[2:4], hy2)


def test_gru_is_not_the_tensorflow_variant():
    # TF applies the reset gate before the matmul: n = tanh(W_in x + b_in + W_hn (r*h) + b_hn)
    cfg, inp = _small("gru", 1, False, T=1, N=2, I=3, H=3)
    p = _params(cfg, inp["w"])[0]
    x, h = inp["x"][0], inp["h0"][0]
    H = cfg["H"]
    sg = oracle.sigmoid
    gi = x @ p["W_ih"].T + p["b_ih"]
    r = sg(gi[:, :H] + h @ p["W_hh"][:H].T + p["b_hh"][:H])
    z = sg(gi[:, H:2 * H] + h @ p["W_hh"][H:2 * H].T + p["b_hh"][H:2 * H])
    n_tf = np.tanh(gi[:, 2 * H:] + (r * h) @ p["W_hh"][2 * H:].T + p["b_hh"][2 * H:])
    h_tf = (1 - z) * n_tf + z * h
    y, _, _, _ = oracle.forward("gru", inp["x"], inp["h0"], None, [p], 1, False)
    assert np.abs(y[0] - h_tf).max() > 1e-3


def test_weight_flatten_roundtrip_is_exact():
    cfg, inp = _small("lstm", 3, True, I=5, H=4)
    params = _params(cfg, inp["w"])
    back = oracle.flatten_weights(params, "lstm", 3, True, 5, 4)
    assert np.array_equal(back, inp["w"])
    # layer 0 takes I inputs, layers above take 2H
    assert params[0]["W_ih"].shape == (16, 5) and params[2]["W_ih"].shape == (16, 8)
