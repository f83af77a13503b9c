"""Pins for the oracle's inter-layer dropout (the masks are passed in), against
things other than the oracle's own masking:

* all-ones masks with dropout 0 give exactly the plain oracle;
* single-layer PyTorch float64 modules chained with the same masks between
  them (what nn.LSTM / nn.GRU / nn.RNN with num_layers > 1 and dropout do in
  training, with their own random masks), forward and every gradient through
  PyTorch's autograd;
* central finite differences of the loss;
* a feature that is dropped everywhere has no influence on the layer above:
  that layer's W_ih column for it gets exactly zero gradient.
"""

import numpy as np
import pytest

import oracle
from layer_rnn_gb300 import workloads as wl


def _case(mode, L, bidir, T, N, I, H, seed):
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, "f32", 0.3, seed)
    inp = wl.make_inputs(cfg)
    inp["w"] = inp["w"] * 2.0
    return cfg, inp


def _masks(cfg, keep_prob, seed):
    D = 2 if cfg["bidir"] else 1
    rng = np.random.default_rng(seed)
    return [(rng.random((cfg["T"], cfg["N"], D * cfg["H"])) < keep_prob).astype(np.float64)
            for _ in range(cfg["L"] - 1)]


def _run(cfg, inp, p, masks):
    return oracle.run_flat(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"],
                           inp["x"], inp["h0"], inp["c0"], inp["w"], inp["dy"],
                           inp["dhy"], inp["dcy"], dropout=p, masks=masks)


CASES = [("lstm", 2, False), ("gru", 3, True), ("rnn_tanh", 2, True), ("lstm", 3, True)]


@pytest.mark.parametrize("mode,L,bidir", CASES)
def test_ones_masks_without_dropout_are_the_plain_oracle(mode, L, bidir):
    cfg, inp = _case(mode, L, bidir, 4, 3, 5, 3, 61)
    D = 2 if bidir else 1
    ones = [np.ones((4, 3, D * 3)) for _ in range(L - 1)]
    a = _run(cfg, inp, 0.0, None)
    b = _run(cfg, inp, 0.0, ones)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("mode,L,bidir", CASES)
def test_matches_chained_torch_layers_with_the_same_masks(mode, L, bidir):
    torch = pytest.importorskip("torch")
    T, N, I, H = 5, 3, 4, 3
    cfg, inp = _case(mode, L, bidir, T, N, I, H, 67)
    p = 0.4
    masks = _masks(cfg, 1.0 - p, 71)
    out = _run(cfg, inp, p, masks)
    params = oracle.unflatten_weights(inp["w"], mode, L, bidir, I, H)
    D = 2 if bidir else 1
    lstm = mode == "lstm"
    layers = []
    for l in range(L):
        kw = dict(input_size=I if l == 0 else D * H, hidden_size=H, num_layers=1,
                  bidirectional=bidir, bias=True)
        m = (torch.nn.LSTM(**kw) if lstm else torch.nn.GRU(**kw) if mode == "gru"
             else torch.nn.RNN(nonlinearity="tanh", **kw)).double()
        with torch.no_grad():
            for d in range(D):
                sfx = "_l0" + ("_reverse" if d == 1 else "")
                q = params[l * D + d]
                getattr(m, "weight_ih" + sfx).copy_(torch.from_numpy(q["W_ih"]))
                getattr(m, "weight_hh" + sfx).copy_(torch.from_numpy(q["W_hh"]))
                getattr(m, "bias_ih" + sfx).copy_(torch.from_numpy(q["b_ih"]))
                getattr(m, "bias_hh" + sfx).copy_(torch.from_numpy(q["b_hh"]))
        layers.append(m)
    x = torch.from_numpy(inp["x"]).requires_grad_(True)
    h0 = torch.from_numpy(inp["h0"]).requires_grad_(True)
    c0 = torch.from_numpy(inp["c0"]).requires_grad_(True) if lstm else None
    cur, hys, cys = x, [], []
    for l, m in enumerate(layers):
        hs = h0[l * D:(l + 1) * D]
        if lstm:
            cur, (hl, cl) = m(cur, (hs, c0[l * D:(l + 1) * D]))
            cys.append(cl)
        else:
            cur, hl = m(cur, hs)
        hys.append(hl)
        if l < L - 1:
            cur = cur * torch.from_numpy(masks[l]) / (1.0 - p)
    hy = torch.cat(hys, 0)
    loss = (cur * torch.from_numpy(inp["dy"])).sum() + (hy * torch.from_numpy(inp["dhy"])).sum()
    if lstm:
        cy = torch.cat(cys, 0)
        loss = loss + (cy * torch.from_numpy(inp["dcy"])).sum()
    loss.backward()
    tol = dict(rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["y"], cur.detach().numpy(), **tol)
    np.testing.assert_allclose(out["hy"], hy.detach().numpy(), **tol)
    np.testing.assert_allclose(out["dx"], x.grad.numpy(), **tol)
    np.testing.assert_allclose(out["dh0"], h0.grad.numpy(), **tol)
    if lstm:
        np.testing.assert_allclose(out["cy"], cy.detach().numpy(), **tol)
        np.testing.assert_allclose(out["dc0"], c0.grad.numpy(), **tol)
    dp = oracle.unflatten_weights(out["dW"], mode, L, bidir, I, H)
    for l, m in enumerate(layers):
        for d in range(D):
            sfx = "_l0" + ("_reverse" if d == 1 else "")
            for name, tname in (("W_ih", "weight_ih"), ("W_hh", "weight_hh"),
                                ("b_ih", "bias_ih"), ("b_hh", "bias_hh")):
                np.testing.assert_allclose(dp[l * D + d][name],
                                           getattr(m, tname + sfx).grad.numpy(), **tol)


@pytest.mark.parametrize("mode,L,bidir", [("lstm", 2, True), ("gru", 2, False)])
def test_dropout_gradients_match_finite_differences(mode, L, bidir):
    cfg, inp = _case(mode, L, bidir, 3, 2, 2, 2, 73)
    p = 0.3
    masks = _masks(cfg, 1.0 - p, 79)
    out = _run(cfg, inp, p, masks)
    params_of = lambda w: oracle.unflatten_weights(w, mode, L, bidir, cfg["I"], cfg["H"])

    def loss_of(d):
        y, hy, cy, _ = oracle.forward(mode, d["x"], d["h0"], d["c0"], params_of(d["w"]), L,
                                      bidir, dropout=p, masks=masks)
        return oracle.loss(y, hy, cy, d["dy"], d["dhy"], d["dcy"] if mode == "lstm" else None)

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


def test_a_dropped_feature_has_no_weight_gradient_above():
    cfg, inp = _case("lstm", 2, False, 4, 3, 3, 4, 83)
    masks = [np.ones((4, 3, 4))]
    masks[0][:, :, 2] = 0.0  # unit 2 of layer 0 never reaches layer 1
    out = _run(cfg, inp, 0.5, masks)
    dp = oracle.unflatten_weights(out["dW"], "lstm", 2, False, 3, 4)
    assert not dp[1]["W_ih"][:, 2].any()
    assert dp[1]["W_ih"][:, [0, 1, 3]].any()


def test_masks_are_checked():
    cfg, inp = _case("gru", 2, False, 3, 2, 2, 2, 5)
    good = np.ones((3, 2, 2))
    for p, masks in ((0.2, []), (0.2, [np.ones((3, 2, 3))]), (1.0, [good]),
                     (0.2, [good * 0.5])):
        with pytest.raises(ValueError):
            _run(cfg, inp, p, masks)
