"""Pins for the oracle's variable-length (padded) batches, against things other
than the masked code itself:

* every length equal to T gives exactly the fixed-length oracle;
* PyTorch's own CPU float64 nn.LSTM / nn.GRU / nn.RNN on a packed sequence
  (pack_padded_sequence / pad_packed_sequence: the packed-sequence form that
  "rnn training example?" (oneDNN issue #218) names as what PyTorch users
  feed), forward and every gradient;
* each sequence of the batch equals the fixed-length oracle run on that
  sequence alone, cut to its length (length 0 included: y is zero, the state
  passes through, dh0 = dhy);
* central finite differences of the loss.
"""

import numpy as np
import pytest

import oracle
from layer_rnn_gb300 import workloads as wl


def _case(mode, L, bidir, T, N, I, H, seed):
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, "f32", 0.3, seed)
    inp = wl.make_inputs(cfg)
    inp["w"] = inp["w"] * 2.0  # away from the linear region of the gates
    return cfg, inp


def _run(cfg, inp, lengths):
    return oracle.run_flat(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"],
                           inp["x"], inp["h0"], inp["c0"], inp["w"], inp["dy"],
                           inp["dhy"], inp["dcy"], lengths=lengths)


CASES = [("lstm", 1, False), ("gru", 1, False), ("rnn_tanh", 1, False),
         ("lstm", 2, True), ("gru", 2, True), ("rnn_tanh", 2, True)]


@pytest.mark.parametrize("mode,L,bidir", CASES)
def test_full_lengths_are_the_fixed_length_oracle(mode, L, bidir):
    cfg, inp = _case(mode, L, bidir, 5, 3, 4, 3, 41)
    a = _run(cfg, inp, None)
    b = _run(cfg, inp, np.full(3, 5))
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("mode,L,bidir", CASES)
def test_matches_torch_packed_sequences(mode, L, bidir):
    torch = pytest.importorskip("torch")
    from torch.nn.utils.rnn import pack_padded_sequence, pad_packed_sequence
    T, N = 6, 4
    cfg, inp = _case(mode, L, bidir, T, N, 5, 4, 43)
    lengths = np.array([4, 6, 1, 3])
    out = _run(cfg, inp, lengths)
    params = oracle.unflatten_weights(inp["w"], mode, L, bidir, cfg["I"], cfg["H"])
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
    packed = pack_padded_sequence(x, torch.from_numpy(lengths), enforce_sorted=False)
    if mode == "lstm":
        c0 = torch.from_numpy(inp["c0"]).requires_grad_(True)
        yp, (hy, cy) = m(packed, (h0, c0))
    else:
        yp, hy = m(packed, h0)
    y, _ = pad_packed_sequence(yp, total_length=T)
    loss = (y * torch.from_numpy(inp["dy"])).sum() + (hy * torch.from_numpy(inp["dhy"])).sum()
    if mode == "lstm":
        loss = loss + (cy * torch.from_numpy(inp["dcy"])).sum()
    loss.backward()
    tol = dict(rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["y"], y.detach().numpy(), **tol)
    np.testing.assert_allclose(out["hy"], hy.detach().numpy(), **tol)
    np.testing.assert_allclose(out["dx"], x.grad.numpy(), **tol)
    np.testing.assert_allclose(out["dh0"], h0.grad.numpy(), **tol)
    if mode == "lstm":
        np.testing.assert_allclose(out["cy"], cy.detach().numpy(), **tol)
        np.testing.assert_allclose(out["dc0"], c0.grad.numpy(), **tol)
    dp = oracle.unflatten_weights(out["dW"], mode, L, bidir, cfg["I"], cfg["H"])
    for l in range(L):
        for d in range(D):
            sfx = "_l%d%s" % (l, "_reverse" if d == 1 else "")
            for name, tname in (("W_ih", "weight_ih"), ("W_hh", "weight_hh"),
                                ("b_ih", "bias_ih"), ("b_hh", "bias_hh")):
                np.testing.assert_allclose(dp[l * D + d][name],
                                           getattr(m, tname + sfx).grad.numpy(), **tol)


@pytest.mark.parametrize("mode,L,bidir", CASES)
def test_each_sequence_is_its_own_fixed_length_run(mode, L, bidir):
    T, N = 5, 4
    cfg, inp = _case(mode, L, bidir, T, N, 3, 3, 47)
    lengths = np.array([5, 2, 0, 3])
    out = _run(cfg, inp, lengths)
    dW_sum = np.zeros_like(out["dW"])
    lstm = mode == "lstm"
    for n, ln in enumerate(lengths):
        sl = slice(n, n + 1)
        one = oracle.run_flat(mode, L, bidir, cfg["I"], cfg["H"], inp["x"][:ln, sl],
                              inp["h0"][:, sl], inp["c0"][:, sl] if lstm else None, inp["w"],
                              inp["dy"][:ln, sl], inp["dhy"][:, sl],
                              inp["dcy"][:, sl] if lstm else None)
        tol = dict(rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(out["y"][:ln, n], one["y"][:, 0], **tol)
        assert not out["y"][ln:, n].any()
        np.testing.assert_allclose(out["hy"][:, n], one["hy"][:, 0], **tol)
        np.testing.assert_allclose(out["dx"][:ln, n], one["dx"][:, 0], **tol)
        assert not out["dx"][ln:, n].any()
        np.testing.assert_allclose(out["dh0"][:, n], one["dh0"][:, 0], **tol)
        if lstm:
            np.testing.assert_allclose(out["cy"][:, n], one["cy"][:, 0], **tol)
            np.testing.assert_allclose(out["dc0"][:, n], one["dc0"][:, 0], **tol)
        dW_sum += one["dW"]
        if ln == 0:  # nothing ran: the state and its gradient pass straight through
            np.testing.assert_array_equal(out["hy"][:, n], inp["h0"][:, n])
            np.testing.assert_array_equal(out["dh0"][:, n], inp["dhy"][:, n])
    np.testing.assert_allclose(out["dW"], dW_sum, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("mode,L,bidir", [("lstm", 1, True), ("gru", 2, False),
                                          ("rnn_tanh", 1, True)])
def test_varlen_gradients_match_finite_differences(mode, L, bidir):
    cfg, inp = _case(mode, L, bidir, 3, 3, 2, 2, 53)
    lengths = np.array([3, 1, 0])
    out = _run(cfg, inp, lengths)
    params_of = lambda w: oracle.unflatten_weights(w, mode, L, bidir, cfg["I"], cfg["H"])

    def loss_of(d):
        y, hy, cy, _ = oracle.forward(mode, d["x"], d["h0"], d["c0"], params_of(d["w"]),
                                      L, bidir, lengths)
        return oracle.loss(y, hy, cy, d["dy"], d["dhy"], d["dcy"] if mode == "lstm" else None)

    grads = dict(x=out["dx"], h0=out["dh0"], w=out["dW"])
    if mode == "lstm":
        grads["c0"] = out["dc0"]
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


def test_lengths_are_checked():
    cfg, inp = _case("gru", 1, False, 3, 2, 2, 2, 5)
    for bad in ([4, 1], [-1, 2], [1, 2, 3]):
        with pytest.raises(ValueError):
            _run(cfg, inp, np.array(bad))
