"""Extreme-value parity of the CUDA paths, through the C ABI, against the
float64 oracle and against closed forms the cell equations fix:

* all weights and biases zero: every sigmoid gate is exactly 1/2 and every
  tanh candidate 0, so one GRU step halves h, one LSTM step halves c (and
  h' = tanh(c') / 2), and a tanh RNN outputs 0 -- exact in binary floating
  point, so h_T = 2^-T h0 and c_T = 2^-T c0 bit for bit;
* saturated gates: a GRU update gate with bias +40 keeps h (z rounds to 1 in
  fp32), an LSTM with input-gate bias -40 and forget-gate bias +40 keeps c;
* pre-activations of magnitude ~100 (sigmoid and tanh deep in saturation,
  exp overflowing in the naive form of the logistic function).

The cell equations are those of "rnn training example?" (oneDNN issue #218,
the PyTorch GRU equations) and the standard LSTM; each case runs on the
tensor-core recurrent kernels (fp32) and on the bf16 layer wavefront."""

import numpy as np
import pytest

from layer_rnn_gb300 import workloads as wl
from tests import harness

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    harness.ensure_built()


# (mode, L, bidir, T, N, I, H, dtype, expected forward path)
PATHS = [
    ("lstm", 1, False, 12, 20, 64, 128, "f32", "tensor"),
    ("gru", 1, True, 12, 20, 64, 128, "f32", "tensor"),
    ("rnn_tanh", 2, False, 12, 20, 64, 128, "f32", "tensor"),
    ("lstm", 2, False, 12, 16, 64, 64, "bf16", "wavefront"),
    ("gru", 2, False, 12, 16, 64, 64, "bf16", "wavefront"),
]


def _ids(cases):
    return ["%s-L%d-%s-%s" % (c[0], c[1], "bi" if c[2] else "uni", c[7]) for c in cases]


def _cfg(case, seed):
    mode, L, bidir, T, N, I, H, dt, _ = case
    return wl.make_config(mode, L, bidir, T, N, I, H, dt, 0.5, seed=seed)


def _params_flat(cfg, inp, fn):
    """Apply fn(params_dict, H, layer) to every (layer, direction) and
    re-flatten."""
    import oracle
    params = oracle.unflatten_weights(inp["w"], cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"],
                                      cfg["H"])
    D = wl.num_directions(cfg)
    for k, p in enumerate(params):
        fn(p, cfg["H"], k // D)
    return wl.round_to(oracle.flatten_weights(params, cfg["mode"], cfg["L"], cfg["bidir"],
                                              cfg["I"], cfg["H"]), cfg["dtype"])


def _check_path(cfg, expected):
    from layer_rnn_gb300 import binding as B
    r = B.Rnn(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"], cfg["dtype"], 0)
    try:
        fwd, _ = B.rnn_get_paths(r.h, cfg["N"])
    finally:
        r.close()
    assert fwd == expected, (fwd, expected)


@pytest.mark.parametrize("case", PATHS, ids=_ids(PATHS))
def test_zero_weights_closed_forms(case):
    cfg = _cfg(case, 301)
    _check_path(cfg, case[8])
    inp = wl.make_inputs(cfg)
    inp["w"] = np.zeros_like(inp["w"])
    gpu = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    harness.assert_parity(cfg, gpu, ref)
    T, L = cfg["T"], cfg["L"]
    D = wl.num_directions(cfg)
    # layer 0 carries the closed form of its own h0 / c0; the layers above
    # see the same recurrence (their input weights are zero too)
    scale = 0.5 ** T
    if cfg["mode"] == "gru":
        assert np.array_equal(gpu["hy"], inp["h0"] * scale)
    elif cfg["mode"] == "lstm":
        assert np.array_equal(gpu["cy"], inp["c0"] * scale)
    else:
        assert np.array_equal(gpu["y"], np.zeros((T, cfg["N"], D * cfg["H"])))
        assert np.array_equal(gpu["hy"], np.zeros((L * D, cfg["N"], cfg["H"])))


@pytest.mark.parametrize("case", [c for c in PATHS if c[0] != "rnn_tanh"],
                         ids=_ids([c for c in PATHS if c[0] != "rnn_tanh"]))
def test_saturated_gates_keep_the_state(case):
    cfg = _cfg(case, 302)
    _check_path(cfg, case[8])
    inp = wl.make_inputs(cfg)

    def saturate(p, H, layer):
        if cfg["mode"] == "gru":
            p["b_ih"][H:2 * H] = 40.0          # update gate z = 1: h' = h
        else:
            p["b_ih"][:H] = -40.0              # input gate i = 0
            p["b_ih"][H:2 * H] = 40.0          # forget gate f = 1: c' = c

    inp["w"] = _params_flat(cfg, inp, saturate)
    gpu = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    harness.assert_parity(cfg, gpu, ref)
    if cfg["dtype"] == "f32":
        # in fp32 the saturated gate is exactly 1 (and the input gate below
        # half an ulp of c), so the state passes through every step unchanged
        if cfg["mode"] == "gru":
            assert np.array_equal(gpu["hy"][0], inp["h0"][0])
        else:
            assert np.array_equal(gpu["cy"][0], inp["c0"][0])


@pytest.mark.parametrize("case", PATHS, ids=_ids(PATHS))
def test_preactivations_near_100(case):
    cfg = _cfg(case, 303)
    _check_path(cfg, case[8])
    inp = wl.make_inputs(cfg)
    # layer 0's input weights ~ U(-b, b) with b chosen so that W_ih x alone
    # has a standard deviation of 100 (x ~ N(0, 1)): most gates saturate hard,
    # some do not.  Only there: with recurrent weights that large the
    # recurrence becomes chaotic, and input weights that large above layer 0
    # multiply the rounding of the layer below by hundreds -- in both cases any
    # two roundings (fp32 against float64) part ways regardless of the kernels.
    b = 100.0 * np.sqrt(3.0 / cfg["I"])

    def widen(p, H, layer):
        if layer == 0:
            p["W_ih"] = p["W_ih"] * (b * np.sqrt(H))

    inp["w"] = _params_flat(cfg, inp, widen)
    gpu = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    for k in ("y", "hy", "cy", "dx", "dh0", "dc0", "dW"):
        if gpu[k] is not None:
            assert np.all(np.isfinite(gpu[k])), k
    harness.assert_parity(cfg, gpu, ref)


# ----------------------------------------------------------------------------
# workspace read-back: the saved activations against the oracle's tape
# ----------------------------------------------------------------------------

WS_CASES = [
    ("lstm", 2, True, 9, 20, 48, 96, "f32", "tensor"),
    ("gru", 1, True, 9, 20, 48, 96, "f32", "tensor"),
    ("rnn_tanh", 2, True, 9, 20, 48, 96, "f32", "tensor"),
    ("lstm", 3, False, 9, 16, 64, 64, "bf16", "wavefront"),
    ("gru", 2, False, 9, 16, 64, 64, "bf16", "wavefront"),
]


def _region(B, r, T, N, region, l, d, ws, dtype, shape):
    import torch
    off, nbytes = B.rnn_workspace_layout(r.h, T, N, region, l, d)
    td = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    esz = 4 if dtype == "f32" else 2
    n = int(np.prod(shape))
    assert nbytes >= n * esz, (region, nbytes, n * esz)
    t = ws[off:off + n * esz].view(td).reshape(shape)
    return harness.from_dev(t), t


@pytest.mark.parametrize("case", WS_CASES, ids=_ids(WS_CASES))
def test_workspace_regions_match_the_oracle_tape(case):
    """After rnn_forward_training the GATES, CSEQ and HSEQ regions hold what
    the backward reuses ("Fused RNN operator for CPU", Operator Registration:
    forward intermediates reused in backward): per (layer, direction) the gate
    activations of every step, the cell states and the hidden states with the
    initial state in the first slot.  The initial-state slots and the hidden
    state sequence against the layer output are compared bit for bit."""
    import oracle
    import torch
    from layer_rnn_gb300 import binding as B
    cfg = _cfg(case, 304)
    _check_path(cfg, case[8])
    inp = wl.make_inputs(cfg)
    mode, L, T, N, I, H, dt = cfg["mode"], cfg["L"], cfg["T"], cfg["N"], cfg["I"], cfg["H"], \
        cfg["dtype"]
    D = wl.num_directions(cfg)
    lstm = mode == "lstm"
    r = B.Rnn(mode, L, cfg["bidir"], I, H, dt, B.RNN_FLAG_SYNC_CHECK)
    try:
        x = harness.to_dev(inp["x"], dt)
        h0 = harness.to_dev(inp["h0"], dt)
        c0 = harness.to_dev(inp["c0"], "f32") if lstm else None
        W = harness.to_dev(inp["w"], dt)
        y = harness.empty((T, N, D * H), dt)
        ws = r.alloc_workspace(T, N)
        ws.fill_(0xFF)
        r.forward_training(x, h0, c0, W, y, None, None, ws)
        torch.cuda.synchronize()
        params = oracle.unflatten_weights(inp["w"], mode, L, cfg["bidir"], I, H)
        y_ref, _, _, cache = oracle.forward(mode, inp["x"], inp["h0"], inp["c0"], params, L,
                                            cfg["bidir"])
        tol = harness.tolerances(cfg)[0]
        y_gpu = harness.from_dev(y)
        G4 = {"lstm": 4, "gru": 4, "rnn_tanh": 1}[mode]
        for l in range(L):
            for d in range(D):
                k = l * D + d
                tape = sorted(cache["tapes"][k], key=lambda rec: rec["t"])
                if mode == "lstm":
                    g_ref = np.stack([np.concatenate([rec[n] for n in "ifgo"], axis=1)
                                      for rec in tape])
                elif mode == "gru":
                    g_ref = np.stack([np.concatenate([rec["r"], rec["z"], rec["n"],
                                                      rec["h_n"]], axis=1) for rec in tape])
                else:
                    g_ref = np.stack([rec["h"] for rec in tape])
                gates, _ = _region(B, r, T, N, B.RNN_WS_GATES, l, d, ws, "f32", (T, N, G4 * H))
                assert harness.rel_err(gates, g_ref) <= tol, ("gates", l, d)
                hs, hs_t = _region(B, r, T, N, B.RNN_WS_HSEQ, l, d, ws, dt, (T + 1, N, H))
                # slot of h0, and slot of the state after time t
                s0 = 0 if d == 0 else T
                slot = (lambda t: t + 1) if d == 0 else (lambda t: t)
                h0_dev = harness.to_dev(inp["h0"][k], dt)
                assert torch.equal(hs_t[s0].contiguous().view(torch.uint8),
                                   h0_dev.contiguous().view(torch.uint8)), ("h0 slot", l, d)
                layer_out = cache["inputs"][l + 1] if l + 1 < L else y_ref
                h_ref = layer_out[:, :, d * H:(d + 1) * H]
                h_gpu = np.stack([hs[slot(t)] for t in range(T)])
                assert harness.rel_err(h_gpu, h_ref) <= tol, ("hseq", l, d)
                if l == L - 1:
                    # the hidden-state sequence is the layer output, bit for bit
                    assert np.array_equal(h_gpu, y_gpu[:, :, d * H:(d + 1) * H]), ("hseq=y", d)
                if lstm:
                    cs, _ = _region(B, r, T, N, B.RNN_WS_CSEQ, l, d, ws, "f32", (T + 1, N, H))
                    assert np.array_equal(cs[s0], inp["c0"][k]), ("c0 slot", l, d)
                    c_ref = np.stack([rec["c"] for rec in tape])
                    c_gpu = np.stack([cs[slot(t)] for t in range(T)])
                    assert harness.rel_err(c_gpu, c_ref) <= tol, ("cseq", l, d)
            if l < L - 1:
                yl, _ = _region(B, r, T, N, B.RNN_WS_YLAYER, l, 0, ws, dt, (T, N, D * H))
                assert harness.rel_err(yl, cache["inputs"][l + 1]) <= tol, ("ylayer", l)
    finally:
        r.close()
