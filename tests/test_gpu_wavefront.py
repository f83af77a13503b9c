"""The layer-wavefront forward (unidirectional bf16 stacks, all layers in one
persistent launch) against the float64 oracle, and against the layer-by-layer
path selected by RNN_FLAG_NO_WAVEFRONT.

Sizes are chosen to cross the kernel's tiling edges: input sizes below, at and
above one 64-element K chunk and not multiples of it, hidden sizes that leave a
ragged last block, batch 1 / 128 / not a multiple of 16, T = 1, 2 to 5 layers,
and all three cell types (the GRU's n gate runs as two packed rows, so its
r * (W_hn h + b_hn) term is exercised separately from W_in x).
"""

import zlib

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


CASES = [
    # mode, L, T, N, I, H
    ("lstm", 3, 7, 20, 48, 64),
    ("gru", 2, 9, 5, 64, 40),
    ("rnn_tanh", 4, 6, 33, 24, 136),
    ("lstm", 2, 1, 1, 8, 8),
    ("gru", 5, 4, 128, 72, 96),
    ("lstm", 2, 5, 128, 200, 1032),
    ("rnn_tanh", 2, 3, 16, 1024, 512),
]


def _cid(c):
    return "%s-L%d-T%d-N%d-I%d-H%d" % c


def _launches(cfg, inp, flags):
    """rec_fwd / input phase kernel counts of one training forward."""
    from layer_rnn_gb300 import binding as B
    T, N, I, H, L = cfg["T"], cfg["N"], cfg["I"], cfg["H"], cfg["L"]
    r = B.Rnn(cfg["mode"], L, False, I, H, "bf16", flags | B.RNN_FLAG_SYNC_CHECK)
    try:
        x = harness.to_dev(inp["x"], "bf16")
        W = harness.to_dev(inp["w"], "bf16")
        y = harness.empty((T, N, H), "bf16")
        ws = r.alloc_workspace(T, N)
        B.rnn_enable_phase_timing(r.h, 1)
        r.forward_training(x, None, None, W, y, None, None, ws)
        ph = B.rnn_get_phase_times(r.h)
        return ph["rec_fwd"][1], ph["input_gemm"][1]
    finally:
        r.close()


@pytest.mark.parametrize("case", CASES, ids=[_cid(c) for c in CASES])
def test_wavefront_parity(case):
    mode, L, T, N, I, H = case
    cfg = wl.make_config(mode, L, False, T, N, I, H, "bf16", 0.5,
                         seed=zlib.crc32(_cid(case).encode()) % 10000)
    inp = wl.make_inputs(cfg)
    # the wavefront path is the one taken: one recurrent launch for all layers
    rec, packs = _launches(cfg, inp, 0)
    assert rec == 1 and packs == L
    gpu = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    harness.assert_parity(cfg, gpu, ref)
    assert np.array_equal(gpu["y_inf"], gpu["y"])
    assert np.array_equal(gpu["hy_inf"], gpu["hy"])


@pytest.mark.parametrize("mode", ["lstm", "gru"])
def test_wavefront_matches_layer_by_layer(mode):
    from layer_rnn_gb300 import binding as B
    cfg = wl.make_config(mode, 3, False, 11, 24, 96, 160, "bf16", 0.5, seed=31)
    inp = wl.make_inputs(cfg)
    rec, _ = _launches(cfg, inp, B.RNN_FLAG_NO_WAVEFRONT)
    assert rec == 3
    a = harness.run_gpu(cfg, inp)
    b = harness.run_gpu(cfg, inp, flags=B.RNN_FLAG_NO_WAVEFRONT)
    ref = harness.run_oracle(cfg, inp)
    harness.assert_parity(cfg, a, ref)
    harness.assert_parity(cfg, b, ref)
    # same arithmetic up to the order of the fp32 accumulation
    for k in ("y", "hy", "cy"):
        if a[k] is not None:
            assert harness.rel_err(a[k], b[k]) < 2e-2, k


def test_wavefront_timeout_is_reported_and_context_survives():
    import torch
    from layer_rnn_gb300 import binding as B
    cfg = wl.make_config("lstm", 2, False, 6, 8, 16, 32, "bf16", 0.3, seed=5)
    inp = wl.make_inputs(cfg)
    T, N, I, H = cfg["T"], cfg["N"], cfg["I"], cfg["H"]
    r = B.Rnn("lstm", 2, False, I, H, "bf16", 0)
    try:
        x = harness.to_dev(inp["x"], "bf16")
        W = harness.to_dev(inp["w"], "bf16")
        y = harness.empty((T, N, H), "bf16")
        ws = r.alloc_workspace(T, N)
        # block 0 (layer 0) never announces step 2: the rest give up after 50 ms
        B.rnn_set_debug(r.h, 0, 2, 50_000_000)
        r.forward_training(x, None, None, W, y, None, None, ws)
        assert r.check_status() == 6  # RNN_ERR_TIMEOUT
        assert r.check_status() == 0
        B.rnn_set_debug(r.h, -1, -1, 2_000_000_000)
        r.forward_training(x, None, None, W, y, None, None, ws)
        assert r.check_status() == 0
        import oracle
        params = oracle.unflatten_weights(inp["w"], "lstm", 2, False, I, H)
        ref, _, _, _ = oracle.forward("lstm", inp["x"], None, None, params, 2, False)
        assert harness.rel_err(harness.from_dev(y), ref) < 2e-2
        torch.cuda.synchronize()
    finally:
        r.close()
