"""Inter-layer dropout through the C ABI (rnn_forward_training_dropout,
rnn_backward_data_dropout, then rnn_backward_weights) against the float64
oracle with the same masks: stacks of 2 to 4 layers, both directions, fp32
and bf16.  A bf16 unidirectional stack runs the layer wavefront, which
applies the masks as each layer writes its output (and, with the wavefront
switched off, layer by layer, where a separate pass applies them)."""

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
    # mode, L, bidir, T, N, I, H, dtype, p
    ("lstm", 2, False, 7, 5, 6, 16, "f32", 0.4),
    ("gru", 3, True, 6, 4, 8, 12, "f32", 0.25),
    ("rnn_tanh", 2, True, 5, 3, 4, 8, "f32", 0.5),
    ("lstm", 3, False, 9, 16, 32, 64, "bf16", 0.3),
    ("gru", 2, True, 6, 33, 16, 40, "bf16", 0.2),
    # unidirectional bf16 stacks: the layer wavefront
    ("gru", 2, False, 8, 40, 16, 48, "bf16", 0.3),
    ("rnn_tanh", 3, False, 7, 24, 16, 40, "bf16", 0.2),
    ("lstm", 4, False, 6, 128, 32, 64, "bf16", 0.3),
]


def _cid(c):
    return "%s-L%d-%s-T%d-N%d-I%d-H%d-%s-p%s" % (c[0], c[1], "bi" if c[2] else "uni", *c[3:])


def _check(case, flags=0):
    mode, L, bidir, T, N, I, H, dt, p = case
    seed = zlib.crc32(_cid(case).encode()) % 10000
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, dt, 0.3, seed=seed)
    inp = wl.make_inputs(cfg)
    D = 2 if bidir else 1
    rng = np.random.default_rng(seed)
    masks = (rng.random((L - 1, T, N, D * H)) >= p).astype(np.uint8)
    gpu = harness.run_gpu(cfg, inp, inference=False, dropout=(p, masks), flags=flags)
    ref = harness.run_oracle(cfg, inp, dropout=(p, list(masks.astype(np.float64))))
    harness.assert_parity(cfg, gpu, ref)


def _fwd_path(cfg, flags=0):
    from layer_rnn_gb300 import binding as B
    r = B.Rnn(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"], cfg["dtype"], flags)
    try:
        return B.rnn_get_paths(r.h, cfg["N"])[0]
    finally:
        r.close()


@pytest.mark.parametrize("case", CASES, ids=[_cid(c) for c in CASES])
def test_dropout_parity(case):
    _check(case)


@pytest.mark.parametrize("case", [c for c in CASES if c[7] == "bf16" and not c[2]],
                         ids=[_cid(c) for c in CASES if c[7] == "bf16" and not c[2]])
def test_dropout_layer_by_layer(case):
    from layer_rnn_gb300 import binding as B
    mode, L, bidir, T, N, I, H, dt, p = case
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, dt, 0.3, seed=1)
    assert _fwd_path(cfg) == "wavefront"
    assert _fwd_path(cfg, B.RNN_FLAG_NO_WAVEFRONT) != "wavefront"
    _check(case, flags=B.RNN_FLAG_NO_WAVEFRONT)


@pytest.mark.parametrize("shape", [("lstm", True, "f32"), ("lstm", False, "bf16"),
                                   ("gru", False, "bf16")])
def test_all_ones_masks_without_dropout_match_the_plain_calls(shape):
    # p = 0 with every mask byte 1: the same results bit for bit (on the
    # wavefront too, where the layer above then reads the undropped copy)
    mode, bidir, dt = shape
    L, T, N, H = 3, 6, 8, 32
    cfg = wl.make_config(mode, L, bidir, T, N, 16, H, dt, 0.3, seed=9)
    inp = wl.make_inputs(cfg)
    masks = np.ones((L - 1, T, N, (2 if bidir else 1) * H), dtype=np.uint8)
    a = harness.run_gpu(cfg, inp, inference=False, dropout=(0.0, masks))
    b = harness.run_gpu(cfg, inp, inference=False)
    for k in ("y", "hy", "cy", "dx", "dh0", "dc0", "dW"):
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("name", ["bi5_gru", "lstm4_bf16"])
def test_dropout_workload_parity(name):
    # the bench's stacks with the bench's masks (p = 0.3): bi5_gru at full
    # size, layer by layer; lstm4_bf16 on the wavefront at T = 128 (the
    # oracle's float64 masks stay below 0.5 GB; every step does the same work)
    cfg = wl.WORKLOADS[name]
    if name == "lstm4_bf16":
        cfg = wl.with_sizes(cfg, T=128)
    inp = wl.make_inputs(cfg)
    p = 0.3
    masks = wl.make_dropout_masks(cfg, p)
    gpu = harness.run_gpu(cfg, inp, inference=False, dropout=(p, masks))
    ref = harness.run_oracle(cfg, inp, dropout=(p, list(masks.astype(np.float64))))
    harness.assert_parity(cfg, gpu, ref)
