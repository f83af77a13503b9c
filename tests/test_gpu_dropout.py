"""Inter-layer dropout through the C ABI (rnn_forward_training_dropout,
rnn_backward_data_dropout, then rnn_backward_weights) against the float64
oracle with the same masks: stacks of 2 and 3 layers, both directions, fp32
and bf16 (a bf16 unidirectional stack, which otherwise takes the wavefront,
runs layer by layer here)."""

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
]


def _cid(c):
    return "%s-L%d-%s-T%d-N%d-I%d-H%d-%s-p%s" % (c[0], c[1], "bi" if c[2] else "uni", *c[3:])


@pytest.mark.parametrize("case", CASES, ids=[_cid(c) for c in CASES])
def test_dropout_parity(case):
    mode, L, bidir, T, N, I, H, dt, p = case
    seed = zlib.crc32(_cid(case).encode()) % 10000
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, dt, 0.3, seed=seed)
    inp = wl.make_inputs(cfg)
    D = 2 if bidir else 1
    rng = np.random.default_rng(seed)
    masks = (rng.random((L - 1, T, N, D * H)) >= p).astype(np.uint8)
    gpu = harness.run_gpu(cfg, inp, inference=False, dropout=(p, masks))
    ref = harness.run_oracle(cfg, inp, dropout=(p, list(masks.astype(np.float64))))
    harness.assert_parity(cfg, gpu, ref)


def test_all_ones_masks_without_dropout_match_the_plain_calls():
    cfg = wl.make_config("lstm", 2, True, 6, 8, 16, 32, "f32", 0.3, seed=9)
    inp = wl.make_inputs(cfg)
    masks = np.ones((1, 6, 8, 64), dtype=np.uint8)
    a = harness.run_gpu(cfg, inp, inference=False, dropout=(0.0, masks))
    b = harness.run_gpu(cfg, inp, inference=False)
    for k in ("y", "hy", "cy", "dx", "dh0", "dc0", "dW"):
        assert np.array_equal(a[k], b[k]), k
