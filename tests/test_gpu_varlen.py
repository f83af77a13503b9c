"""Variable-length (padded) batches through the C ABI against the float64
oracle with the same lengths: rnn_forward_training_varlen,
rnn_backward_data_varlen, rnn_backward_weights and
rnn_forward_inference_varlen.

Lengths cover the degenerate cases: 0 (nothing runs: y is zero, hy = h0,
dh0 = dhy), 1, T - 1 and T; both directions and stacked layers (the reverse
direction starts at each sequence's last valid step; the layer above reads
zeros past the length), fp32 and bf16, batches that are not multiples of a
tile.
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
    # mode, L, bidir, T, N, I, H, dtype
    ("lstm", 1, False, 7, 5, 6, 16, "f32"),
    ("gru", 2, True, 6, 4, 8, 12, "f32"),
    ("rnn_tanh", 2, True, 5, 3, 4, 8, "f32"),
    ("lstm", 2, True, 9, 6, 10, 24, "f32"),
    ("lstm", 1, False, 40, 20, 64, 96, "f32"),
    ("lstm", 2, True, 9, 6, 16, 24, "bf16"),
    ("gru", 1, False, 8, 33, 16, 40, "bf16"),
]


def _cid(c):
    return "%s-L%d-%s-T%d-N%d-I%d-H%d-%s" % (c[0], c[1], "bi" if c[2] else "uni", *c[3:])


def _lengths(T, N, seed):
    base = [T, 0, 1, T - 1, T // 2]
    rng = np.random.default_rng(seed)
    extra = rng.integers(0, T + 1, size=max(0, N - len(base)))
    return np.array((base + list(extra))[:N], dtype=np.int32)


@pytest.mark.parametrize("case", CASES, ids=[_cid(c) for c in CASES])
def test_varlen_parity(case):
    mode, L, bidir, T, N, I, H, dt = case
    seed = zlib.crc32(_cid(case).encode()) % 10000
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, dt, 0.3, seed=seed)
    inp = wl.make_inputs(cfg)
    lengths = _lengths(T, N, seed)
    gpu = harness.run_gpu(cfg, inp, lengths=lengths)
    ref = harness.run_oracle(cfg, inp, lengths=lengths)
    harness.assert_parity(cfg, gpu, ref)
    for n, ln in enumerate(lengths):
        # nothing past a sequence's length: output and input gradient exactly zero
        assert not gpu["y"][ln:, n].any(), n
        assert not gpu["dx"][ln:, n].any(), n
    # inference runs the same kernels without the workspace: bit for bit
    assert np.array_equal(gpu["y_inf"], gpu["y"])
    assert np.array_equal(gpu["hy_inf"], gpu["hy"])
    if gpu["cy"] is not None:
        assert np.array_equal(gpu["cy_inf"], gpu["cy"])


def test_full_lengths_match_the_fixed_length_calls():
    # every length equal to T: the CUDA-core varlen path and the default path
    # (tensor cores where they fit) agree with each other within the bars
    cfg = wl.make_config("gru", 1, True, 6, 8, 16, 32, "f32", 0.3, seed=3)
    inp = wl.make_inputs(cfg)
    a = harness.run_gpu(cfg, inp, lengths=np.full(8, 6, dtype=np.int32))
    b = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    harness.assert_parity(cfg, a, ref)
    harness.assert_parity(cfg, b, ref)
