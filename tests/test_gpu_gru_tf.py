"""The TensorFlow-flavour GRU (RNN_GRU_TF, reset gate before the candidate's
recurrent product) through the C ABI against the float64 oracle's mode
"gru_tf" ("rnn training example?", oneDNN issue #218: the TensorFlow GRU
equations, n = tanh(W_in x + b_in + W_hn (r * h) + b_hn)).

Small ragged cases (both directions, stacks, fp32 and bf16, T = 1, N = 1),
variable lengths, inter-layer dropout, and the Deep Speech 2 GRU layer shape
(T 300, N 20, I = H = 800) in fp32 and bf16; the result differs from the
PyTorch flavour of the same weights, and inference equals training bit for
bit.
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
    # L, bidir, T, N, I, H, dtype
    (1, False, 7, 5, 19, 36, "f32"),
    (2, True, 6, 3, 11, 28, "f32"),
    (3, False, 5, 6, 9, 40, "f32"),
    (1, False, 1, 1, 1, 4, "f32"),
    (1, True, 20, 33, 64, 96, "f32"),
    (2, False, 8, 9, 24, 48, "bf16"),
    (1, True, 6, 3, 16, 24, "bf16"),
]


def _cid(c):
    return "L%d-%s-T%d-N%d-I%d-H%d-%s" % (c[0], "bi" if c[1] else "uni", *c[2:])


def _cfg(case, h0_std=0.5, tag=""):
    L, bidir, T, N, I, H, dt = case
    seed = zlib.crc32((_cid(case) + tag).encode()) % 10000
    return wl.make_config("gru_tf", L, bidir, T, N, I, H, dt, h0_std, seed=seed)


@pytest.mark.parametrize("case", CASES, ids=[_cid(c) for c in CASES])
def test_gru_tf_parity(case):
    cfg = _cfg(case)
    inp = wl.make_inputs(cfg)
    gpu = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    harness.assert_parity(cfg, gpu, ref)
    assert np.array_equal(gpu["y_inf"], gpu["y"])
    assert np.array_equal(gpu["hy_inf"], gpu["hy"])


def test_gru_tf_differs_from_the_pytorch_flavour():
    cfg = _cfg(CASES[0])
    inp = wl.make_inputs(cfg)
    tf = harness.run_gpu(cfg, inp, inference=False)
    pt_cfg = dict(cfg, mode="gru")
    pt = harness.run_gpu(pt_cfg, inp, inference=False)
    assert np.abs(tf["y"] - pt["y"]).max() > 1e-3
    harness.assert_parity(pt_cfg, pt, harness.run_oracle(pt_cfg, inp))


@pytest.mark.parametrize("case", [CASES[1], CASES[5]], ids=[_cid(CASES[1]), _cid(CASES[5])])
def test_gru_tf_variable_lengths(case):
    cfg = _cfg(case, tag="varlen")
    inp = wl.make_inputs(cfg)
    T, N = cfg["T"], cfg["N"]
    lengths = np.array(([T, 0, 1, T - 1] + [T // 2] * N)[:N], dtype=np.int32)
    gpu = harness.run_gpu(cfg, inp, lengths=lengths)
    ref = harness.run_oracle(cfg, inp, lengths=lengths)
    harness.assert_parity(cfg, gpu, ref)
    for n, ln in enumerate(lengths):
        assert not gpu["y"][ln:, n].any(), n


def test_gru_tf_dropout():
    case = (3, True, 6, 4, 8, 12, "f32")
    cfg = _cfg(case, tag="dropout")
    inp = wl.make_inputs(cfg)
    rng = np.random.default_rng(5)
    masks = (rng.random((2, 6, 4, 24)) >= 0.3).astype(np.uint8)
    gpu = harness.run_gpu(cfg, inp, inference=False, dropout=(0.3, masks))
    ref = harness.run_oracle(cfg, inp, dropout=(0.3, list(masks.astype(np.float64))))
    harness.assert_parity(cfg, gpu, ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gru_tf_ds2_shape(dtype):
    base = wl.WORKLOADS["ds2_gru"]
    cfg = dict(base, mode="gru_tf", dtype=dtype, name="ds2_gru_tf_" + dtype)
    inp = wl.make_inputs(cfg)
    gpu = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    res = harness.assert_parity(cfg, gpu, ref)
    print(cfg["name"], {k: "%.2e" % v[0] for k, v in res.items()
                        if not k.startswith("d") or k in ("dx", "dh0")})
    assert np.array_equal(gpu["y_inf"], gpu["y"])
