"""Variable-length (padded) batches through the C ABI against the float64
oracle with the same lengths: rnn_forward_training_varlen,
rnn_backward_data_varlen, rnn_backward_weights and
rnn_forward_inference_varlen.

Lengths cover the degenerate cases: 0 (nothing runs: y is zero, hy = h0,
dh0 = dhy), 1, T - 1 and T; both directions and stacked layers (the reverse
direction starts at each sequence's last valid step; the layer above reads
zeros past the length), fp32 and bf16, batches that are not multiples of a
tile.  The tensor-core recurrent kernels run the shapes they fit (their
choice is asserted for the DS2 hidden size, both modes, and for a
bidirectional layer whose directions run in turn); the staged CUDA-core
kernels run the same lengths when the tensor cores are switched off.
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


# shapes whose recurrent phases take the tensor-core kernels or the layer
# wavefront with lengths: mode, L, bidir, T, N, I, H, dtype, (fwd, bwd) paths
TC_CASES = [
    ("lstm", 1, False, 9, 20, 48, 800, "f32", ("tensor", "tensor")),  # the DS2 layer
    ("gru", 1, False, 8, 48, 40, 800, "f32", ("tensor", "tensor")),
    ("lstm", 1, True, 5, 24, 32, 800, "f32", ("tensor", "tensor")),   # directions in turn
    ("rnn_tanh", 1, False, 7, 40, 24, 256, "f32", ("tensor", "tensor")),
    ("gru", 1, True, 6, 36, 16, 200, "bf16", ("tensor", "tensor")),
    # unidirectional bf16 stacks: the wavefront; batches of 64..128 take the
    # batch-as-M backward
    ("lstm", 2, False, 6, 72, 16, 256, "bf16", ("wavefront", "tensor")),
    ("lstm", 4, False, 7, 128, 32, 128, "bf16", ("wavefront", "tensor")),
    ("gru", 3, False, 8, 40, 16, 48, "bf16", ("wavefront", "tensor")),
    ("rnn_tanh", 2, False, 9, 96, 24, 40, "bf16", ("wavefront", "tensor")),
]


def _paths(cfg, flags=0):
    from layer_rnn_gb300 import binding as B
    r = B.Rnn(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"], cfg["dtype"], flags)
    try:
        return B.rnn_get_paths_varlen(r.h, cfg["N"])
    finally:
        r.close()


def _check_case(case, flags=0, expect=None):
    mode, L, bidir, T, N, I, H, dt = case
    seed = zlib.crc32(_cid(case).encode()) % 10000
    cfg = wl.make_config(mode, L, bidir, T, N, I, H, dt, 0.3, seed=seed)
    if expect is not None:
        assert _paths(cfg, flags) == expect
    inp = wl.make_inputs(cfg)
    lengths = _lengths(T, N, seed)
    gpu = harness.run_gpu(cfg, inp, lengths=lengths, flags=flags)
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


@pytest.mark.parametrize("case", CASES, ids=[_cid(c) for c in CASES])
def test_varlen_parity(case):
    _check_case(case)


@pytest.mark.parametrize("case", TC_CASES, ids=[_cid(c[:8]) for c in TC_CASES])
def test_varlen_tensor_core_kernels(case):
    _check_case(case[:8], expect=case[8])


STAGED = [CASES[3], CASES[6], TC_CASES[0][:8], TC_CASES[6][:8]]


@pytest.mark.parametrize("case", STAGED, ids=[_cid(c) for c in STAGED])
def test_varlen_staged_kernels(case):
    from layer_rnn_gb300 import binding as B
    _check_case(case, flags=B.RNN_FLAG_SIMT_RECURRENT, expect=("staged", "staged"))


@pytest.mark.parametrize("shape", [(6, 8, 16, 32), (5, 20, 32, 800)])
def test_full_lengths_match_the_fixed_length_calls(shape):
    # every length equal to T: the varlen calls and the fixed-length calls
    # agree with each other within the bars, and bit for bit where both run
    # the same recurrent kernels
    from layer_rnn_gb300 import binding as B
    T, N, I, H = shape
    cfg = wl.make_config("gru", 1, True, T, N, I, H, "f32", 0.3, seed=3)
    inp = wl.make_inputs(cfg)
    a = harness.run_gpu(cfg, inp, lengths=np.full(N, T, dtype=np.int32))
    b = harness.run_gpu(cfg, inp)
    ref = harness.run_oracle(cfg, inp)
    harness.assert_parity(cfg, a, ref)
    harness.assert_parity(cfg, b, ref)
    r = B.Rnn(cfg["mode"], cfg["L"], cfg["bidir"], I, H, cfg["dtype"], 0)
    try:
        same = B.rnn_get_paths_varlen(r.h, N) == B.rnn_get_paths(r.h, N)
    finally:
        r.close()
    if same:
        for k in ("y", "hy", "dx", "dh0", "dW"):
            assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("shape", [("lstm", 3, 8, 24, 16, 32), ("gru", 2, 6, 80, 16, 48),
                                   ("rnn_tanh", 2, 5, 16, 8, 24)])
def test_full_lengths_on_the_wavefront(shape):
    # every length equal to T on a unidirectional bf16 stack: the varlen calls
    # run the wavefront and the tensor-core backward as the fixed-length calls
    # do, and give the same results bit for bit
    from layer_rnn_gb300 import binding as B
    mode, L, T, N, I, H = shape
    cfg = wl.make_config(mode, L, False, T, N, I, H, "bf16", 0.3, seed=5)
    r = B.Rnn(mode, L, False, I, H, "bf16", 0)
    try:
        paths = B.rnn_get_paths_varlen(r.h, N)
        assert paths == B.rnn_get_paths(r.h, N)
        assert paths[0] == "wavefront"
    finally:
        r.close()
    inp = wl.make_inputs(cfg)
    a = harness.run_gpu(cfg, inp, lengths=np.full(N, T, dtype=np.int32))
    b = harness.run_gpu(cfg, inp)
    for k in ("y", "hy", "cy", "dx", "dh0", "dc0", "dW", "y_inf", "hy_inf"):
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("name", ["ds2_lstm", "ds2_gru", "lstm4_bf16"])
def test_varlen_workload_parity(name):
    # the bench's batches with the bench's lengths (one sequence of length T,
    # the others uniform in [T/2, T]), at full size, in the bench's launch
    # configuration
    cfg = wl.WORKLOADS[name]
    inp = wl.make_inputs(cfg)
    lengths = wl.make_lengths(cfg)
    gpu = harness.run_gpu(cfg, inp, lengths=lengths)
    ref = harness.run_oracle(cfg, inp, lengths=lengths)
    harness.assert_parity(cfg, gpu, ref)
    for n, ln in enumerate(lengths):
        assert not gpu["y"][ln:, n].any(), n
    assert np.array_equal(gpu["y_inf"], gpu["y"])
