"""Host-side checks of the C ABI (no GPU needed): the library loads and exports
every symbol the header declares; argument validation; the canonical weight
layout agrees with the oracle's independent layout; workspace regions are
aligned and disjoint."""

import ctypes
import os
import re

import numpy as np
import pytest

from layer_rnn_gb300 import workloads as wl
from tests import harness

HEADER = os.path.join(harness.ROOT, "include", "layer_rnn.h")


@pytest.fixture(scope="module")
def B():
    if not os.path.exists("/usr/local/cuda/bin/nvcc") and not os.path.exists(
            os.path.join(harness.ROOT, "layer_rnn_gb300", "liblayer_rnn.so")):
        pytest.skip("no nvcc and no prebuilt library")
    harness.ensure_built()
    from layer_rnn_gb300 import binding
    binding.lib()
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rnn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("rnn_create", "rnn_destroy", "rnn_weight_layout", "rnn_workspace_size",
               "rnn_forward_training", "rnn_forward_inference", "rnn_backward_data",
               "rnn_backward_weights"):
        assert fn in names


def test_library_exports_every_declared_symbol(B):
    L = ctypes.CDLL(B.LIB_PATH)
    for name in declared_functions():
        assert hasattr(L, name), name
    # and the binding knows every one of them
    assert set(declared_functions()) == set(B.SIGNATURES)


def test_create_validates_arguments(B):
    h = ctypes.c_void_p()
    lib = B.lib()
    bad = [(4, 1, 0, 4, 4, 0), (-1, 1, 0, 4, 4, 0), (1, 0, 0, 4, 4, 0), (1, 1, 2, 4, 4, 0), (1, 1, 0, 0, 4, 0),
           (1, 1, 0, 4, 0, 0), (1, 1, 0, 4, 4, 2)]
    for args in bad:
        assert lib.rnn_create(ctypes.byref(h), *args, 0) == 1, args
    assert lib.rnn_create(ctypes.byref(h), 1, 1, 0, 4, 4, 0, 0x80) == 1
    assert lib.rnn_create(None, 1, 1, 0, 4, 4, 0, 0) == 1
    assert lib.rnn_create(ctypes.byref(h), 1, 1, 0, 4, 70000, 0, 0) == 2
    assert lib.rnn_destroy(None) == 0
    assert B.rnn_status_string(6) == "step barrier timed out"


@pytest.mark.parametrize("mode,L,bidir,I,H", [("lstm", 1, False, 4, 8), ("gru", 3, True, 5, 7),
                                              ("gru_tf", 2, True, 5, 7),
                                              ("rnn_tanh", 2, True, 800, 800),
                                              ("lstm", 4, False, 1024, 1024)])
def test_weight_layout_matches_oracle_layout(B, mode, L, bidir, I, H):
    import oracle
    h = B.rnn_create(B.MODES[mode], L, bidir, I, H, 0)
    try:
        cfg = wl.make_config(mode, L, bidir, 1, 1, I, H)
        assert B.rnn_weight_count(h) == wl.weight_count(cfg)
        D = 2 if bidir else 1
        pos = 0
        names = ["W_ih", "W_hh", "b_ih", "b_hh"]
        for l, d, name, shape in oracle.weight_shapes(mode, L, bidir, I, H):
            off, rows, cols = B.rnn_weight_layout(h, l, d, names.index(name))
            assert off == pos
            assert rows * cols == int(np.prod(shape))
            assert rows == shape[0]
            pos += int(np.prod(shape))
        assert pos == B.rnn_weight_count(h)
        with pytest.raises(B.RnnError):
            B.rnn_weight_layout(h, L, 0, 0)
        with pytest.raises(B.RnnError):
            B.rnn_weight_layout(h, 0, D, 0)
    finally:
        B.rnn_destroy(h)


@pytest.mark.parametrize("mode,L,bidir,dtype", [("lstm", 1, False, 0), ("gru", 2, True, 0),
                                                ("gru_tf", 2, False, 1),
                                                ("rnn_tanh", 3, True, 1), ("lstm", 4, False, 1)])
def test_workspace_regions_disjoint_and_aligned(B, mode, L, bidir, dtype):
    T, N, I, H = 7, 3, 5, 6
    h = B.rnn_create(B.MODES[mode], L, bidir, I, H, dtype)
    try:
        total = B.rnn_workspace_size(h, T, N)
        D = 2 if bidir else 1
        spans = []
        for region in range(9):
            per_layer = region == B.RNN_WS_YLAYER
            glob = region in (B.RNN_WS_GX, B.RNN_WS_DY, B.RNN_WS_GEMM)
            for l in range(1 if glob else L):
                for d in range(1 if (glob or per_layer) else D):
                    off, nb = B.rnn_workspace_layout(h, T, N, region, l, d)
                    if nb == 0:
                        continue
                    assert off % 256 == 0
                    assert off + nb <= total
                    spans.append((off, off + nb, region, l, d))
        spans = sorted(set(spans))
        for a, b in zip(spans, spans[1:]):
            assert a[1] <= b[0], (a, b)
        e = 2 if dtype else 4
        G = {"lstm": 4, "gru": 3, "gru_tf": 3, "rnn_tanh": 1}[mode]
        assert B.rnn_workspace_layout(h, T, N, B.RNN_WS_DGX, 0, 0)[1] == T * N * G * H * e
        assert B.rnn_workspace_layout(h, T, N, B.RNN_WS_HSEQ, 0, 0)[1] == (T + 1) * N * H * e
        assert (B.rnn_workspace_layout(h, T, N, B.RNN_WS_CSEQ, 0, 0)[1] > 0) == (mode == "lstm")
        assert (B.rnn_workspace_layout(h, T, N, B.RNN_WS_DGH, 0, 0)[1] > 0) == (mode == "gru")
        with pytest.raises(B.RnnError):
            B.rnn_workspace_size(h, 0, N)
        with pytest.raises(B.RnnError):
            B.rnn_workspace_layout(h, T, N, 9, 0, 0)
    finally:
        B.rnn_destroy(h)


def test_compute_calls_reject_bad_arguments_before_any_launch(B):
    # null / misaligned pointers and a short workspace are refused on the host
    lib = B.lib()
    h = B.rnn_create(B.RNN_LSTM, 1, False, 4, 8, 0)
    try:
        ws = B.rnn_workspace_size(h, 5, 2)
        assert lib.rnn_forward_training(h, None, 5, 2, None, None, None, 256, 256, None, None,
                                        256, ws) == 1
        assert lib.rnn_forward_training(h, None, 5, 2, 260, None, None, 256, 256, None, None,
                                        256, ws) == 4
        assert lib.rnn_forward_training(h, None, 5, 2, 256, None, None, 256, 256, None, None,
                                        256 + 16, ws) == 4
        assert lib.rnn_forward_training(h, None, 5, 2, 256, None, None, 256, 256, None, None,
                                        256, ws - 1) == 3
        assert lib.rnn_backward_data(h, None, 5, 2, 256, None, None, None, 256, None, None, 256,
                                     ws) == 1
        assert lib.rnn_backward_weights(h, None, 5, 2, 256, None, None, 256, ws - 1, 256) == 3
        assert lib.rnn_forward_inference(h, None, 0, 2, 256, None, None, 256, 256, None,
                                         None) == 1
    finally:
        B.rnn_destroy(h)


def test_varlen_calls_reject_bad_arguments_before_any_launch(B):
    # a NULL or misaligned lengths buffer, then the checks of the calls without
    # lengths, all on the host
    lib = B.lib()
    h = B.rnn_create(B.RNN_GRU, 1, True, 4, 8, 0)
    try:
        ws = B.rnn_workspace_size(h, 5, 2)
        assert lib.rnn_forward_training_varlen(h, None, 5, 2, None, 256, None, None, 256, 256,
                                               None, None, 256, ws) == 1
        assert lib.rnn_forward_inference_varlen(h, None, 5, 2, None, 256, None, None, 256, 256,
                                                None, None) == 1
        assert lib.rnn_backward_data_varlen(h, None, 5, 2, None, 256, 256, None, None, 256, None,
                                            None, 256, ws) == 1
        assert lib.rnn_forward_training_varlen(h, None, 5, 2, 258, 256, None, None, 256, 256,
                                               None, None, 256, ws) == 4
        assert lib.rnn_forward_inference_varlen(h, None, 5, 2, 258, 256, None, None, 256, 256,
                                                None, None) == 4
        assert lib.rnn_backward_data_varlen(h, None, 5, 2, 258, 256, 256, None, None, 256, None,
                                            None, 256, ws) == 4
        assert lib.rnn_forward_training_varlen(h, None, 5, 2, 512, None, None, None, 256, 256,
                                               None, None, 256, ws) == 1
        assert lib.rnn_forward_training_varlen(h, None, 5, 2, 512, 256, None, None, 256, 256,
                                               None, None, 256, ws - 1) == 3
        assert lib.rnn_backward_data_varlen(h, None, 5, 2, 512, 256, 256, None, None, 256, None,
                                            None, 256, ws - 1) == 3
        assert lib.rnn_forward_inference_varlen(h, None, 0, 2, 512, 256, None, None, 256, 256,
                                                None, None) == 1
    finally:
        B.rnn_destroy(h)


def test_dropout_calls_reject_bad_arguments_before_any_launch(B):
    lib = B.lib()
    h = B.rnn_create(B.RNN_LSTM, 2, False, 4, 8, 0)
    try:
        ws = B.rnn_workspace_size(h, 5, 2)
        args = (256, None, None, 256, 256, None, None, 256, ws)
        for p, masks in ((0.2, None), (1.0, 512), (-0.1, 512), (float("nan"), 512)):
            assert lib.rnn_forward_training_dropout(h, None, 5, 2, p, masks, *args) == 1, p
            assert lib.rnn_backward_data_dropout(h, None, 5, 2, p, masks, 256, 256, None, None,
                                                 256, None, None, 256, ws) == 1, p
        # the checks of the calls without dropout still apply
        assert lib.rnn_forward_training_dropout(h, None, 5, 2, 0.2, 512, 256, None, None, 256,
                                                256, None, None, 256, ws - 1) == 3
    finally:
        B.rnn_destroy(h)


@pytest.mark.parametrize("shape,expect", [
    # the DS2 layer's dense GEMMs on 148 SMs (fp32, scaled fp16 pairs)
    ((6000, 3200, 800, 1), (256, 1)),   # input projection: 5 waves of 47 x 13
    ((6000, 800, 3200, 1), (160, 1)),   # dX: 2 waves of 47 x 5 (3 of 47 x 7 at 128)
    ((3200, 800, 6000, 1), (160, 1)),   # dW: one wave of 25 x 5, no split
    # bf16 stacks: the widest tile
    ((65536, 4096, 1024, 0), (256, 1)),
    # narrow outputs take 64-wide tiles
    ((1000, 48, 256, 1), (64, 1)),
])
def test_gemm_shape_model_picks_the_documented_shapes(B, shape, expect):
    M, N, K, sp = shape
    assert B.rnn_debug_gemm_shape(M, N, K, sp, 148) == expect


def test_gemm_shape_model_properties(B):
    rng = np.random.default_rng(7)
    for _ in range(200):
        M, N, K = (int(v) for v in rng.integers(1, 20000, size=3))
        sp = int(rng.integers(0, 2))
        bn, ks = B.rnn_debug_gemm_shape(M, N, K, sp, 148)
        assert bn in (64, 128, 160, 192, 256) and 1 <= ks <= 8
        assert (bn == 64) == (N <= 64)
        assert bn <= max(128, (N + 31) // 32 * 32)
        nkt = (K * 2 + 127) // 128
        assert ks == 1 or nkt // ks >= 4
        assert B.rnn_debug_gemm_shape(M, N, K, sp, 148, allow_split=False)[1] == 1
    with pytest.raises(B.RnnError):
        B.rnn_debug_gemm_shape(0, 10, 10, 1, 148)
