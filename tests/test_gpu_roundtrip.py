"""Bit-exact round trips of the packed operand forms, through the C ABI test
hooks: every packed form the kernels read must hold exactly the canonical
values, nothing lost, nothing invented.

* scaled fp16 pairs of the dense phases' fp32 operands: the largest
  magnitude, the power-of-two scale it fixes, hi = fp16(value * s) and
  lo = fp16(value * s - hi) bit for bit as documented, hi + lo within 2^-22
  of value * s; the transposing variants put element (i, j) at (j, i).  The
  shapes cover the vectorised, tiled-transpose and generic kernels (aligned
  and ragged sizes).
* bf16 K-major copies: dst == src^T bit for bit, aligned and ragged.
* the layer wavefront's packed rows: unpacked here from the documented
  layout (independently of the library), every row equals the canonical
  W_ih / W_hh row of its unit and gate, the pads are zero, the biases are the
  folded sums ("Exposing Cudnn v5 RNN models" (Keras issue #3692), the
  "matrix pre-transposition" rung of its cuDNN table names the packing).
"""

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


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("rows,cols,transpose", [
    (256, 800, 0), (6000 // 8, 800, 1), (3200, 64, 1),   # vectorised / tiled transpose
    (37, 19, 0), (37, 19, 1), (130, 75, 1), (1, 1, 0),    # ragged: the generic kernel
])
def test_f16_split_pairs(rows, cols, transpose):
    import torch
    from layer_rnn_gb300 import binding as B
    rng = np.random.Generator(np.random.PCG64(rows * 1000 + cols))
    # magnitudes over many binades, negative zero, subnormals
    v = (rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-12, 12, (rows, cols))))
    v = v.astype(np.float32)
    v.ravel()[:3] = np.array([-0.0, 1e-40, -3e-39], dtype=np.float32)[: min(3, v.size)]
    src = torch.from_numpy(v).cuda()
    shape = (cols, rows) if transpose else (rows, cols)
    hi = torch.full(shape, float("nan"), dtype=torch.float16, device="cuda")
    lo = torch.full(shape, float("nan"), dtype=torch.float16, device="cuda")
    mx = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    B.rnn_debug_split_f16(src.data_ptr(), rows, cols, cols, hi.data_ptr(), lo.data_ptr(),
                          shape[1], transpose, mx.data_ptr(), _stream())
    torch.cuda.synchronize()
    ref = v.T if transpose else v
    mb = int(mx[0].item()) & 0xFFFFFFFF
    assert mb == int(np.abs(v).max().view(np.uint32))
    # the documented scale: the largest magnitude lands in [2^13, 2^14)
    E = (mb >> 23) - 127
    s = 1.0 if mb == 0 or mb >= 0x7F800000 else 2.0 ** min(max(13 - E, -126), 126)
    x = (ref.astype(np.float64) * s).astype(np.float32)  # exact: s is a power of two
    eh = x.astype(np.float16)                             # round to nearest even
    el = (x - eh.astype(np.float32)).astype(np.float16)   # x - hi is exact in fp32
    h, l = hi.cpu().numpy(), lo.cpu().numpy()
    assert np.array_equal(h.view(np.uint16), eh.view(np.uint16))
    assert np.array_equal(l.view(np.uint16), el.view(np.uint16))
    err = np.abs(x.astype(np.float64) - h.astype(np.float64) - l.astype(np.float64))
    assert np.all(err <= 2.0 ** -22 * np.abs(x) + 2.0 ** -25)


@pytest.mark.parametrize("rows,cols", [(512, 1024), (128, 4096), (33, 17), (200, 72)])
def test_bf16_transpose_is_exact(rows, cols):
    import torch
    from layer_rnn_gb300 import binding as B
    rng = np.random.Generator(np.random.PCG64(rows + 7 * cols))
    bits = rng.integers(0, 1 << 16, (rows, cols), dtype=np.uint16)
    src = torch.from_numpy(bits.view(np.int16)).cuda()
    dst = torch.full((cols, rows), -1, dtype=torch.int16, device="cuda")
    B.rnn_debug_transpose_bf16(src.data_ptr(), rows, cols, cols, dst.data_ptr(), rows,
                               _stream())
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy().view(np.uint16), bits.T)


@pytest.mark.parametrize("mode", ["lstm", "gru", "rnn_tanh"])
@pytest.mark.parametrize("layer", [0, 1])
def test_wavefront_rows_are_the_canonical_rows(mode, layer):
    import oracle
    import torch
    from layer_rnn_gb300 import binding as B
    cfg = wl.make_config(mode, 2, False, 4, 16, 72, 104, "bf16", 0.0, seed=41)
    inp = wl.make_inputs(cfg)
    H, I = cfg["H"], cfg["I"]
    r = B.Rnn(mode, 2, False, I, H, "bf16", 0)
    try:
        W = harness.to_dev(inp["w"], "bf16")
        cap_rows, cap_k = 4 * (H + 256), I + H + 256
        wp = torch.full((cap_rows * cap_k,), -1, dtype=torch.int16, device="cuda")
        bias = torch.full((cap_rows,), float("nan"), dtype=torch.float32, device="cuda")
        Pr, Ur, R, kp, Kxp = B.rnn_debug_wf_pack(r.h, _stream(), cfg["N"], layer, W.data_ptr(),
                                                 wp.data_ptr(), wp.numel() * 2,
                                                 bias.data_ptr(), bias.numel() * 4)
        torch.cuda.synchronize()
    finally:
        r.close()
    rows = Pr * Ur * R
    packed = wp.cpu().numpy()[: rows * kp].view(np.uint16).reshape(rows, kp)
    pb = bias.cpu().numpy()[:rows]
    params = oracle.unflatten_weights(inp["w"], mode, 2, False, I, H)[layer]
    I_l = I if layer == 0 else H
    bits = lambda a: wl.to_storage(a, "bf16").view(np.uint16)  # noqa: E731
    wih, whh = bits(params["W_ih"]), bits(params["W_hh"])
    bih = params["b_ih"].astype(np.float64)
    bhh = params["b_hh"].astype(np.float64)
    assert Pr * Ur >= H and R == (1 if mode == "rnn_tanh" else 4) and Kxp >= I_l
    for blk in range(Pr):
        for u in range(Ur):
            j = blk * Ur + u
            for g in range(R):
                row = packed[(blk * Ur + u) * R + g]
                if j >= H:
                    assert not row.any() and pb[(blk * Ur + u) * R + g] == 0.0
                    continue
                src = 2 if (mode == "gru" and g == 3) else g
                use_x = not (mode == "gru" and g == 3)
                use_h = not (mode == "gru" and g == 2)
                x_part = wih[src * H + j] if use_x else np.zeros(I_l, np.uint16)
                h_part = whh[src * H + j] if use_h else np.zeros(H, np.uint16)
                assert np.array_equal(row[:I_l], x_part), (blk, u, g)
                assert not row[I_l:Kxp].any()
                assert np.array_equal(row[Kxp:Kxp + H], h_part), (blk, u, g)
                assert not row[Kxp + H:].any()
                if mode == "gru" and g == 2:
                    b = bih[src * H + j]
                elif mode == "gru" and g == 3:
                    b = bhh[src * H + j]
                else:
                    b = np.float32(np.float32(bih[src * H + j]) + np.float32(bhh[src * H + j]))
                assert pb[(blk * Ur + u) * R + g] == np.float32(b), (blk, u, g)
