"""Shared helpers for the tests: library build check, device marshalling and
the parity metric.

Parity metric (per output tensor): normwise maximum relative error
``max|gpu - ref| / max|ref|`` -- robust to entries of the reference near zero.
Bars: 1e-4 for fp32 forward outputs (y, hy, cy), 1e-3 for fp32 gradients
(dx, dh0, dc0, every weight / bias gradient tensor), 2e-2 for every output of
a bf16 workload.  Reported beside it: the elementwise relative error
``|gpu - ref| / max(|ref|, 1e-6 max|ref|)`` at its 99.9th percentile.
"""

import os

import numpy as np

from layer_rnn_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TOL_F32_FWD = 1e-4
TOL_F32_GRAD = 1e-3
TOL_BF16 = 2e-2


def ensure_built():
    """Build liblayer_rnn.so when it is missing or older than its sources."""
    from layer_rnn_gb300 import build_lib
    lib = build_lib.LIB
    srcs = build_lib.sources() + [os.path.join(ROOT, "include", "layer_rnn.h")]
    srcs += [os.path.join(build_lib.CSRC, f) for f in os.listdir(build_lib.CSRC)
             if f.endswith((".cuh", ".h"))]
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs):
        build_lib.build()
    return lib


def rel_err(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    scale = np.abs(ref).max() if ref.size else 0.0
    diff = np.abs(gpu - ref).max() if ref.size else 0.0
    if scale == 0.0:
        return float(diff)
    return float(diff / scale)


def elementwise_err(gpu, ref, q=99.9):
    """The q-th percentile over the entries of |gpu - ref| / max(|ref|,
    1e-6 * max|ref|): the elementwise relative error reported beside the
    normwise one, which a few large entries can dominate."""
    gpu = np.asarray(gpu, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    floor = 1e-6 * np.abs(ref).max()
    if floor == 0.0:
        return float(np.percentile(np.abs(gpu - ref), q))
    return float(np.percentile(np.abs(gpu - ref) / np.maximum(np.abs(ref), floor), q))


def tolerances(cfg):
    if cfg["dtype"] == "bf16":
        return TOL_BF16, TOL_BF16
    return TOL_F32_FWD, TOL_F32_GRAD


# ----------------------------------------------------------------------------
# device marshalling (torch is used for device memory and streams only)
# ----------------------------------------------------------------------------

from layer_rnn_gb300.tensors import empty, from_dev, to_dev  # noqa: E402,F401


def run_gpu(cfg, inp, flags=0, poison=True, inference=True, stream=None, lengths=None,
            dropout=None):
    """Training forward + backward_data + backward_weights (+ inference forward)
    through the C ABI.  Returns float64 numpy arrays.  lengths: per-sequence
    valid lengths [N] (the *_varlen calls), or None.  dropout: (p, masks) with
    masks [L-1, T, N, D*H] of 0/1 (the *_dropout calls), or None."""
    import torch
    from layer_rnn_gb300 import binding as B
    T, N, I, H, L = cfg["T"], cfg["N"], cfg["I"], cfg["H"], cfg["L"]
    D = wl.num_directions(cfg)
    dt = cfg["dtype"]
    lstm = cfg["mode"] == "lstm"
    r = B.Rnn(cfg["mode"], L, cfg["bidir"], I, H, dt, flags | B.RNN_FLAG_SYNC_CHECK)
    try:
        assert r.weight_count() == inp["w"].size
        x = to_dev(inp["x"], dt)
        h0 = to_dev(inp["h0"], dt)
        c0 = to_dev(inp["c0"], "f32") if lstm else None
        W = to_dev(inp["w"], dt)
        dy = to_dev(inp["dy"], dt)
        dhy = to_dev(inp["dhy"], dt)
        dcy = to_dev(inp["dcy"], "f32") if lstm else None
        y = empty((T, N, D * H), dt)
        hy = empty((L * D, N, H), dt)
        cy = empty((L * D, N, H), "f32") if lstm else None
        ws = r.alloc_workspace(T, N)
        if poison:
            ws.fill_(0xFF)  # NaN bit patterns: anything read before written shows
            y.fill_(float("nan"))
        lens = masks = None
        if lengths is not None:
            lens = torch.tensor(np.asarray(lengths), dtype=torch.int32, device="cuda")
            r.forward_training_varlen(lens, x, h0, c0, W, y, hy, cy, ws, stream)
        elif dropout is not None:
            masks = torch.tensor(np.asarray(dropout[1]), dtype=torch.uint8, device="cuda")
            r.forward_training_dropout(dropout[0], masks, x, h0, c0, W, y, hy, cy, ws, stream)
        else:
            r.forward_training(x, h0, c0, W, y, hy, cy, ws, stream)
        dx = empty((T, N, I), dt)
        dh0 = empty((L * D, N, H), dt)
        dc0 = empty((L * D, N, H), "f32") if lstm else None
        dW = empty((inp["w"].size,), dt)
        if poison:
            dW.fill_(float("nan"))
            dx.fill_(float("nan"))
        if lens is not None:
            r.backward_data_varlen(lens, W, dy, dhy, dcy, dx, dh0, dc0, ws, stream)
        elif masks is not None:
            r.backward_data_dropout(dropout[0], masks, W, dy, dhy, dcy, dx, dh0, dc0, ws, stream)
        else:
            r.backward_data(W, dy, dhy, dcy, dx, dh0, dc0, ws, stream)
        r.backward_weights(x, h0, y, ws, dW, stream)
        out = dict(y=from_dev(y), hy=from_dev(hy), cy=from_dev(cy), dx=from_dev(dx),
                   dh0=from_dev(dh0), dc0=from_dev(dc0), dW=from_dev(dW))
        if inference:
            yi = empty((T, N, D * H), dt)
            hyi = empty((L * D, N, H), dt)
            cyi = empty((L * D, N, H), "f32") if lstm else None
            if lens is not None:
                r.forward_inference_varlen(lens, x, h0, c0, W, yi, hyi, cyi, stream)
            else:
                r.forward_inference(x, h0, c0, W, yi, hyi, cyi, stream)
            out["y_inf"] = from_dev(yi)
            out["hy_inf"] = from_dev(hyi)
            out["cy_inf"] = from_dev(cyi)
        torch.cuda.synchronize()
        return out
    finally:
        r.close()


def run_oracle(cfg, inp, lengths=None, dropout=None):
    import oracle
    p, masks = dropout if dropout is not None else (0.0, None)
    return oracle.run_flat(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"], inp["x"],
                           inp["h0"], inp["c0"], inp["w"], inp["dy"], inp["dhy"], inp["dcy"],
                           lengths=lengths, dropout=p, masks=masks)


def weight_tensors(cfg, flat):
    """Split a flat canonical buffer into named per-(l,d) tensors (sizes only)."""
    import oracle
    params = oracle.unflatten_weights(flat, cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"],
                                      cfg["H"])
    D = wl.num_directions(cfg)
    out = {}
    for k, p in enumerate(params):
        for name, v in p.items():
            out["%s[l%d,d%d]" % (name, k // D, k % D)] = v
    return out


def compare(cfg, gpu, ref):
    """Dict name -> (error, bar) for every output."""
    tf, tg = tolerances(cfg)
    res = {}
    for k in ("y", "hy", "cy"):
        if ref[k] is not None:
            res[k] = (rel_err(gpu[k], ref[k]), tf)
    for k in ("dx", "dh0", "dc0"):
        if ref[k] is not None:
            res[k] = (rel_err(gpu[k], ref[k]), tg)
    gw = weight_tensors(cfg, gpu["dW"])
    rw = weight_tensors(cfg, ref["dW"])
    for k in rw:
        res["d" + k] = (rel_err(gw[k], rw[k]), tg)
    return res


def elementwise_report(cfg, gpu, ref):
    """Dict name -> 99.9th-percentile elementwise relative error, for every
    output compare() covers."""
    res = {}
    for k in ("y", "hy", "cy", "dx", "dh0", "dc0"):
        if ref[k] is not None:
            res[k] = elementwise_err(gpu[k], ref[k])
    gw = weight_tensors(cfg, gpu["dW"])
    rw = weight_tensors(cfg, ref["dW"])
    for k in rw:
        res["d" + k] = elementwise_err(gw[k], rw[k])
    return res


def assert_parity(cfg, gpu, ref):
    res = compare(cfg, gpu, ref)
    bad = {k: v for k, v in res.items() if not (v[0] <= v[1])}
    worst = max(res.items(), key=lambda kv: kv[1][0] / kv[1][1])
    assert not bad, "parity failures %s (worst %s)" % (bad, worst)
    return res
