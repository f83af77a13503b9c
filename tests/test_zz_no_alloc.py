"""rnn_forward_inference_static: the inference forward that allocates nothing.

Callers that cannot allocate device memory (a memory pool that owns the device,
an allocator that must not be re-entered, a fixed memory budget) use this
entry point instead of rnn_forward_inference, which allocates its scratch on
first use.  Its scratch lives in a 32 MiB static device array.  This file is
collected last so that a failure here does not hide the other tests.
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


def _inputs(cfg, seed):
    inp = wl.make_inputs(cfg, seed=seed)
    dt = cfg["dtype"]
    lstm = cfg["mode"] == "lstm"
    return dict(x=harness.to_dev(inp["x"], dt), h0=harness.to_dev(inp["h0"], dt),
                c0=harness.to_dev(inp["c0"], "f32") if lstm else None,
                W=harness.to_dev(inp["w"], dt))


def _outputs(cfg):
    T, N, H, L = cfg["T"], cfg["N"], cfg["H"], cfg["L"]
    D = wl.num_directions(cfg)
    dt = cfg["dtype"]
    lstm = cfg["mode"] == "lstm"
    return dict(y=harness.empty((T, N, D * H), dt), hy=harness.empty((L * D, N, H), dt),
                cy=harness.empty((L * D, N, H), "f32") if lstm else None)


def _call(B, fn, r, cfg, i, o):
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    fn(r.h, r._stream(None), cfg["T"], cfg["N"], ptr(i["x"]), ptr(i["h0"]), ptr(i["c0"]),
       ptr(i["W"]), ptr(o["y"]), ptr(o["hy"]), ptr(o["cy"]))


CASES = [
    wl.make_config("gru", 2, True, 40, 6, 48, 72, "f32", 0.3, seed=61, name="gru_bi2"),
    wl.make_config("lstm", 1, False, 300, 4, 800, 800, "f32", 0.0, seed=62, name="ds2_lstm_n4"),
    wl.make_config("lstm", 3, False, 30, 16, 64, 128, "bf16", 0.2, seed=63, name="lstm3_bf16"),
]


@pytest.mark.parametrize("cfg", CASES, ids=[c["name"] for c in CASES])
def test_static_scratch_matches_allocating_entry_point(cfg):
    import torch
    from layer_rnn_gb300 import binding as B
    r = B.Rnn(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"], cfg["dtype"],
              B.RNN_FLAG_SYNC_CHECK)
    try:
        tol = harness.tolerances(cfg)[0]
        for call, seed in enumerate((cfg["seed"], cfg["seed"] + 1000)):  # two calls in a row
            i = _inputs(cfg, seed)
            ref = _outputs(cfg)
            got = _outputs(cfg)
            for t in got.values():
                if t is not None:
                    t.fill_(float("nan"))
            _call(B, B.rnn_forward_inference, r, cfg, i, ref)
            free_before = torch.cuda.mem_get_info()[0]
            _call(B, B.rnn_forward_inference_static, r, cfg, i, got)
            torch.cuda.synchronize()
            if call == 1:
                # nothing allocated by the second call
                assert torch.cuda.mem_get_info()[0] == free_before
            for k in ("y", "hy", "cy"):
                if ref[k] is None:
                    continue
                a, b = harness.from_dev(got[k]), harness.from_dev(ref[k])
                assert np.all(np.isfinite(a)), (call, k)
                assert harness.rel_err(a, b) <= tol, (call, k, harness.rel_err(a, b))
    finally:
        r.close()


def test_static_scratch_rejects_oversized_problems():
    from layer_rnn_gb300 import binding as B
    cfg = wl.WORKLOADS["ds2_lstm"]  # input projection 76.8 MB > 32 MiB
    r = B.Rnn("lstm", 1, False, cfg["I"], cfg["H"], "f32", 0)
    try:
        i = _inputs(wl.with_sizes(cfg, T=2), cfg["seed"])
        o = _outputs(wl.with_sizes(cfg, T=2))
        ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        code = B.lib().rnn_forward_inference_static(
            r.h, r._stream(None), cfg["T"], cfg["N"], ptr(i["x"]), None, None, ptr(i["W"]),
            ptr(o["y"]), None, None)
        assert code == 3  # RNN_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
    finally:
        r.close()


def test_static_call_timeout_is_reported_by_check_status():
    """A step barrier that runs out of time inside a static call (one block
    skips its flag release, so the others wait until the short limit) is
    recorded in the array's own status word: rnn_check_status returns it and
    clears it, and the next static call is correct again."""
    import torch
    from layer_rnn_gb300 import binding as B
    cfg = CASES[0]
    r = B.Rnn(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"], cfg["dtype"], 0)
    try:
        i = _inputs(cfg, cfg["seed"])
        ref = _outputs(cfg)
        _call(B, B.rnn_forward_inference, r, cfg, i, ref)
        assert B.rnn_check_status(r.h, r._stream(None)) == 0
        B.rnn_set_debug(r.h, 0, 3, 50_000_000)  # block 0 skips step 3; 50 ms limit
        got = _outputs(cfg)
        _call(B, B.rnn_forward_inference_static, r, cfg, i, got)
        torch.cuda.synchronize()
        assert B.rnn_check_status(r.h, r._stream(None)) == 6  # RNN_ERR_TIMEOUT
        assert B.rnn_check_status(r.h, r._stream(None)) == 0  # cleared
        B.rnn_set_debug(r.h, -1, -1, 2_000_000_000)
        _call(B, B.rnn_forward_inference_static, r, cfg, i, got)
        assert B.rnn_check_status(r.h, r._stream(None)) == 0
        for k in ("y", "hy"):
            a, b = harness.from_dev(got[k]), harness.from_dev(ref[k])
            assert harness.rel_err(a, b) <= harness.tolerances(cfg)[0], k
    finally:
        r.close()
