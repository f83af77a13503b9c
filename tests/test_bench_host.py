"""Host logic of bench.py that needs no GPU: the DRAM-traffic figure of the
roofline line is taken from profiles/traffic.json only while the kernel's
source and every header it includes (transitively) are unchanged since the
capture."""

import json
import os

import numpy as np
import pytest


def _tree(tmp_path):
    csrc = tmp_path / "layer_rnn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text('#include "common.cuh"\n#include "rec.h"\nkernel v1\n')
    (csrc / "common.cuh").write_text("header v1\n")
    (csrc / "rec.h").write_text('#include "host_common.h"\ndecls v1\n')
    (csrc / "host_common.h").write_text("shared decls v1\n")
    (csrc / "wf.h").write_text("another part's decls v1\n")
    (tmp_path / "profiles").mkdir()
    return csrc


def _write_traffic(tmp_path, sha, nbytes=123456):
    doc = {"ds2_lstm": {"rec_fwd": {"kernel": "k", "source": "layer_rnn_gb300/csrc/k.cu",
                                    "sources_sha256": sha, "dram_bytes_per_launch": nbytes}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(doc))


@pytest.fixture
def bench_at(tmp_path, monkeypatch):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return bench


def test_traffic_reported_while_sources_match(tmp_path, bench_at):
    _tree(tmp_path)
    _write_traffic(tmp_path, bench_at.kernel_source_sha256("layer_rnn_gb300/csrc/k.cu"))
    assert bench_at.traffic_for("rec_fwd", {"name": "ds2_lstm"}) == 123456
    # no entry for this phase or workload
    assert bench_at.traffic_for("rec_bwd", {"name": "ds2_lstm"}) is None
    assert bench_at.traffic_for("rec_fwd", {"name": "lstm4_bf16"}) is None


@pytest.mark.parametrize("changed", ["k.cu", "common.cuh", "rec.h", "host_common.h"])
def test_traffic_dropped_when_kernel_or_included_header_changes(tmp_path, bench_at, changed):
    csrc = _tree(tmp_path)
    _write_traffic(tmp_path, bench_at.kernel_source_sha256("layer_rnn_gb300/csrc/k.cu"))
    with open(os.path.join(csrc, changed), "a") as f:
        f.write("edit\n")
    assert bench_at.traffic_for("rec_fwd", {"name": "ds2_lstm"}) is None


@pytest.mark.parametrize("changed", ["wf.h", "other.cu", "new.cuh"])
def test_sources_not_included_do_not_affect_the_hash(tmp_path, bench_at, changed):
    csrc = _tree(tmp_path)
    before = bench_at.kernel_source_sha256("layer_rnn_gb300/csrc/k.cu")
    with open(os.path.join(csrc, changed), "a") as f:
        f.write("edit\n")
    assert bench_at.kernel_source_sha256("layer_rnn_gb300/csrc/k.cu") == before


def test_include_closure_is_transitive(tmp_path, bench_at):
    _tree(tmp_path)
    names = [os.path.basename(p)
             for p in bench_at.include_closure("layer_rnn_gb300/csrc/k.cu")]
    assert names == ["k.cu", "common.cuh", "host_common.h", "rec.h"]


def test_entries_without_a_source_hash_are_ignored(tmp_path, bench_at):
    _tree(tmp_path)
    doc = {"ds2_lstm": {"rec_fwd": {"kernel": "k", "source": "layer_rnn_gb300/csrc/k.cu",
                                    "dram_bytes_per_launch": 1}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(doc))
    assert bench_at.traffic_for("rec_fwd", {"name": "ds2_lstm"}) is None


def test_committed_traffic_entries_name_existing_profiles():
    import bench
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        doc = json.load(f)
    for wl, phases in doc.items():
        if wl.startswith("_"):
            continue
        for ph, ent in phases.items():
            assert os.path.exists(os.path.join(bench.ROOT, ent["source"])), (wl, ph)
            assert os.path.exists(os.path.join(bench.ROOT, ent["profile"])), (wl, ph)
            assert ent["dram_bytes_per_launch"] > 0


def test_bench_lengths_follow_the_stated_recipe():
    # one sequence of the full T, the others in [ceil(T/2), T], seeded
    from layer_rnn_gb300 import workloads as wl
    for name in ("ds2_lstm", "lstm4_bf16", "tiny_lstm"):
        cfg = wl.WORKLOADS[name]
        T, N = cfg["T"], cfg["N"]
        a = wl.make_lengths(cfg)
        assert a.dtype == np.int32 and a.shape == (N,)
        assert a[0] == T and a.max() == T and a.min() >= (T + 1) // 2
        assert np.array_equal(a, wl.make_lengths(cfg))
        assert not np.array_equal(a, wl.make_lengths(cfg, seed=cfg["seed"] + 1)) or N < 3


def test_bench_dropout_masks_follow_the_stated_recipe():
    # 0/1 bytes over [L-1, T, N, D*H], ones with probability 1 - p, seeded
    from layer_rnn_gb300 import workloads as wl
    cfg = wl.WORKLOADS["bi5_gru"]
    m = wl.make_dropout_masks(cfg, 0.3)
    assert m.dtype == np.uint8 and m.shape == (cfg["L"] - 1, cfg["T"], cfg["N"], 2 * cfg["H"])
    assert set(np.unique(m)) <= {0, 1}
    assert abs(m.mean() - 0.7) < 0.01
    assert np.array_equal(m, wl.make_dropout_masks(cfg, 0.3))
    assert wl.make_dropout_masks(wl.WORKLOADS["ds2_lstm"], 0.3).shape[0] == 0
