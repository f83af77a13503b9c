"""Writes the oracle regression fixture ``tiny_lstm_oracle.json``.

Calls only the float64 oracle (and the seeded workload generator for the
inputs).  Re-run it only when the oracle's arithmetic changes for a reason
that a page, or a stated reading of one, justifies.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from layer_rnn_gb300 import workloads as wl  # noqa: E402


def main():
    cfg = wl.WORKLOADS["tiny_lstm"]
    inp = wl.make_inputs(cfg)
    out = oracle.run_flat(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"],
                          inp["x"], inp["h0"], inp["c0"], inp["w"], inp["dy"],
                          inp["dhy"], inp["dcy"])
    doc = dict(source="float64 oracle on the seeded tiny_lstm workload "
                      "(T=5, N=2, I=4, H=8, 1 layer, unidirectional); written by make_golden.py",
               workload=cfg,
               outputs={k: [float(v) for v in out[k].ravel()] for k in
                        ("y", "hy", "cy", "dx", "dh0", "dc0", "dW")})
    with open(os.path.join(HERE, "tiny_lstm_oracle.json"), "w") as f:
        json.dump(doc, f, indent=0)


if __name__ == "__main__":
    main()
