"""Seeded synthetic workloads for the fused RNN operator.

This module only draws random numbers and converts storage formats; it holds
none of the operator's arithmetic.  Both the CUDA-path tests and the oracle
tests take their inputs from here, so the two sides see identical values.

The shapes are the Deep Speech 2 layer sizes that the MXNet "Fused RNN operator
for CPU" design page benchmarks (section Performance: seq_length 300,
batch 20, input 800, hidden 800, single direction; 5-layer bidirectional
vRNN / LSTM / GRU), plus a tiny LSTM and a large bf16 4-layer stack.  No
dataset is involved: the pages use DS2 only as a source of layer sizes.

Recipe (per workload, one ``numpy.random.Generator(PCG64(seed))``, draws in this
order): x ~ N(0,1) [T,N,I]; h0 ~ N(0, s^2) [L*D,N,H]; c0 likewise (s = 0 means
zeros, drawn anyway so later draws do not depend on it); the flat canonical
weight buffer ~ U(-b, b) with b = 1/sqrt(H) (weights and biases alike);
dy ~ N(0,1) [T,N,D*H]; dhy ~ N(0,1) and dcy ~ N(0,1) [L*D,N,H].  Every array is
then rounded to the workload's storage type (fp32, or bf16 with round to
nearest even) and returned as float64 holding exactly the stored values.
"""

import math

import numpy as np

GATES = {"rnn_tanh": 1, "lstm": 4, "gru": 3, "gru_tf": 3}
MODE_IDS = {"rnn_tanh": 0, "lstm": 1, "gru": 2, "gru_tf": 3}
DTYPE_IDS = {"f32": 0, "bf16": 1}


def _cfg(name, mode, L, bidir, T, N, I, H, dtype, h0_std, seed):
    return dict(name=name, mode=mode, L=L, bidir=bidir, T=T, N=N, I=I, H=H,
                dtype=dtype, h0_std=h0_std, seed=seed)


WORKLOADS = {
    # tiny LSTM: 1 layer, unidirectional, fp32
    "tiny_lstm": _cfg("tiny_lstm", "lstm", 1, False, 5, 2, 4, 8, "f32", 0.1, 101),
    # Deep Speech 2 shaped single layers, fp32, h0 = c0 = 0
    "ds2_lstm": _cfg("ds2_lstm", "lstm", 1, False, 300, 20, 800, 800, "f32", 0.0, 202),
    "ds2_gru": _cfg("ds2_gru", "gru", 1, False, 300, 20, 800, 800, "f32", 0.0, 303),
    # 5-layer bidirectional stacks, fp32
    "bi5_rnn_tanh": _cfg("bi5_rnn_tanh", "rnn_tanh", 5, True, 300, 20, 800, 800, "f32", 0.1, 404),
    "bi5_lstm": _cfg("bi5_lstm", "lstm", 5, True, 300, 20, 800, 800, "f32", 0.1, 405),
    "bi5_gru": _cfg("bi5_gru", "gru", 5, True, 300, 20, 800, 800, "f32", 0.1, 406),
    # large 4-layer LSTM, bf16 storage, fp32 cell state / accumulation
    "lstm4_bf16": _cfg("lstm4_bf16", "lstm", 4, False, 512, 128, 1024, 1024, "bf16", 0.0, 505),
}


def make_config(mode, L, bidir, T, N, I, H, dtype="f32", h0_std=0.1, seed=0,
                name="custom"):
    """A workload dict of the same form as ``WORKLOADS`` entries."""
    return _cfg(name, mode, L, bidir, T, N, I, H, dtype, h0_std, seed)


def with_sizes(cfg, **over):
    """Copy of a workload with some sizes replaced (e.g. a shorter T)."""
    c = dict(cfg)
    c.update(over)
    c["name"] = cfg["name"] + "".join("_%s%s" % (k, v) for k, v in sorted(over.items()))
    return c


def num_directions(cfg):
    return 2 if cfg["bidir"] else 1


def weight_count(cfg):
    """Elements of the canonical flat weight buffer (sizes only)."""
    G, H, D = GATES[cfg["mode"]], cfg["H"], num_directions(cfg)
    total = 0
    for l in range(cfg["L"]):
        I_l = cfg["I"] if l == 0 else D * H
        total += D * (G * H * I_l + G * H * H + 2 * G * H)
    return total


# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------

def bf16_bits(a):
    """float -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)
    u = u.astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_float(bits):
    """bf16 bit patterns (uint16) -> float32."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def round_to(a, dtype):
    """Round to the storage type; returned as float64 holding exact values."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_to_float(bf16_bits(a)).astype(np.float64)
    raise ValueError(dtype)


def to_storage(a, dtype):
    """float64 values (already representable) -> numpy array in storage form
    (float32, or uint16 bf16 bit patterns)."""
    if dtype == "f32":
        return np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return np.ascontiguousarray(bf16_bits(a))


# ----------------------------------------------------------------------------
# generator
# ----------------------------------------------------------------------------

def make_inputs(cfg, seed=None):
    """Draw one workload's inputs.  Returns float64 arrays rounded to storage."""
    rng = np.random.Generator(np.random.PCG64(cfg["seed"] if seed is None else seed))
    T, N, I, H, L = cfg["T"], cfg["N"], cfg["I"], cfg["H"], cfg["L"]
    D = num_directions(cfg)
    dt = cfg["dtype"]
    s = cfg["h0_std"]
    bound = 1.0 / math.sqrt(H)
    x = rng.standard_normal((T, N, I))
    h0 = rng.standard_normal((L * D, N, H)) * s
    c0 = rng.standard_normal((L * D, N, H)) * s
    w = rng.uniform(-bound, bound, size=weight_count(cfg))
    dy = rng.standard_normal((T, N, D * H))
    dhy = rng.standard_normal((L * D, N, H))
    dcy = rng.standard_normal((L * D, N, H))
    out = dict(x=x, h0=h0, c0=c0, w=w, dy=dy, dhy=dhy, dcy=dcy)
    out = {k: round_to(v, dt) for k, v in out.items()}
    if cfg["mode"] != "lstm":
        out["c0"] = None
        out["dcy"] = None
    return out


def make_lengths(cfg, seed=None):
    """Per-sequence valid lengths for a padded batch of the workload: one
    sequence of the full T (the padding length is the longest sequence's),
    the others uniform integers in [ceil(T/2), T] -- a mix of utterance
    lengths within a factor of two, as a length-bucketed batch holds."""
    rng = np.random.Generator(np.random.PCG64((cfg["seed"] if seed is None else seed) + 7919))
    T, N = cfg["T"], cfg["N"]
    lens = rng.integers((T + 1) // 2, T + 1, size=N)
    lens[0] = T
    return lens.astype(np.int32)


def make_dropout_masks(cfg, p, seed=None):
    """0/1 inter-layer dropout masks, [L-1, T, N, D*H] uint8, each element 1
    with probability 1 - p (Bernoulli draws from the seeded generator)."""
    rng = np.random.Generator(np.random.PCG64((cfg["seed"] if seed is None else seed) + 104729))
    L, T, N, H = cfg["L"], cfg["T"], cfg["N"], cfg["H"]
    D = num_directions(cfg)
    return (rng.random((max(0, L - 1), T, N, D * H)) >= p).astype(np.uint8)
