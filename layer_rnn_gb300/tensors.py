"""Device-tensor marshalling for callers of the binding: numpy arrays in the
workloads' float64 form to torch device tensors of the storage type and back.
Torch provides device memory only; nothing here computes the operator."""

import numpy as np

from layer_rnn_gb300 import workloads as wl


def to_dev(a, dtype, device="cuda"):
    """float64 numpy array -> device tensor of the storage type (f32 / bf16,
    bf16 rounded to nearest even); None stays None."""
    import torch
    if a is None:
        return None
    st = wl.to_storage(a, dtype)
    if dtype == "bf16":
        return torch.from_numpy(st.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(st).to(device)


def from_dev(t):
    """Device tensor (f32 / bf16) -> float64 numpy array; None stays None."""
    import torch
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
        return wl.bf16_to_float(bits).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def empty(shape, dtype, device="cuda"):
    """Uninitialised device tensor of the storage type."""
    import torch
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    return torch.empty(shape, dtype=td, device=device)
