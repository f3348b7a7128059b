"""Helpers shared by the GPU parity tests (conversions and error measures)."""
import numpy as np
import torch

from serving_kda_chunked_gated_gb300 import inputs as I

TOL_O = 2e-3      # relative L2 on o (and y), bf16 outputs
TOL_S = 1e-3      # relative L2 on final states


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def to_dev(x, dev, bf16=False):
    if x is None:
        return None
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def qkv_to_dev(d, dev):
    bf = d["dtype"] == "bf16"
    return (to_dev(d["q"], dev, bf), to_dev(d["k"], dev, bf), to_dev(d["v"], dev, bf))


def f64(d, key):
    x = d[key]
    if x is None:
        return None
    if x.dtype == np.uint16:
        return I.bf16_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def host(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
