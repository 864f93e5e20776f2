"""Shared helpers for the parity tests: device upload of generated inputs and
the error metric (max over rows of the per-row relative L2 error)."""
import numpy as np


def rel_l2_rows(got, ref):
    """max_m ||got[m] - ref[m]||_2 / ||ref[m]||_2 (float64)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.linalg.norm(got - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    return float(np.max(num / np.maximum(den, 1e-300)))


def to_device(d, bits, with_bf16=False):
    """numpy inputs from quantized_weight_gb300.inputs.make -> CUDA tensors."""
    import torch
    dev = "cuda"
    out = {
        "codes": torch.from_numpy(d["codes"]).to(dev),
        "scales": torch.from_numpy(d["scales"].view(np.float16)).to(dev),
        "biases": None if d["biases"] is None else torch.from_numpy(d["biases"].view(np.float16)).to(dev),
        "x": torch.from_numpy(d["x"]).to(dev),
    }
    if with_bf16:
        out["x_bf16"] = torch.from_numpy(d["x_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    return out
