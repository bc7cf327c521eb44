"""Helpers for the GPU parity tests (device transfer, error metric)."""
import numpy as np
import pytest


def require_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_recurrences_gb300 as ss
    from linear_recurrences_gb300 import build
    build.build()
    ss.lib()
    return torch


def rel_err(y, ref) -> float:
    """max_i |y_i - ref_i| / max(1, |ref_i|), the parity metric."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    if y.size == 0:
        return 0.0
    return float(np.max(np.abs(y - ref) / np.maximum(1.0, np.abs(ref))))


def to_dev(arr, dev, io="f32"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr))
    if io == "bf16" and arr.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


def to_host_f64(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)
