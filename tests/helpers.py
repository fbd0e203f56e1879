"""Shared test helpers: the error metric, the record of achieved parity margins, and moving
generator output to torch."""
import json
import os

import numpy as np

FP32_TOL = 1e-4   # max relative error, fp32 I/O (fp32 state)
BF16_TOL = 2e-2   # max relative error, bf16 I/O (fp32 state)


def rel_err(got, ref) -> float:
    """max_i |got_i - ref_i| / max(|ref_i|, rms(ref)): relative error with the
    denominator floored at the RMS of the reference, so that elements near zero
    are judged on the tensor's own scale."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    den = np.maximum(np.abs(r), rms)
    den = np.where(den == 0.0, 1.0, den)
    return float(np.max(np.abs(g - r) / den))


def to_torch(a, bf16: bool, device="cuda"):
    """Typed generator output (float32, or uint16 bf16 bits) -> torch tensor on device."""
    import torch
    a = np.ascontiguousarray(a)
    if bf16 and a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a.astype(np.float32)).to(device)


def to_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


# Achieved errors of the parity checks of this session (name -> {quantity: error, "tol": bar}).
# The terminal summary prints them; with SSM_PARITY_LOG=<path> they are also written as JSON.
MARGINS = {}


def record_margin(name: str, tol: float, **errors) -> None:
    MARGINS[name] = {**{k: float(v) for k, v in errors.items()}, "tol": float(tol)}


def dump_margins():
    path = os.environ.get("SSM_PARITY_LOG")
    if path and MARGINS:
        with open(path, "w") as f:
            json.dump(MARGINS, f, indent=1, sort_keys=True)
