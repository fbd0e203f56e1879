"""The five synthetic workloads (shapes, dtypes, seeds, value distributions).

Recipe shared by every workload (all seeded, all synthetic):
  u, z, B, C, D ~ N(0, 1); delta_raw ~ N(0, delta_sd) (sd, not variance);
  delta_bias = inverse softplus of dt, dt log-uniform on [1e-3, 1e-1];
  A[d, n] = -(n + 1); decode initial state ~ N(0, 0.1).
Each value is drawn in double, rounded to fp32, and for bf16 tensors rounded
once more to bf16 (round to nearest even).  A, D and delta_bias are fp32.

Flat element index of a [batch][L][d_inner] tensor is (b*L + t)*d_inner + d;
of a [batch][L][d_state] tensor (b*L + t)*d_state + n; decode tensors carry a
leading step axis: [steps][batch][...].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import bf16_to_f32, delta_bias, dev_fill_normal, normal, normal_at

# Stream ids, one per tensor of a workload.
TID_U, TID_DELTA, TID_Z, TID_B, TID_C, TID_D, TID_BIAS, TID_STATE0 = 1, 2, 3, 4, 5, 6, 7, 8
DT_MIN, DT_MAX = 1e-3, 1e-1


@dataclass(frozen=True)
class Workload:
    key: str
    desc: str
    batch: int
    L: int            # sequence length (scan) or number of decode steps
    d_inner: int
    d_state: int
    bf16: bool        # I/O dtype of u, delta, z, B, C, y
    seed: int
    delta_sd: float
    decode: bool = False
    state_sd: float = 0.0
    heads: int = 0    # > 0: chunked-SSD workload (one A and one step size per head of 64 channels)

    @property
    def elements(self) -> int:
        return self.batch * self.L * self.d_inner


WORKLOADS = {
    "tiny": Workload("tiny", "tiny fp32 scan", 1, 64, 16, 4, False, 0, 1.0),
    "mamba130m": Workload("mamba130m", "Mamba-130M-layer-shaped scan, fp32",
                          2, 2048, 1536, 16, False, 1, 0.5),
    "mamba2p8b": Workload("mamba2p8b", "Mamba-2.8B-layer-shaped scan, bf16 I/O",
                          8, 2048, 5120, 16, True, 2, 0.5),
    "long": Workload("long", "long-context scan, 1,048,576 tokens, bf16 I/O",
                     1, 1 << 20, 2048, 16, True, 3, 0.5),
    # the long-context scan's first 65,536 tokens (same seed and layout, so the same values):
    # the size its profiler captures run on
    "long64k": Workload("long64k", "long-context scan, first 65,536 of 1,048,576 tokens, bf16 I/O",
                        1, 1 << 16, 2048, 16, True, 3, 0.5),
    "decode": Workload("decode", "selective_state_update, 1024 sequential steps, bf16 I/O",
                       256, 1024, 5120, 16, True, 4, 0.5, decode=True, state_sd=0.1),
    "ssd2p7b": Workload("ssd2p7b", "Mamba-2-2.7B-layer-shaped chunked SSD scan (80 heads of 64, "
                        "d_state 128), bf16 I/O", 8, 2048, 5120, 128, True, 5, 0.5, heads=80),
}


def ssd_A_head(w: Workload) -> np.ndarray:
    """One decay rate per head: A_h = -(1 + h mod 16)."""
    return -(1.0 + (np.arange(w.heads) % 16)).astype(np.float32)


def ssd_dt_bias(w: Workload) -> np.ndarray:
    return delta_bias(w.seed, TID_BIAS, DT_MIN, DT_MAX, w.heads)


def host_ssd_inputs(w: Workload, b_sel=None, d_sel=None):
    """SSD workload inputs for batches b_sel and channels d_sel (whole heads or not), as the
    equivalent per-channel scan operands in float64 for the oracle: delta and delta_bias
    broadcast from the head, A[d, n] = A_head[h]."""
    assert w.heads > 0
    b_sel = np.arange(w.batch) if b_sel is None else np.asarray(b_sel, dtype=np.int64)
    d_sel = np.arange(w.d_inner) if d_sel is None else np.asarray(d_sel, dtype=np.int64)
    P = w.d_inner // w.heads
    h_sel = d_sel // P
    t = np.arange(w.L, dtype=np.int64)
    out = {}
    for name, tid in (("u", TID_U), ("z", TID_Z)):
        idx = ((b_sel[:, None, None] * w.L + t[None, :, None]) * w.d_inner + d_sel[None, None, :]).ravel()
        out[name] = _as_f64(normal_at(w.seed, tid, 0.0, 1.0, idx, True), True).reshape(len(b_sel), w.L, len(d_sel))
    idx = ((b_sel[:, None, None] * w.L + t[None, :, None]) * w.heads + h_sel[None, None, :]).ravel()
    out["delta"] = _as_f64(normal_at(w.seed, TID_DELTA, 0.0, w.delta_sd, idx, True), True).reshape(
        len(b_sel), w.L, len(d_sel))
    for name, tid in (("B", TID_B), ("C", TID_C)):
        parts = [normal(w.seed, tid, 0.0, 1.0, int(b) * w.L * w.d_state, w.L * w.d_state, True) for b in b_sel]
        out[name] = _as_f64(np.concatenate(parts), True).reshape(len(b_sel), w.L, w.d_state)
    out["A"] = np.repeat(ssd_A_head(w)[h_sel][:, None], w.d_state, axis=1).astype(np.float64)
    out["D"] = D_vector(w)[d_sel].astype(np.float64)
    out["delta_bias"] = ssd_dt_bias(w)[h_sel].astype(np.float64)
    return out


def device_ssd_inputs(w: Workload, device="cuda"):
    """Full-size SSD inputs on the GPU: x, z [batch, L, d_inner], dt [batch, L, heads],
    B, C [batch, L, d_state] (bf16), A_head, dt_bias [heads], D [d_inner] (fp32)."""
    import torch
    assert w.heads > 0
    stream = torch.cuda.current_stream(device).cuda_stream
    out = {}
    for name, tid, shape, sd in (("x", TID_U, (w.batch, w.L, w.d_inner), 1.0),
                                 ("z", TID_Z, (w.batch, w.L, w.d_inner), 1.0),
                                 ("dt", TID_DELTA, (w.batch, w.L, w.heads), w.delta_sd),
                                 ("B", TID_B, (w.batch, w.L, w.d_state), 1.0),
                                 ("C", TID_C, (w.batch, w.L, w.d_state), 1.0)):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        dev_fill_normal(w.seed, tid, 0.0, sd, 0, t.numel(), True, t.data_ptr(), stream)
        out[name] = t
    out["A_head"] = torch.from_numpy(ssd_A_head(w)).to(device)
    out["dt_bias"] = torch.from_numpy(ssd_dt_bias(w)).to(device)
    out["D"] = torch.from_numpy(D_vector(w)).to(device)
    return out


def A_matrix(w: Workload) -> np.ndarray:
    return np.tile(-np.arange(1, w.d_state + 1, dtype=np.float32), (w.d_inner, 1))


def D_vector(w: Workload) -> np.ndarray:
    return normal(w.seed, TID_D, 0.0, 1.0, 0, w.d_inner, False)


def bias_vector(w: Workload) -> np.ndarray:
    return delta_bias(w.seed, TID_BIAS, DT_MIN, DT_MAX, w.d_inner)


def _as_f64(a: np.ndarray, bf16: bool) -> np.ndarray:
    return (bf16_to_f32(a) if bf16 else a).astype(np.float64)


def _act_params(w: Workload, tid: int):
    return (0.0, w.delta_sd) if tid == TID_DELTA else (0.0, 1.0)


def host_scan_inputs(w: Workload, b_sel=None, d_sel=None, t_count=None, raw: bool = False):
    """Inputs of a scan workload restricted to batches b_sel, channels d_sel and
    the first t_count steps, as float64 arrays for the oracle (values are the
    exact rounded numbers the device holds).  With raw=True the typed arrays
    (float32, or uint16 bf16 bits) are returned instead, for upload."""
    b_sel = np.arange(w.batch) if b_sel is None else np.asarray(b_sel, dtype=np.int64)
    d_sel = np.arange(w.d_inner) if d_sel is None else np.asarray(d_sel, dtype=np.int64)
    T = w.L if t_count is None else int(t_count)
    nb, nd = len(b_sel), len(d_sel)
    t = np.arange(T, dtype=np.int64)
    out = {}
    full_d = nd == w.d_inner and np.array_equal(d_sel, np.arange(w.d_inner))
    for name, tid in (("u", TID_U), ("delta", TID_DELTA), ("z", TID_Z)):
        mean, sd = _act_params(w, tid)
        parts = []
        for b in b_sel:
            if full_d:
                parts.append(normal(w.seed, tid, mean, sd, int(b) * w.L * w.d_inner,
                                    T * w.d_inner, w.bf16))
            else:
                idx = ((int(b) * w.L + t)[:, None] * w.d_inner + d_sel[None, :]).ravel()
                parts.append(normal_at(w.seed, tid, mean, sd, idx, w.bf16))
        a = np.concatenate(parts).reshape(nb, T, nd)
        out[name] = a if raw else _as_f64(a, w.bf16)
    for name, tid in (("B", TID_B), ("C", TID_C)):
        parts = [normal(w.seed, tid, 0.0, 1.0, int(b) * w.L * w.d_state, T * w.d_state, w.bf16)
                 for b in b_sel]
        a = np.concatenate(parts).reshape(nb, T, w.d_state)
        out[name] = a if raw else _as_f64(a, w.bf16)
    A, D, bias = A_matrix(w)[d_sel], D_vector(w)[d_sel], bias_vector(w)[d_sel]
    out["A"], out["D"], out["delta_bias"] = (A, D, bias) if raw else (
        A.astype(np.float64), D.astype(np.float64), bias.astype(np.float64))
    return out


def host_decode_inputs(w: Workload, steps: int, b_sel=None, d_sel=None, raw: bool = False):
    """Decode workload inputs for the first `steps` steps, restricted to b_sel/d_sel:
    per-step u, delta, z [steps, nb, nd]; B, C [steps, nb, d_state]; the initial
    state [nb, nd, d_state] (fp32); A, D, delta_bias for d_sel."""
    assert w.decode
    b_sel = np.arange(w.batch) if b_sel is None else np.asarray(b_sel, dtype=np.int64)
    d_sel = np.arange(w.d_inner) if d_sel is None else np.asarray(d_sel, dtype=np.int64)
    nb, nd = len(b_sel), len(d_sel)
    s = np.arange(steps, dtype=np.int64)
    out = {}
    for name, tid in (("u", TID_U), ("delta", TID_DELTA), ("z", TID_Z)):
        mean, sd = _act_params(w, tid)
        idx = ((s[:, None, None] * w.batch + b_sel[None, :, None]) * w.d_inner
               + d_sel[None, None, :]).ravel()
        a = normal_at(w.seed, tid, mean, sd, idx, w.bf16).reshape(steps, nb, nd)
        out[name] = a if raw else _as_f64(a, w.bf16)
    n = np.arange(w.d_state, dtype=np.int64)
    for name, tid in (("B", TID_B), ("C", TID_C)):
        idx = ((s[:, None, None] * w.batch + b_sel[None, :, None]) * w.d_state
               + n[None, None, :]).ravel()
        a = normal_at(w.seed, tid, 0.0, 1.0, idx, w.bf16).reshape(steps, nb, w.d_state)
        out[name] = a if raw else _as_f64(a, w.bf16)
    idx = ((b_sel[:, None, None] * w.d_inner + d_sel[None, :, None]) * w.d_state
           + n[None, None, :]).ravel()
    st = normal_at(w.seed, TID_STATE0, 0.0, w.state_sd, idx, False).reshape(nb, nd, w.d_state)
    out["state0"] = st if raw else st.astype(np.float64)
    A, D, bias = A_matrix(w)[d_sel], D_vector(w)[d_sel], bias_vector(w)[d_sel]
    out["A"], out["D"], out["delta_bias"] = (A, D, bias) if raw else (
        A.astype(np.float64), D.astype(np.float64), bias.astype(np.float64))
    return out


def device_inputs(w: Workload, device="cuda", steps: int | None = None):
    """Full-size inputs filled directly on the GPU (bit-identical to the host draws).

    Scan: u, delta, z [batch, L, d_inner]; B, C [batch, L, d_state].
    Decode: u, delta, z [steps, batch, d_inner]; B, C [steps, batch, d_state];
    state0 [batch, d_inner, d_state] fp32.  A, D, delta_bias are fp32 copies."""
    import torch

    dt = torch.bfloat16 if w.bf16 else torch.float32
    stream = torch.cuda.current_stream(device).cuda_stream
    out = {}
    if w.decode:
        S = w.L if steps is None else steps
        act_shape, bc_shape = (S, w.batch, w.d_inner), (S, w.batch, w.d_state)
    else:
        act_shape, bc_shape = (w.batch, w.L, w.d_inner), (w.batch, w.L, w.d_state)
    for name, tid, shape in (("u", TID_U, act_shape), ("delta", TID_DELTA, act_shape),
                             ("z", TID_Z, act_shape), ("B", TID_B, bc_shape), ("C", TID_C, bc_shape)):
        mean, sd = _act_params(w, tid)
        t = torch.empty(shape, dtype=dt, device=device)
        dev_fill_normal(w.seed, tid, mean, sd, 0, t.numel(), w.bf16, t.data_ptr(), stream)
        out[name] = t
    if w.decode:
        st = torch.empty((w.batch, w.d_inner, w.d_state), dtype=torch.float32, device=device)
        dev_fill_normal(w.seed, TID_STATE0, 0.0, w.state_sd, 0, st.numel(), False, st.data_ptr(),
                        stream)
        out["state0"] = st
    out["A"] = torch.from_numpy(A_matrix(w)).to(device)
    out["D"] = torch.from_numpy(D_vector(w)).to(device)
    out["delta_bias"] = torch.from_numpy(bias_vector(w)).to(device)
    return out
