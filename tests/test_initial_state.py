"""ssm_scan_fwd_from_state: the scan continuing from a saved state, against the oracle,
and chaining a sequence processed in two segments."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import BF16_TOL, FP32_TOL, rel_err, to_f64, to_torch

pytestmark = pytest.mark.gpu


def _case(batch, L, d_inner, d_state, bf16, seed):
    w = W.Workload("h0", "initial-state case", batch, L, d_inner, d_state, bf16, seed, 0.5)
    raw = W.host_scan_inputs(w, raw=True)
    h0 = np.random.default_rng(seed).normal(scale=0.3, size=(batch, d_inner, d_state)).astype(np.float32)
    return w, raw, h0


@pytest.mark.parametrize("lanes", ["1", "2", "4"])
@pytest.mark.parametrize("bf16,batch,L,d_inner,d_state", [
    (False, 2, 1500, 64, 16), (True, 1, 3000, 32, 16), (False, 2, 40, 24, 5), (True, 3, 1, 16, 3)])
def test_from_state_matches_oracle(lanes, bf16, batch, L, d_inner, d_state, monkeypatch):
    monkeypatch.setenv("SSM_SCAN_LANES", lanes)
    w, raw, h0 = _case(batch, L, d_inner, d_state, bf16, seed=300 + L % 97)
    t = {k: to_torch(v, bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    y, last = ssm.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                 delta_bias=t["delta_bias"], initial_state=torch.from_numpy(h0).cuda())
    torch.cuda.synchronize()
    x = {k: (W._as_f64(v, bf16) if k in ("u", "delta", "z", "B", "C") else v.astype(np.float64))
         for k, v in raw.items()}
    y_ref, last_ref = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                      delta_bias=x["delta_bias"], initial_state=h0.astype(np.float64))
    tol = BF16_TOL if bf16 else FP32_TOL
    assert rel_err(to_f64(y), y_ref) <= tol and rel_err(to_f64(last), last_ref) <= tol


@pytest.mark.parametrize("bf16", [False, True])
def test_two_segments_equal_one_call(bf16):
    w = W.WORKLOADS["mamba130m"] if not bf16 else W.Workload("seg", "segments", 2, 4096, 512, 16, True, 9, 0.5)
    raw = W.host_scan_inputs(w, raw=True)
    t = {k: to_torch(v, w.bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    y, last = ssm.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                 delta_bias=t["delta_bias"])
    L1 = 1000
    part = lambda a, b: {k: (v[:, a:b].contiguous() if k in ("u", "delta", "z", "B", "C") else v)
                         for k, v in t.items()}
    p1, p2 = part(0, L1), part(L1, w.L)
    y1, l1 = ssm.selective_scan(p1["u"], p1["delta"], p1["A"], p1["B"], p1["C"], D=p1["D"], z=p1["z"],
                                delta_bias=p1["delta_bias"])
    y2, l2 = ssm.selective_scan(p2["u"], p2["delta"], p2["A"], p2["B"], p2["C"], D=p2["D"], z=p2["z"],
                                delta_bias=p2["delta_bias"], initial_state=l1)
    torch.cuda.synchronize()
    tol = BF16_TOL if w.bf16 else FP32_TOL
    assert rel_err(to_f64(torch.cat([y1, y2], 1)), to_f64(y)) <= tol
    assert rel_err(to_f64(l2), to_f64(last)) <= tol


def test_empty_sequence_copies_initial_state():
    h0 = torch.randn(2, 16, 4, device="cuda")
    u = torch.empty((2, 0, 16), device="cuda")
    B = torch.empty((2, 0, 4), device="cuda")
    last = torch.zeros(2, 16, 4, device="cuda")
    ssm.ssm_scan_fwd_from_state(u, u, -torch.ones(16, 4, device="cuda"), B, B, None, None, None,
                                True, h0, torch.empty_like(u), last)
    torch.cuda.synchronize()
    assert torch.equal(last, h0)
