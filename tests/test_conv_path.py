"""The block's conv1d + SiLU fused in front of the scan (ssm_scan_fwd_conv) and of the
decode step (ssm_state_update_conv), against the oracle's conv1d_silu + scan."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import BF16_TOL, FP32_TOL, rel_err, to_f64, to_torch

pytestmark = pytest.mark.gpu


def _case(batch, L, d_inner, d_state, bf16, d_conv, seed):
    w = W.Workload("cv", "conv case", batch, L, d_inner, d_state, bf16, seed, 0.5)
    raw = W.host_scan_inputs(w, raw=True)
    r = np.random.default_rng(seed)
    cw = r.normal(scale=0.5, size=(d_inner, d_conv)).astype(np.float32)
    cb = r.normal(scale=0.2, size=d_inner).astype(np.float32)
    return w, raw, cw, cb


def _oracle(w, raw, cw, cb, h0=None):
    x = {k: (W._as_f64(v, w.bf16) if k in ("u", "delta", "z", "B", "C") else v.astype(np.float64))
         for k, v in raw.items()}
    u = oracle.conv1d_silu(x["u"], cw, cb)
    y, last = oracle.scan_fwd(u, x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                              delta_bias=x["delta_bias"], initial_state=h0)
    return u, y, last


@pytest.mark.parametrize("bf16,batch,L,d_inner,d_state,d_conv", [
    (False, 2, 1500, 64, 16, 4), (True, 1, 3000, 32, 16, 4), (False, 2, 77, 40, 5, 3),
    (True, 3, 33, 16, 16, 2), (False, 1, 20, 8, 4, 1)])
def test_scan_conv_matches_oracle(bf16, batch, L, d_inner, d_state, d_conv):
    w, raw, cw, cb = _case(batch, L, d_inner, d_state, bf16, d_conv, seed=500 + L)
    t = {k: to_torch(v, bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    cw_t, cb_t = torch.from_numpy(cw).cuda(), torch.from_numpy(cb).cuda()
    y = torch.empty_like(t["u"])
    last = torch.empty((batch, d_inner, d_state), device="cuda")
    u_out = torch.empty_like(t["u"])
    io = ssm.SSM_BF16 if bf16 else ssm.SSM_F32
    nb = ssm.ssm_scan_fwd_workspace_size(batch, L, d_inner, d_state, io)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    ssm.ssm_scan_fwd_conv(t["u"], cw_t, cb_t, t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                          t["delta_bias"], True, None, y, last, u_out, ws)
    torch.cuda.synchronize()
    u_ref, y_ref, last_ref = _oracle(w, raw, cw, cb)
    tol = BF16_TOL if bf16 else FP32_TOL
    assert rel_err(to_f64(u_out), u_ref) <= tol
    assert rel_err(to_f64(y), y_ref) <= tol and rel_err(to_f64(last), last_ref) <= tol


def test_scan_conv_without_bias_via_selective_scan():
    w, raw, cw, _ = _case(2, 500, 24, 16, False, 4, seed=61)
    t = {k: to_torch(v, False) for k, v in raw.items()}
    y, last = ssm.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                 delta_bias=t["delta_bias"], conv_weight=torch.from_numpy(cw).cuda())
    torch.cuda.synchronize()
    _, y_ref, last_ref = _oracle(w, raw, cw, None)
    assert rel_err(to_f64(y), y_ref) <= FP32_TOL and rel_err(to_f64(last), last_ref) <= FP32_TOL


@pytest.mark.parametrize("bf16,d_conv", [(False, 4), (True, 4), (False, 2)])
def test_decode_conv_reproduces_scan_conv(bf16, d_conv):
    w, raw, cw, cb = _case(3, 30, 48, 16, bf16, d_conv, seed=71 + d_conv)
    t = {k: to_torch(v, bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    cw_t, cb_t = torch.from_numpy(cw).cuda(), torch.from_numpy(cb).cuda()
    state = torch.zeros((3, 48, 16), device="cuda")
    conv_state = torch.zeros((3, 48, d_conv - 1), device="cuda")
    ys = []
    for s in range(w.L):
        y = torch.empty((3, 48), dtype=t["u"].dtype, device="cuda")
        ssm.ssm_state_update_conv(state, conv_state, t["u"][:, s].contiguous(), cw_t, cb_t,
                                  t["delta"][:, s].contiguous(), t["A"], t["B"][:, s].contiguous(),
                                  t["C"][:, s].contiguous(), t["D"], t["z"][:, s].contiguous(), y,
                                  t["delta_bias"], True)
        ys.append(y)
    torch.cuda.synchronize()
    _, y_ref, last_ref = _oracle(w, raw, cw, cb)
    tol = BF16_TOL if bf16 else FP32_TOL
    assert rel_err(to_f64(torch.stack(ys, 1)), y_ref) <= tol
    assert rel_err(to_f64(state), last_ref) <= tol
    if d_conv > 1:  # the window holds the last d_conv - 1 inputs, oldest first
        xin = to_f64(t["u"])
        np.testing.assert_array_equal(to_f64(conv_state), np.transpose(xin[:, -(d_conv - 1):, :], (0, 2, 1)))
