"""The block's conv1d + SiLU fused in front of the scan (ssm_scan_fwd_conv) and of the
decode step (ssm_state_update_conv), against the oracle's conv1d_silu + scan."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import record_margin, BF16_TOL, FP32_TOL, rel_err, to_f64, to_torch

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


@pytest.mark.parametrize("key", ["mamba130m", "mamba2p8b"])
def test_scan_conv_full_size_sampled(key):
    """ssm_scan_fwd_conv at the bench's full sizes (the u tensor is the block input x; 4-tap
    weights); the conv is per channel, so the oracle checks u and y on sampled channels over
    every batch row and step, and their final states."""
    w = W.WORKLOADS[key]
    dev = W.device_inputs(w)
    r = np.random.default_rng(w.seed)
    cw = r.normal(scale=0.5, size=(w.d_inner, 4)).astype(np.float32)
    cb = r.normal(scale=0.2, size=w.d_inner).astype(np.float32)
    y = torch.empty_like(dev["u"])
    u_out = torch.empty_like(dev["u"])
    last = torch.empty((w.batch, w.d_inner, w.d_state), device="cuda")
    io = ssm.SSM_BF16 if w.bf16 else ssm.SSM_F32
    nb = ssm.ssm_scan_fwd_workspace_size(w.batch, w.L, w.d_inner, w.d_state, io)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    ssm.ssm_scan_fwd_conv(dev["u"], torch.from_numpy(cw).cuda(), torch.from_numpy(cb).cuda(), dev["delta"],
                          dev["A"], dev["B"], dev["C"], dev["D"], dev["z"], dev["delta_bias"], True, None,
                          y, last, u_out, ws)
    torch.cuda.synchronize()
    d_sel = np.unique(np.concatenate([[0, 1, 31, 32, w.d_inner - 1],
                                      np.random.default_rng(w.seed + 1).choice(w.d_inner, 7, replace=False)]))
    ds = torch.from_numpy(d_sel).cuda()
    got_u, got_y = to_f64(u_out.index_select(2, ds)), to_f64(y.index_select(2, ds))
    got_last = to_f64(last.index_select(1, ds))
    del dev, y, u_out
    x = W.host_scan_inputs(w, d_sel=d_sel)
    u_ref = oracle.conv1d_silu(x["u"], cw[d_sel], cb[d_sel])
    y_ref, last_ref = oracle.scan_fwd(u_ref, x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                      delta_bias=x["delta_bias"])
    tol = BF16_TOL if w.bf16 else FP32_TOL
    eu, ey, el = rel_err(got_u, u_ref), rel_err(got_y, y_ref), rel_err(got_last, last_ref)
    record_margin(f"conv+scan {key} (full size, sampled)", tol, u=eu, y=ey, last_state=el)
    assert eu <= tol and ey <= tol and el <= tol, f"u err {eu:.3g}, y err {ey:.3g}, last err {el:.3g}"


@pytest.mark.parametrize("lanes", ["1", "2", "4"])
@pytest.mark.parametrize("bf16,batch,L,d_inner,d_state,d_conv", [
    (False, 2, 3000, 96, 16, 4), (True, 1, 4100, 64, 16, 3), (False, 3, 700, 40, 5, 4)])
def test_scan_conv_both_kernels_from_state(lanes, bf16, batch, L, d_inner, d_state, d_conv, monkeypatch):
    """The conv path in every kernel variant (one, two or four lanes per channel pair), over many ragged time
    chunks (each chunk after the first starts its window from the inputs before it), from a
    given initial state."""
    monkeypatch.setenv("SSM_SCAN_LANES", lanes)
    w, raw, cw, cb = _case(batch, L, d_inner, d_state, bf16, d_conv, seed=800 + L + int(lanes))
    h0 = np.random.default_rng(L).normal(scale=0.3, size=(batch, d_inner, d_state)).astype(np.float32)
    t = {k: to_torch(v, bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    y = torch.empty_like(t["u"])
    u_out = torch.empty_like(t["u"])
    last = torch.empty((batch, d_inner, d_state), device="cuda")
    io = ssm.SSM_BF16 if bf16 else ssm.SSM_F32
    nb = ssm.ssm_scan_fwd_workspace_size(batch, L, d_inner, d_state, io)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    ssm.ssm_scan_fwd_conv(t["u"], torch.from_numpy(cw).cuda(), torch.from_numpy(cb).cuda(), t["delta"], t["A"],
                          t["B"], t["C"], t["D"], t["z"], t["delta_bias"], True, torch.from_numpy(h0).cuda(),
                          y, last, u_out, ws)
    torch.cuda.synchronize()
    u_ref, y_ref, last_ref = _oracle(w, raw, cw, cb, h0=h0.astype(np.float64))
    tol = BF16_TOL if bf16 else FP32_TOL
    eu, ey, el = rel_err(to_f64(u_out), u_ref), rel_err(to_f64(y), y_ref), rel_err(to_f64(last), last_ref)
    assert eu <= tol and ey <= tol and el <= tol, f"u err {eu:.3g}, y err {ey:.3g}, last err {el:.3g}"
