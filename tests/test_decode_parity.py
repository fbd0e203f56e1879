"""GPU parity of ssm_state_update against the oracle, and decode == scan."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import record_margin, BF16_TOL, FP32_TOL, rel_err, to_f64, to_torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("d_state", [1, 4, 6, 8, 12, 16])
def test_decode_steps_small(d_state, bf16):
    w = W.Workload("dec", "decode edge case", 5, 6, 24, d_state, bf16, 21 + d_state, 0.5,
                   decode=True, state_sd=0.1)
    raw = W.host_decode_inputs(w, w.L, raw=True)
    x = W.host_decode_inputs(w, w.L)
    io = lambda k, s: to_torch(raw[k][s], bf16)
    state = torch.from_numpy(raw["state0"]).cuda()
    A, D, bias = (torch.from_numpy(raw[k]).cuda() for k in ("A", "D", "delta_bias"))
    st_ref = x["state0"]
    tol = BF16_TOL if bf16 else FP32_TOL
    for s in range(w.L):
        y = ssm.selective_state_update(state, io("u", s), io("delta", s), A, io("B", s), io("C", s),
                                       D=D, z=io("z", s), delta_bias=bias)
        y_ref, st_ref = oracle.state_update(st_ref, x["u"][s], x["delta"][s], x["A"], x["B"][s],
                                            x["C"][s], D=x["D"], z=x["z"][s],
                                            delta_bias=x["delta_bias"])
        torch.cuda.synchronize()
        assert rel_err(to_f64(y), y_ref) <= tol
        assert rel_err(to_f64(state), st_ref) <= tol


@pytest.mark.parametrize("bf16", [False, True])
def test_decode_reproduces_scan(bf16):
    w = W.Workload("cmp", "decode vs scan", 2, 40, 64, 16, bf16, 5, 0.5)
    raw = W.host_scan_inputs(w, raw=True)
    t = {k: to_torch(v, bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    y_scan, last_scan = ssm.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                                           z=t["z"], delta_bias=t["delta_bias"])
    state = torch.zeros((2, 64, 16), device="cuda")
    ys = []
    for s in range(w.L):
        ys.append(ssm.selective_state_update(state, t["u"][:, s].contiguous(),
                                             t["delta"][:, s].contiguous(), t["A"],
                                             t["B"][:, s].contiguous(), t["C"][:, s].contiguous(),
                                             D=t["D"], z=t["z"][:, s].contiguous(),
                                             delta_bias=t["delta_bias"]))
    torch.cuda.synchronize()
    y_dec = torch.stack(ys, 1)
    # same fp32 arithmetic in the same order per step: agreement to rounding
    assert rel_err(to_f64(y_dec), to_f64(y_scan)) <= (1e-2 if bf16 else 1e-5)
    assert rel_err(to_f64(state), to_f64(last_scan)) <= 1e-5


def test_decode_workload_full_size_sampled():
    """256 x 5120 x 16 fp32 state, 1024 sequential bf16 steps on the GPU; the oracle
    follows sampled channels through all steps and checks every y and the final state."""
    w = W.WORKLOADS["decode"]
    dev = W.device_inputs(w)
    state = dev["state0"].clone()
    y_all = torch.empty((w.L, w.batch, w.d_inner), dtype=torch.bfloat16, device="cuda")
    for s in range(w.L):
        ssm.ssm_state_update(state, dev["u"][s], dev["delta"][s], dev["A"], dev["B"][s], dev["C"][s],
                             dev["D"], dev["z"][s], y_all[s], dev["delta_bias"], True)
    torch.cuda.synchronize()
    r = np.random.default_rng(4)
    b_sel = np.unique(np.concatenate([[0, w.batch - 1], r.choice(w.batch, 6, replace=False)]))
    d_sel = np.unique(np.concatenate([[0, w.d_inner - 1], r.choice(w.d_inner, 6, replace=False)]))
    x = W.host_decode_inputs(w, w.L, b_sel=b_sel, d_sel=d_sel)
    st = x["state0"]
    y_ref = np.empty((w.L, len(b_sel), len(d_sel)))
    for s in range(w.L):
        y_ref[s], st = oracle.state_update(st, x["u"][s], x["delta"][s], x["A"], x["B"][s],
                                           x["C"][s], D=x["D"], z=x["z"][s],
                                           delta_bias=x["delta_bias"], nthreads=1)
    bs, ds = torch.from_numpy(b_sel).cuda(), torch.from_numpy(d_sel).cuda()
    y_g = to_f64(y_all.index_select(1, bs).index_select(2, ds))
    st_g = to_f64(state.index_select(0, bs).index_select(1, ds))
    record_margin("decode 256x5120x16, 1024 steps (sampled)", BF16_TOL, y=rel_err(y_g, y_ref),
                  state=rel_err(st_g, st))
    assert rel_err(y_g, y_ref) <= BF16_TOL
    assert rel_err(st_g, st) <= BF16_TOL


@pytest.mark.parametrize("bf16", [False, True])
def test_decode_more_batch_rows_than_one_grid_column(bf16):
    """140,001 batch rows: more than the 2 x 65,535 a single pass of the 2-D grid covers (each
    CTA row serves two batch rows), so the kernel loops over batch rows; the odd count leaves
    the last pass with a single row.  Every row against the oracle."""
    batch, d_inner, N = 140001, 8, 4
    r = np.random.default_rng(140001)
    rnd = lambda *s: r.standard_normal(s).astype(np.float32)
    u, delta, z = rnd(batch, d_inner), 0.5 * rnd(batch, d_inner), rnd(batch, d_inner)
    B, C = rnd(batch, N), rnd(batch, N)
    state0 = 0.1 * rnd(batch, d_inner, N)
    A = -np.tile(np.arange(1, N + 1, dtype=np.float32), (d_inner, 1))
    D, bias = rnd(d_inner), (0.1 * rnd(d_inner)).astype(np.float32)
    io = lambda a: torch.from_numpy(a).cuda().to(torch.bfloat16 if bf16 else torch.float32)
    state = torch.from_numpy(state0).cuda()
    y = ssm.selective_state_update(state, io(u), io(delta), torch.from_numpy(A).cuda(), io(B), io(C),
                                   D=torch.from_numpy(D).cuda(), z=io(z),
                                   delta_bias=torch.from_numpy(bias).cuda())
    torch.cuda.synchronize()
    q = lambda a: io(a).float().cpu().numpy().astype(np.float64)  # the values the device holds
    y_ref, st_ref = oracle.state_update(state0, q(u), q(delta), A, q(B), q(C), D=D, z=q(z), delta_bias=bias)
    tol = BF16_TOL if bf16 else FP32_TOL
    ey, es = rel_err(to_f64(y), y_ref), rel_err(to_f64(state), st_ref)
    record_margin(f"decode {batch}x{d_inner}x{N} {'bf16' if bf16 else 'fp32'}, one step", tol, y=ey, state=es)
    assert ey <= tol and es <= tol, f"y err {ey:.3g}, state err {es:.3g}"
