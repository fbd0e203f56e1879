"""ssm_scan_bwd (the training backward with recomputed states) against the oracle's
reverse-mode gradients, on chunked and ragged sequences, with and without the optional
operands."""
import numpy as np
import pytest
import torch

import inputgen
import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import record_margin, BF16_TOL, FP32_TOL, rel_err, to_f64, to_torch

pytestmark = pytest.mark.gpu


def _run(batch, L, d_inner, d_state, bf16, seed, use_D=True, use_z=True, use_bias=True,
         with_h0=False, with_dlast=False):
    w = W.Workload("bw", "backward case", batch, L, d_inner, d_state, bf16, seed, 0.5)
    raw = W.host_scan_inputs(w, raw=True)
    r = np.random.default_rng(seed)
    dy_raw = inputgen.normal(seed, 99, 0.0, 1.0, 0, batch * L * d_inner, bf16).reshape(batch, L, d_inner)
    h0 = r.normal(scale=0.3, size=(batch, d_inner, d_state)).astype(np.float32) if with_h0 else None
    dlast = r.normal(size=(batch, d_inner, d_state)).astype(np.float32) if with_dlast else None
    io = lambda k: bf16 and k in ("u", "delta", "z", "B", "C")
    t = {k: to_torch(v, io(k)) for k, v in raw.items()}
    dy = to_torch(dy_raw, bf16)
    g = ssm.selective_scan_backward(
        t["u"], t["delta"], t["A"], t["B"], t["C"], dy, D=t["D"] if use_D else None,
        z=t["z"] if use_z else None, delta_bias=t["delta_bias"] if use_bias else None,
        initial_state=torch.from_numpy(h0).cuda() if with_h0 else None,
        dlast_state=torch.from_numpy(dlast).cuda() if with_dlast else None)
    torch.cuda.synchronize()
    x = {k: (W._as_f64(v, bf16) if io(k) else v.astype(np.float64)) for k, v in raw.items()}
    ref = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], W._as_f64(dy_raw, bf16),
                          D=x["D"] if use_D else None, z=x["z"] if use_z else None,
                          delta_bias=x["delta_bias"] if use_bias else None,
                          initial_state=h0, dlast=dlast)
    tol = BF16_TOL if bf16 else FP32_TOL
    errs = {}
    for k, v in g.items():
        if k == "dinitial_state" and not with_h0 and not with_dlast and L == 0:
            continue
        errs[k] = rel_err(to_f64(v), ref[k])
    bad = {k: e for k, e in errs.items() if e > tol}
    assert not bad, f"gradient errors above {tol}: {bad} (all: {errs})"


@pytest.mark.parametrize("bf16", [False, True])
def test_backward_chunked(bf16):
    _run(2, 1500, 64, 16, bf16, seed=11)


def test_backward_long_sequence_few_channels():
    _run(1, 5000, 32, 16, False, seed=12, with_h0=True, with_dlast=True)


@pytest.mark.parametrize("d_state", [1, 3, 5, 8, 12, 16])
def test_backward_small_states_ragged(d_state):
    _run(3, 77, 40, d_state, False, seed=13 + d_state, with_dlast=True)


@pytest.mark.parametrize("flags", [dict(use_D=False), dict(use_z=False), dict(use_bias=False),
                                   dict(use_D=False, use_z=False, use_bias=False)])
def test_backward_optional_operands(flags):
    _run(2, 200, 32, 16, False, seed=17, **flags)


def test_backward_single_step():
    _run(2, 1, 16, 4, False, seed=19, with_h0=True)


@pytest.mark.parametrize("chunks", ["2", "5"])
@pytest.mark.parametrize("bf16", [False, True])
def test_backward_handover_chain(chunks, bf16, monkeypatch):
    """Time chunks run as a chain from the last back to the first, each handing its adjoint carry
    to the chunk before it (the plan the 2.8B shape takes), ragged, with an incoming dL/dlast
    and an initial state."""
    monkeypatch.setenv("SSM_BWD_CHUNKS", chunks)
    monkeypatch.setenv("SSM_BWD_HANDOVER", "1")
    _run(2, 1500, 96, 16, bf16, seed=23 + int(chunks), with_h0=True, with_dlast=True)


@pytest.mark.parametrize("key", ["mamba130m", "mamba2p8b"])
def test_backward_full_size_sampled(key):
    """The bench's backward at full size (inputs and dy ~ N(0, 1) filled on the device, the
    launch configuration the bench times).  Every gradient but dB and dC is per channel, so the
    oracle checks them exactly on sampled channels over every batch row and step; dB and dC
    (sums over all channels) are covered at the smaller sizes above."""
    w = W.WORKLOADS[key]
    dev = W.device_inputs(w)
    dy = torch.empty_like(dev["u"])
    inputgen.dev_fill_normal(w.seed, 9, 0.0, 1.0, 0, dy.numel(), w.bf16, dy.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    g = ssm.selective_scan_backward(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], dy,
                                    D=dev["D"], z=dev["z"], delta_bias=dev["delta_bias"])
    torch.cuda.synchronize()
    d_sel = np.unique(np.concatenate([[0, 1, 31, 32, w.d_inner - 1],
                                      np.random.default_rng(w.seed).choice(w.d_inner, 7, replace=False)]))
    ds = torch.from_numpy(d_sel).cuda()
    got = {k: to_f64(g[k].index_select(2, ds)) for k in ("du", "ddelta", "dz")}
    got["dA"] = to_f64(g["dA"].index_select(0, ds))
    got["dD"] = to_f64(g["dD"].index_select(0, ds))
    got["ddelta_bias"] = to_f64(g["ddelta_bias"].index_select(0, ds))
    got["dinitial_state"] = to_f64(g["dinitial_state"].index_select(1, ds))
    del dev, dy, g
    x = W.host_scan_inputs(w, d_sel=d_sel)
    t = np.arange(w.L, dtype=np.int64)
    idx = ((np.arange(w.batch)[:, None, None] * w.L + t[None, :, None]) * w.d_inner
           + d_sel[None, None, :]).ravel()
    dy_ref = W._as_f64(inputgen.normal_at(w.seed, 9, 0.0, 1.0, idx, w.bf16), w.bf16).reshape(
        w.batch, w.L, len(d_sel))
    ref = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy_ref, D=x["D"], z=x["z"],
                          delta_bias=x["delta_bias"])
    tol = BF16_TOL if w.bf16 else FP32_TOL
    errs = {k: rel_err(v, ref[k]) for k, v in got.items()}
    record_margin(f"backward {w.key} (full size, sampled)", tol, **errs)
    bad = {k: e for k, e in errs.items() if e > tol}
    assert not bad, f"gradient errors above {tol}: {bad} (all: {errs})"


def test_backward_launch_count():
    """ssm_scan_bwd_launches: forward recompute + gradients, plus the reverse summaries when the
    plan joins its chunks by summaries (the 130M shape) rather than a hand-over chain or not at
    all (the 2.8B shape on a 148-SM B300)."""
    big = ssm.ssm_scan_bwd_launches(8, 2048, 5120, 16, ssm.SSM_BF16)
    small = ssm.ssm_scan_bwd_launches(2, 2048, 1536, 16, ssm.SSM_F32)
    assert big in (2, 3) and small in (2, 3)
    if torch.cuda.get_device_properties(0).multi_processor_count == 148:
        assert (big, small) == (2, 3)
    assert ssm.ssm_scan_bwd_launches(2, 0, 1536, 16, ssm.SSM_F32) == 0
