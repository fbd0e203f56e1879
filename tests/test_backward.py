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
from tests.helpers import BF16_TOL, FP32_TOL, rel_err, to_f64, to_torch

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


@pytest.mark.parametrize("d_state", [1, 3, 8])
def test_backward_small_states_ragged(d_state):
    _run(3, 77, 40, d_state, False, seed=13 + d_state, with_dlast=True)


@pytest.mark.parametrize("flags", [dict(use_D=False), dict(use_z=False), dict(use_bias=False),
                                   dict(use_D=False, use_z=False, use_bias=False)])
def test_backward_optional_operands(flags):
    _run(2, 200, 32, 16, False, seed=17, **flags)


def test_backward_single_step():
    _run(2, 1, 16, 4, False, seed=19, with_h0=True)
