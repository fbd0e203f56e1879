"""GPU parity of ssm_scan_fwd against the float64 oracle, element by element,
on the seeded workloads and on edge cases (ragged tiles and chunks, optional
operands, empty sequences, every d_state)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import BF16_TOL, FP32_TOL, record_margin, rel_err, to_f64, to_torch

pytestmark = pytest.mark.gpu


def _random_case(batch, L, d_inner, d_state, bf16, seed, delta_sd=0.5):
    """Small case drawn from the workload recipe (same distributions, own seed)."""
    w = W.Workload("case", "edge case", batch, L, d_inner, d_state, bf16, seed, delta_sd)
    return w, W.host_scan_inputs(w, raw=True)


def _run_gpu(raw, bf16, use_D=True, use_z=True, use_bias=True, softplus=True):
    t = {k: to_torch(v, bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    y, last = ssm.selective_scan(t["u"], t["delta"], t["A"], t["B"], t["C"],
                                 D=t["D"] if use_D else None, z=t["z"] if use_z else None,
                                 delta_bias=t["delta_bias"] if use_bias else None,
                                 softplus=softplus)
    torch.cuda.synchronize()
    return to_f64(y), to_f64(last)


def _run_oracle(w, raw, use_D=True, use_z=True, use_bias=True, softplus=True):
    x = {k: (W._as_f64(v, w.bf16) if k in ("u", "delta", "z", "B", "C") else v.astype(np.float64))
         for k, v in raw.items()}
    return oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"] if use_D else None,
                           z=x["z"] if use_z else None,
                           delta_bias=x["delta_bias"] if use_bias else None, softplus_flag=softplus)


def _check(w, raw, name=None, **flags):
    y, last = _run_gpu(raw, w.bf16, **flags)
    y_ref, last_ref = _run_oracle(w, raw, **flags)
    tol = BF16_TOL if w.bf16 else FP32_TOL
    ey, el = rel_err(y, y_ref), rel_err(last, last_ref)
    if name:
        record_margin(name, tol, y=ey, last_state=el)
    assert ey <= tol and el <= tol, f"y err {ey:.3g}, last_state err {el:.3g} (tol {tol})"
    return ey, el


def test_tiny_workload_full():
    w = W.WORKLOADS["tiny"]
    raw = W.host_scan_inputs(w, raw=True)
    _check(w, raw, name="scan tiny (1x64x16x4 fp32)")


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("d_state", [1, 3, 4, 7, 16])
def test_every_state_size(d_state, bf16):
    w, raw = _random_case(2, 77, 40, d_state, bf16, seed=100 + d_state)
    _check(w, raw)


@pytest.mark.parametrize("flags", [dict(use_D=False), dict(use_z=False), dict(use_bias=False),
                                   dict(softplus=False, use_bias=False),
                                   dict(use_D=False, use_z=False, use_bias=False)])
def test_optional_operands(flags):
    w, raw = _random_case(2, 65, 136, 16, False, seed=7)
    if not flags.get("softplus", True):
        raw["delta"] = np.abs(raw["delta"]) * 0.1  # keep delta positive without softplus
    _check(w, raw, **flags)


@pytest.mark.parametrize("lanes", ["1", "4"])
def test_positive_and_mixed_A(lanes, monkeypatch):
    """A is taken as given: positive entries (a growing state, exp(delta A) > 1) and a mix of
    signs and magnitudes per channel, over a sequence short enough to stay finite, and over
    several time chunks so that the look-back folds exp(A sum delta) > 1 as well."""
    monkeypatch.setenv("SSM_SCAN_LANES", lanes)
    monkeypatch.setenv("SSM_SCAN_CHUNKS", "4")
    w, raw = _random_case(2, 300, 64, 16, False, seed=211)
    r = np.random.default_rng(211)
    raw["A"] = r.uniform(-3.0, 0.05, size=raw["A"].shape).astype(np.float32)
    raw["A"][:8] = np.abs(raw["A"][:8]) * 0.02 + 0.01  # eight channels with every A positive
    _check(w, raw, name=f"scan 2x300x64x16 fp32, mixed-sign A, {lanes} lane(s)")


@pytest.mark.parametrize("bf16", [False, True])
def test_many_time_chunks_ragged(bf16):
    # 8 channels and 5000 steps: the GPU is filled by cutting time into many chunks
    # (last one ragged), so the chunk-summary composition is exercised.
    w, raw = _random_case(1, 5000, 8, 16, bf16, seed=11)
    _check(w, raw)


def test_single_step_and_short_sequences():
    for L in (1, 2, 31, 33):
        w, raw = _random_case(3, L, 24, 5, False, seed=L)
        _check(w, raw)


def test_empty_sequence_gives_zero_state():
    dev = "cuda"
    u = torch.empty((2, 0, 16), device=dev)
    A = -torch.ones((16, 4), device=dev)
    B = torch.empty((2, 0, 4), device=dev)
    last = torch.full((2, 16, 4), 7.0, device=dev)
    y = torch.empty_like(u)
    ssm.ssm_scan_fwd(u, u, A, B, B, None, None, None, True, y, last, None)
    torch.cuda.synchronize()
    assert torch.all(last == 0)


def test_zero_step_size_is_exact():
    """delta = 0 (softplus off, no bias): y = D u silu(z), state 0 -- exact up to the gate's rounding."""
    w, raw = _random_case(1, 50, 32, 16, False, seed=3)
    raw["delta"][:] = 0
    y, last = _run_gpu(raw, False, use_bias=False, softplus=False)
    assert np.all(last == 0.0)
    u, z = raw["u"].astype(np.float64), raw["z"].astype(np.float64)
    ref = raw["D"].astype(np.float64) * u * z / (1 + np.exp(-z))
    assert rel_err(y, ref) < 1e-6


def _sampled_channels(d_inner, k, seed):
    r = np.random.default_rng(seed)
    edge = [0, 1, 127, 128, d_inner - 1]
    pick = r.choice(d_inner, size=k, replace=False)
    return np.unique(np.concatenate([edge, pick]))


@pytest.mark.parametrize("key", ["mamba130m", "mamba2p8b"])
def test_full_size_workload_sampled(key):
    """Full-size workload on the GPU (inputs filled on the device); the oracle
    recomputes sampled channels over the whole sequence for every batch."""
    w = W.WORKLOADS[key]
    dev = W.device_inputs(w)
    y, last = ssm.selective_scan(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], D=dev["D"],
                                 z=dev["z"], delta_bias=dev["delta_bias"], softplus=True)
    torch.cuda.synchronize()
    d_sel = _sampled_channels(w.d_inner, 12, w.seed)
    b_sel = np.arange(w.batch)
    raw = W.host_scan_inputs(w, b_sel=b_sel, d_sel=d_sel)
    # device fill and host draws must agree bit for bit on the sampled slice
    np.testing.assert_array_equal(to_f64(dev["u"][:, :, d_sel]), raw["u"])
    y_ref, last_ref = oracle.scan_fwd(raw["u"], raw["delta"], raw["A"], raw["B"], raw["C"],
                                      D=raw["D"], z=raw["z"], delta_bias=raw["delta_bias"])
    tol = BF16_TOL if w.bf16 else FP32_TOL
    ds = torch.from_numpy(d_sel).cuda()
    ey = rel_err(to_f64(y.index_select(2, ds)), y_ref)
    el = rel_err(to_f64(last.index_select(1, ds)), last_ref)
    record_margin(f"scan {key} (full size, sampled channels)", tol, y=ey, last_state=el)
    assert ey <= tol and el <= tol, f"y err {ey:.3g}, last_state err {el:.3g}"


def test_long_context_sampled():
    """1,048,576-token sequence in one call; the oracle runs the full sequence on
    sampled channels, checking every y and the final state."""
    w = W.WORKLOADS["long"]
    dev = W.device_inputs(w)
    y, last = ssm.selective_scan(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], D=dev["D"],
                                 z=dev["z"], delta_bias=dev["delta_bias"], softplus=True)
    torch.cuda.synchronize()
    d_sel = _sampled_channels(w.d_inner, 3, w.seed)
    ds = torch.from_numpy(d_sel).cuda()
    y_s = to_f64(y.index_select(2, ds))
    last_s = to_f64(last.index_select(1, ds))
    del dev, y
    raw = W.host_scan_inputs(w, d_sel=d_sel)
    y_ref, last_ref = oracle.scan_fwd(raw["u"], raw["delta"], raw["A"], raw["B"], raw["C"],
                                      D=raw["D"], z=raw["z"], delta_bias=raw["delta_bias"])
    ey, el = rel_err(y_s, y_ref), rel_err(last_s, last_ref)
    record_margin("scan long (1x1048576x2048x16 bf16, sampled channels)", BF16_TOL, y=ey, last_state=el)
    assert ey <= BF16_TOL and el <= BF16_TOL, f"y err {ey:.3g}, last_state err {el:.3g}"


def test_bad_arguments_raise():
    x = torch.zeros((1, 4, 8), device="cuda")
    A = torch.zeros((8, 4), device="cuda")
    Bm = torch.zeros((1, 4, 4), device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(ssm.SsmError):
        # offset view: data pointer no longer 16-byte aligned
        xs = torch.zeros(1 * 4 * 8 + 1, device="cuda")[1:].view(1, 4, 8)
        ssm.ssm_scan_fwd(xs, x, A, Bm, Bm, None, None, None, True, y, None, None)


@pytest.mark.parametrize("lanes", ["1", "2", "4"])
@pytest.mark.parametrize("bf16,d_state,batch,L,d_inner", [
    (False, 16, 2, 3000, 96), (True, 16, 1, 4100, 64), (False, 5, 3, 700, 40), (True, 1, 2, 257, 24)])
def test_both_kernels(lanes, bf16, d_state, batch, L, d_inner, monkeypatch):
    """Every kernel variant (the states of a channel pair on one, two or four lanes), chunked
    and ragged, against the oracle."""
    monkeypatch.setenv("SSM_SCAN_LANES", lanes)
    w, raw = _random_case(batch, L, d_inner, d_state, bf16, seed=900 + d_state + int(lanes))
    _check(w, raw, name=f"scan {batch}x{L}x{d_inner}x{d_state} {'bf16' if bf16 else 'fp32'}, {lanes} lane(s)")
