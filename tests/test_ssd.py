"""ssm_ssd_fwd (chunked tensor-core form for one A and one step size per head) against the
oracle's scan run on the equivalent per-channel operands."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import record_margin, BF16_TOL, rel_err, to_f64

pytestmark = pytest.mark.gpu


def _run(w, use_D=True, use_z=True, use_bias=True, d_sel=None, tag=""):
    dev = W.device_ssd_inputs(w)
    y, last = ssm.selective_scan_ssd(dev["x"], dev["dt"], dev["A_head"], dev["B"], dev["C"],
                                     D=dev["D"] if use_D else None, z=dev["z"] if use_z else None,
                                     dt_bias=dev["dt_bias"] if use_bias else None)
    torch.cuda.synchronize()
    x = W.host_ssd_inputs(w, d_sel=d_sel)
    y_ref, last_ref = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"],
                                      D=x["D"] if use_D else None, z=x["z"] if use_z else None,
                                      delta_bias=x["delta_bias"] if use_bias else None)
    if d_sel is not None:
        ds = torch.from_numpy(np.asarray(d_sel)).cuda()
        y, last = y.index_select(2, ds), last.index_select(1, ds)
    ey, el = rel_err(to_f64(y), y_ref), rel_err(to_f64(last), last_ref)
    record_margin(f"ssd {w.batch}x{w.L}x{w.d_inner}x{w.d_state}, {w.heads} heads{tag}", BF16_TOL, y=ey,
                  last_state=el)
    assert ey <= BF16_TOL and el <= BF16_TOL, f"y err {ey:.3g}, last_state err {el:.3g}"


@pytest.mark.parametrize("N", [16, 32, 64, 128])
def test_ssd_small_ragged(N):
    # 200 steps: three full chunks of 64 and a ragged one
    _run(W.Workload("ssd", "ssd case", 2, 200, 128, N, True, 40 + N, 0.5, heads=2))


@pytest.mark.parametrize("flags", [dict(use_D=False), dict(use_z=False), dict(use_bias=False)])
def test_ssd_optional_operands(flags):
    _run(W.Workload("ssd", "ssd case", 1, 130, 192, 64, True, 7, 0.5, heads=3), **flags)


def test_ssd_single_step_and_one_chunk():
    _run(W.Workload("ssd", "ssd case", 3, 1, 64, 16, True, 8, 0.5, heads=1))
    _run(W.Workload("ssd", "ssd case", 1, 64, 64, 128, True, 9, 0.5, heads=1))


def test_ssd_full_size_sampled():
    """Mamba-2-2.7B-shaped layer on the GPU; the oracle follows sampled channels of three heads."""
    w = W.WORKLOADS["ssd2p7b"]
    d_sel = np.concatenate([np.arange(0, 4), np.arange(64 * 37 + 30, 64 * 37 + 34), np.arange(5116, 5120)])
    _run(w, d_sel=d_sel)


def test_ssd_without_softplus():
    """softplus_flag = 0: the step size is dt (+ bias) as given; here dt = |raw| / 8, which is
    exact in bf16 on either side, and no bias, so every step size is positive."""
    w = W.Workload("ssd", "ssd case", 2, 150, 128, 32, True, 77, 0.5, heads=2)
    dev = W.device_ssd_inputs(w)
    dt = dev["dt"].abs() / 8
    y, last = ssm.selective_scan_ssd(dev["x"], dt, dev["A_head"], dev["B"], dev["C"], D=dev["D"],
                                     z=dev["z"], dt_bias=None, softplus=False)
    torch.cuda.synchronize()
    x = W.host_ssd_inputs(w)
    y_ref, last_ref = oracle.scan_fwd(x["u"], np.abs(x["delta"]) / 8, x["A"], x["B"], x["C"], D=x["D"],
                                      z=x["z"], delta_bias=None, softplus_flag=False)
    ey, el = rel_err(to_f64(y), y_ref), rel_err(to_f64(last), last_ref)
    record_margin(f"ssd {w.batch}x{w.L}x{w.d_inner}x{w.d_state}, {w.heads} heads, no softplus", BF16_TOL, y=ey, last_state=el)
    assert ey <= BF16_TOL and el <= BF16_TOL, f"y err {ey:.3g}, last_state err {el:.3g}"


def test_ssd_empty_sequence_gives_zero_state():
    w = W.Workload("ssd", "ssd case", 2, 0, 128, 64, True, 3, 0.5, heads=2)
    x = torch.empty((2, 0, 128), dtype=torch.bfloat16, device="cuda")
    dt = torch.empty((2, 0, 2), dtype=torch.bfloat16, device="cuda")
    bc = torch.empty((2, 0, 64), dtype=torch.bfloat16, device="cuda")
    A = torch.from_numpy(W.ssd_A_head(w)).cuda()
    y, last = ssm.selective_scan_ssd(x, dt, A, bc, bc)
    torch.cuda.synchronize()
    assert y.shape == (2, 0, 128) and torch.count_nonzero(last).item() == 0


@pytest.mark.parametrize("N", [16, 32, 64, 128])
def test_ssd_tcgen05_chain_ragged(N, monkeypatch):
    """The opt-in per-head chain with every product on tcgen05 (SSM_SSD_KERNEL=tc), ragged."""
    monkeypatch.setenv("SSM_SSD_KERNEL", "tc")
    _run(W.Workload("ssd", "ssd case", 2, 200, 128, N, True, 60 + N, 0.5, heads=2), tag=", tcgen05 chain")


def test_ssd_tcgen05_chain_full_size_sampled(monkeypatch):
    monkeypatch.setenv("SSM_SSD_KERNEL", "tc")
    w = W.WORKLOADS["ssd2p7b"]
    d_sel = np.concatenate([np.arange(0, 4), np.arange(64 * 53 + 10, 64 * 53 + 14), np.arange(5100, 5104)])
    _run(w, d_sel=d_sel, tag=", tcgen05 chain")


def _ssd_call(dev, ws=None):
    y = torch.empty_like(dev["x"])
    last = torch.empty((dev["x"].shape[0], dev["x"].shape[2], dev["B"].shape[2]), device="cuda")
    if ws is None:
        b, L, d = dev["x"].shape
        ws = torch.empty((ssm.ssm_ssd_fwd_workspace_size(b, L, d, dev["dt"].shape[2], dev["B"].shape[2]),),
                         dtype=torch.uint8, device="cuda")
    ssm.ssm_ssd_fwd(dev["x"], dev["dt"], dev["A_head"], dev["B"], dev["C"], dev["D"], dev["z"], dev["dt_bias"],
                    True, y, last, ws)
    return y, last, ws


@pytest.mark.parametrize("kernel", ["mma", "tc"])
@pytest.mark.parametrize("L,parts", [(130, 2), (200, 2), (200, 3), (2048, 2), (2048, 5), (2048, 32)])
def test_ssd_time_parts_match_one_walk(L, parts, kernel, monkeypatch):
    """Time parts (each starting from the state the part before hands over) run the same
    operations in the same order as one walk over all chunks: bit-identical outputs, for the
    mma.sync chain and the tcgen05 chain."""
    monkeypatch.setenv("SSM_SSD_KERNEL", kernel)
    w = W.Workload("ssd", "ssd case", 2, L, 192, 64, True, 300 + L, 0.5, heads=3)
    dev = W.device_ssd_inputs(w)
    monkeypatch.setenv("SSM_SSD_PARTS", "1")
    y1, l1, _ = _ssd_call(dev)
    monkeypatch.setenv("SSM_SSD_PARTS", str(parts))
    y2, l2, ws = _ssd_call(dev)
    torch.cuda.synchronize()
    assert ssm.ssm_get_status(ws) == 0
    assert torch.equal(y1, y2) and torch.equal(l1, l2)


@pytest.mark.parametrize("kernel", ["mma", "tc"])
def test_ssd_time_part_wait_reports_timeout(kernel, monkeypatch):
    """A time part's wait for the state of the part before is bounded: with a tag nobody writes
    and a 64-poll limit it gives up, the call reports SSM_ERR_LOOKBACK_TIMEOUT and the next call
    is clean again.  No GPU fault is involved: the CTAs just finish."""
    w = W.Workload("ssd", "ssd case", 1, 256, 128, 32, True, 71, 0.5, heads=2)
    dev = W.device_ssd_inputs(w)
    monkeypatch.setenv("SSM_SSD_KERNEL", kernel)
    monkeypatch.setenv("SSM_SSD_PARTS", "2")
    monkeypatch.setenv("SSM_LOOKBACK_SELFTEST", "1")
    monkeypatch.setenv("SSM_LOOKBACK_MAX_POLLS", "64")
    _, _, ws = _ssd_call(dev)
    assert ssm.ssm_get_status(ws) == ssm.SSM_ERR_LOOKBACK_TIMEOUT
    monkeypatch.delenv("SSM_LOOKBACK_SELFTEST")
    monkeypatch.delenv("SSM_LOOKBACK_MAX_POLLS")
    _, _, ws = _ssd_call(dev, ws)
    assert ssm.ssm_get_status(ws) == 0


@pytest.mark.parametrize("kernel", ["mma", "tc"])
def test_ssd_status_word_reports_ok(kernel, monkeypatch):
    """Every chunked SSD call writes its status word at the start of the workspace (the waits
    that could raise it are bounded); a completed call reads back as SSM_OK."""
    monkeypatch.setenv("SSM_SSD_KERNEL", kernel)
    w = W.Workload("ssd", "ssd case", 1, 130, 128, 64, True, 91, 0.5, heads=2)
    dev = W.device_ssd_inputs(w)
    y = torch.empty_like(dev["x"])
    # every byte 7: a status word the call did not write would read as the timeout code
    ws = torch.full((ssm.ssm_ssd_fwd_workspace_size(1, 130, 128, 2, 64),), 7, dtype=torch.uint8, device="cuda")
    assert ssm.ssm_get_status(ws) == ssm.SSM_ERR_LOOKBACK_TIMEOUT
    ssm.ssm_ssd_fwd(dev["x"], dev["dt"], dev["A_head"], dev["B"], dev["C"], dev["D"], dev["z"], dev["dt_bias"],
                    True, y, None, ws)
    assert ssm.ssm_get_status(ws) == 0
