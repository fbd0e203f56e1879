"""The time-chunk look-back of the forward scan: many chunks (look-back windows of more than
32 predecessors), deterministic results, the status word, and the bounded wait (a wait that
runs out is reported by ssm_get_status, and the GPU stays usable)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import BF16_TOL, FP32_TOL, record_margin, rel_err, to_f64, to_torch

pytestmark = pytest.mark.gpu


def _inputs(batch, L, d_inner, d_state, bf16, seed):
    w = W.Workload("lb", "look-back case", batch, L, d_inner, d_state, bf16, seed, 0.5)
    raw = W.host_scan_inputs(w, raw=True)
    t = {k: to_torch(v, bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}
    return w, raw, t


def _call(t, batch, L, d_inner, d_state, bf16):
    io = ssm.SSM_BF16 if bf16 else ssm.SSM_F32
    ws = torch.empty(ssm.ssm_scan_fwd_workspace_size(batch, L, d_inner, d_state, io),
                     dtype=torch.uint8, device="cuda")
    y = torch.empty_like(t["u"])
    last = torch.empty((batch, d_inner, d_state), device="cuda")
    ssm.ssm_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                     True, y, last, ws)
    return y, last, ws


@pytest.mark.parametrize("chunks", ["40", "150"])
def test_many_chunks_match_oracle(chunks, monkeypatch):
    """40 and 150 time chunks: the last chunks look back over more than one window of 32."""
    monkeypatch.setenv("SSM_SCAN_CHUNKS", chunks)
    batch, L, d_inner, d_state, bf16 = 1, 20000, 64, 16, False
    w, raw, t = _inputs(batch, L, d_inner, d_state, bf16, seed=41)
    y, last, ws = _call(t, batch, L, d_inner, d_state, bf16)
    assert ssm.ssm_get_status(ws) == 0
    x = {k: (W._as_f64(v, bf16) if k in ("u", "delta", "z", "B", "C") else v.astype(np.float64))
         for k, v in raw.items()}
    y_ref, last_ref = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                      delta_bias=x["delta_bias"])
    ey, el = rel_err(to_f64(y), y_ref), rel_err(to_f64(last), last_ref)
    record_margin(f"scan 1x20000x64x16 fp32, {chunks} chunks", FP32_TOL, y=ey, last_state=el)
    assert ey <= FP32_TOL and el <= FP32_TOL, f"y err {ey:.3g}, last_state err {el:.3g}"


@pytest.mark.parametrize("lanes", ["1", "2", "4"])
def test_two_equal_chunks_match_oracle(lanes, monkeypatch):
    """Two chunks of equal length (the plan for one uneven wave of CTAs): the second chunk runs
    no aggregate and waits for the first's end state; ragged length and channel count."""
    monkeypatch.setenv("SSM_SCAN_CHUNKS", "2")
    monkeypatch.setenv("SSM_SCAN_ALPHA", "1.0")
    monkeypatch.setenv("SSM_SCAN_LANES", lanes)
    batch, L, d_inner, d_state, bf16 = 3, 1001, 72, 16, False
    w, raw, t = _inputs(batch, L, d_inner, d_state, bf16, seed=47 + int(lanes))
    y, last, ws = _call(t, batch, L, d_inner, d_state, bf16)
    assert ssm.ssm_get_status(ws) == 0
    x = {k: v.astype(np.float64) for k, v in raw.items()}
    y_ref, last_ref = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                      delta_bias=x["delta_bias"])
    ey, el = rel_err(to_f64(y), y_ref), rel_err(to_f64(last), last_ref)
    record_margin(f"scan 3x1001x72x16 fp32, two equal chunks, {lanes} lane(s)", FP32_TOL, y=ey, last_state=el)
    assert ey <= FP32_TOL and el <= FP32_TOL, f"y err {ey:.3g}, last_state err {el:.3g}"


@pytest.mark.parametrize("chunks", ["3", "5"])
def test_chunk_chain_matches_oracle(chunks, monkeypatch):
    """Time chunks as a chain (four lanes per pair): no aggregate passes, every chunk continues
    from its predecessor's end state; ragged length and channel count."""
    monkeypatch.setenv("SSM_SCAN_CHUNKS", chunks)
    monkeypatch.setenv("SSM_SCAN_CHAIN", "1")
    monkeypatch.setenv("SSM_SCAN_LANES", "4")
    batch, L, d_inner, d_state, bf16 = 2, 1501, 72, 16, False
    w, raw, t = _inputs(batch, L, d_inner, d_state, bf16, seed=61 + int(chunks))
    y, last, ws = _call(t, batch, L, d_inner, d_state, bf16)
    assert ssm.ssm_get_status(ws) == 0
    x = {k: v.astype(np.float64) for k, v in raw.items()}
    y_ref, last_ref = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                      delta_bias=x["delta_bias"])
    ey, el = rel_err(to_f64(y), y_ref), rel_err(to_f64(last), last_ref)
    record_margin(f"scan 2x1501x72x16 fp32, chain of {chunks} chunks", FP32_TOL, y=ey, last_state=el)
    assert ey <= FP32_TOL and el <= FP32_TOL, f"y err {ey:.3g}, last_state err {el:.3g}"


def test_results_are_deterministic():
    """The carry is folded forward from whichever inclusive prefix the look-back finds, in the
    order the chunks themselves use, so repeated calls agree bit for bit."""
    batch, L, d_inner, d_state, bf16 = 2, 30000, 128, 16, True
    _, _, t = _inputs(batch, L, d_inner, d_state, bf16, seed=42)
    y0, l0, _ = _call(t, batch, L, d_inner, d_state, bf16)
    for _ in range(3):
        y, last, _ = _call(t, batch, L, d_inner, d_state, bf16)
        torch.cuda.synchronize()
        assert torch.equal(y, y0) and torch.equal(last, l0)


def test_bounded_wait_reports_timeout_and_gpu_stays_usable(monkeypatch):
    """With the self-test switch every look-back waits for records of a tag that no CTA
    writes; the waits give up after 64 polls, the kernel finishes, ssm_get_status reports
    SSM_ERR_LOOKBACK_TIMEOUT, and the next ordinary call is correct and reports OK."""
    batch, L, d_inner, d_state, bf16 = 1, 8192, 64, 16, False
    w, raw, t = _inputs(batch, L, d_inner, d_state, bf16, seed=43)
    y_ok, last_ok, ws_ok = _call(t, batch, L, d_inner, d_state, bf16)
    assert ssm.ssm_get_status(ws_ok) == 0
    monkeypatch.setenv("SSM_LOOKBACK_SELFTEST", "1")
    monkeypatch.setenv("SSM_LOOKBACK_MAX_POLLS", "64")
    _, _, ws = _call(t, batch, L, d_inner, d_state, bf16)
    assert ssm.ssm_get_status(ws) == ssm.SSM_ERR_LOOKBACK_TIMEOUT
    assert "waited too long" in ssm.ssm_status_string(ssm.SSM_ERR_LOOKBACK_TIMEOUT)
    monkeypatch.delenv("SSM_LOOKBACK_SELFTEST")
    monkeypatch.delenv("SSM_LOOKBACK_MAX_POLLS")
    y, last, ws2 = _call(t, batch, L, d_inner, d_state, bf16)
    assert ssm.ssm_get_status(ws2) == 0
    assert torch.equal(y, y_ok) and torch.equal(last, last_ok)
    # the same workspace, reused by an ordinary call, reports OK again
    y3 = torch.empty_like(t["u"])
    ssm.ssm_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                     True, y3, None, ws)
    assert ssm.ssm_get_status(ws) == 0
    assert torch.equal(y3, y_ok)


def test_get_status_without_workspace_checks_the_stream():
    assert ssm.ssm_get_status(None) == 0


def test_backward_recompute_reports_timeout(monkeypatch):
    """The backward's forward recompute runs the chunked look-back kernel in the backward's
    workspace: a wait that runs out is reported by ssm_get_status on that workspace, and the
    next ordinary call gives the same gradients as before."""
    batch, L, d_inner, d_state, bf16 = 1, 8192, 64, 16, False
    _, _, t = _inputs(batch, L, d_inner, d_state, bf16, seed=44)
    dy = torch.randn(batch, L, d_inner, device="cuda")

    def run():
        g = dict(du=torch.empty_like(t["u"]), ddelta=torch.empty_like(t["u"]), dz=torch.empty_like(t["u"]),
                 dA=torch.empty((d_inner, d_state), device="cuda"),
                 dB=torch.empty((batch, L, d_state), device="cuda"),
                 dC=torch.empty((batch, L, d_state), device="cuda"),
                 dD=torch.empty(d_inner, device="cuda"), dbias=torch.empty(d_inner, device="cuda"))
        ws = torch.empty(ssm.ssm_scan_bwd_workspace_size(batch, L, d_inner, d_state, ssm.SSM_F32),
                         dtype=torch.uint8, device="cuda")
        ssm.ssm_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                         True, None, dy, None, g["du"], g["ddelta"], g["dA"], g["dB"], g["dC"], g["dD"],
                         g["dz"], g["dbias"], None, ws)
        return g, ws

    g0, ws0 = run()
    assert ssm.ssm_get_status(ws0) == 0
    monkeypatch.setenv("SSM_LOOKBACK_SELFTEST", "1")
    monkeypatch.setenv("SSM_LOOKBACK_MAX_POLLS", "64")
    _, ws1 = run()
    assert ssm.ssm_get_status(ws1) == ssm.SSM_ERR_LOOKBACK_TIMEOUT
    monkeypatch.delenv("SSM_LOOKBACK_SELFTEST")
    monkeypatch.delenv("SSM_LOOKBACK_MAX_POLLS")
    g2, ws2 = run()
    assert ssm.ssm_get_status(ws2) == 0
    for k in ("du", "ddelta", "dz"):  # per element: bit for bit
        assert torch.equal(g2[k], g0[k]), k
    for k in ("dA", "dB", "dC", "dD", "dbias"):
        # atomic sums over 128 time chunks: the order, and with cancellation the last few bits
        # of a sum relative to its terms, vary from run to run
        scale = g0[k].abs().max().item()
        assert torch.allclose(g2[k], g0[k], rtol=1e-5, atol=1e-5 * scale), k
