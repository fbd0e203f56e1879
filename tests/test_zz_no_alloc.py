"""ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device memory where
they call it (the library supplies a fixed scratch array instead of a caller workspace).
It must give the same results as ssm_scan_fwd, bit for bit, call after call, and refuse
problems whose scratch need exceeds the array.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import selective_state_space_161_b300 as ssm
from inputgen import workloads as W
from tests.helpers import BF16_TOL, FP32_TOL, rel_err, to_f64, to_torch

pytestmark = pytest.mark.gpu


def _inputs(w):
    raw = W.host_scan_inputs(w, raw=True)
    return {k: to_torch(v, w.bf16 and k in ("u", "delta", "z", "B", "C")) for k, v in raw.items()}


@pytest.mark.parametrize("bf16,batch,L,d_inner", [(False, 2, 2048, 1536), (True, 1, 6000, 256)])
def test_noalloc_matches_workspace_entry_point(bf16, batch, L, d_inner):
    w = W.Workload("na", "no-alloc check", batch, L, d_inner, 16, bf16, 77, 0.5)
    io = ssm.SSM_BF16 if bf16 else ssm.SSM_F32
    need = ssm.ssm_scan_fwd_workspace_size(batch, L, d_inner, 16, io)
    assert 0 < need <= ssm.SSM_NOALLOC_SCRATCH_BYTES  # the case really uses the scratch
    t = _inputs(w)
    y_ref = torch.empty_like(t["u"])
    last_ref = torch.empty((batch, d_inner, 16), device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ssm.ssm_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
                     True, y_ref, last_ref, ws)
    tol = BF16_TOL if bf16 else FP32_TOL
    for _ in range(2):  # two calls in a row share the library's scratch
        y = torch.full_like(t["u"], float("nan"))
        last = torch.full((batch, d_inner, 16), float("nan"), device="cuda")
        ssm.ssm_scan_fwd_noalloc(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                 t["delta_bias"], True, y, last)
        torch.cuda.synchronize()
        # same plan, same kernels: the results must agree bit for bit, so stale records left
        # in the shared scratch by the previous call cannot hide inside the tolerance
        assert torch.equal(y, y_ref) and torch.equal(last, last_ref)
        assert rel_err(to_f64(y), to_f64(y_ref)) <= tol
        assert rel_err(to_f64(last), to_f64(last_ref)) <= tol
        assert ssm.ssm_get_status(None) == 0


def test_noalloc_refuses_problems_beyond_its_scratch(monkeypatch):
    lib = ssm.load_library()
    x = torch.zeros(64, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    # The default plan keeps the records within one wave of CTAs (a few MiB); forcing 4096
    # time chunks on a 1,048,576-token sequence over 2048 channels needs far more.
    monkeypatch.setenv("SSM_SCAN_CHUNKS", "4096")
    need = ssm.ssm_scan_fwd_workspace_size(1, 1 << 20, 2048, 16, ssm.SSM_BF16)
    assert need > ssm.SSM_NOALLOC_SCRATCH_BYTES
    rc = lib.ssm_scan_fwd_noalloc(p, p, p, p, p, None, None, None, 1, p, None, 1, 1 << 20, 2048,
                                  16, ssm.SSM_BF16, None)
    assert rc == ssm.SSM_ERR_SCRATCH_LIMIT and "scratch" in ssm.ssm_status_string(rc)
