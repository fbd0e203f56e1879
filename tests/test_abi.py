"""The C ABI library: it loads, exports every symbol include/ssm.h declares,
and rejects bad arguments on the host (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

import selective_state_space_161_b300 as ssm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"SSM_API\s+[\w\s\*]+?\b(ssm_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = ssm.load_library()
    declared = _declared()
    assert {"ssm_scan_fwd", "ssm_state_update", "ssm_scan_fwd_workspace_size"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(ssm.EXPORTED_SYMBOLS) <= declared


def test_version_and_status_strings():
    assert ssm.ssm_version() >= 100
    assert ssm.ssm_status_string(0) == "ok"
    assert "aligned" in ssm.ssm_status_string(4)


def _scan_rc(**kw):
    lib = ssm.load_library()
    args = dict(u=None, delta=None, A=None, B=None, C=None, D=None, z=None, bias=None, sp=1, y=None,
                last=None, batch=1, L=8, d_inner=8, d_state=4, io=0, ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return lib.ssm_scan_fwd(*args.values())


def test_host_validation_before_any_device_call():
    assert _scan_rc(io=7) == 3                     # dtype
    assert _scan_rc(d_state=0) == 2                # d_state range
    assert _scan_rc(d_state=17) == 2
    assert _scan_rc(d_inner=6) == 2                # fp32 needs d_inner % 4 == 0
    assert _scan_rc(d_inner=12, io=1) == 2         # bf16 needs d_inner % 8 == 0
    assert _scan_rc(batch=-1) == 2
    assert _scan_rc(L=-3) == 2
    assert _scan_rc(batch=0) == 0                  # empty problem: nothing to do
    assert _scan_rc(d_inner=0) == 0
    lib = ssm.load_library()
    assert lib.ssm_state_update(*([None] * 10), 1, 2, 8, 0, 0, None) == 2


def _ssd_rc(**kw):
    lib = ssm.load_library()
    args = dict(x=None, dt=None, A=None, B=None, C=None, D=None, z=None, bias=None, sp=1, y=None,
                last=None, batch=1, L=64, d_inner=128, heads=2, d_state=64, io=1, ws=None, ws_bytes=0,
                stream=None)
    args.update(kw)
    return lib.ssm_ssd_fwd(*args.values())


def test_ssd_host_validation_before_any_device_call():
    assert _ssd_rc(io=0) == 3                      # bf16 only
    assert _ssd_rc(d_state=48) == 2                # d_state in {16, 32, 64, 128}
    assert _ssd_rc(d_state=256) == 2
    assert _ssd_rc(d_inner=192) == 2               # head dimension 64: d_inner == 64 * heads
    assert _ssd_rc(heads=0) == 2
    assert _ssd_rc(L=-1) == 2
    assert _ssd_rc(batch=0) == 0                   # empty problem
    assert _ssd_rc() == 1                          # A missing
    assert ssm.ssm_ssd_fwd_workspace_size(2, 64, 128, 2, 64) == (
        256 + 2 * 1 * 64 * 64 * 4 + 256 + 2 * 128 * 64 * 4)  # status, Gram, flags, hand-over


def _bwd_rc(**kw):
    lib = ssm.load_library()
    args = dict(u=None, delta=None, A=None, B=None, C=None, D=None, z=None, bias=None, sp=1, h0=None,
                dy=None, dlast=None, du=None, ddelta=None, dA=None, dB=None, dC=None, dD=None, dz=None,
                dbias=None, dinit=None, batch=1, L=8, d_inner=8, d_state=4, io=0, ws=None, ws_bytes=0,
                stream=None)
    args.update(kw)
    return lib.ssm_scan_bwd(*args.values())


def test_backward_host_validation_before_any_device_call():
    assert _bwd_rc(io=5) == 3
    assert _bwd_rc(d_state=17) == 2
    assert _bwd_rc(d_inner=6) == 2
    assert _bwd_rc(batch=0) == 0
    assert _bwd_rc() == 1                          # A and dA missing
    # D given without dD (and z without dz): every gradient of a given operand must be asked for
    import ctypes
    one = ctypes.c_void_p(16)
    assert _bwd_rc(A=one, dA=one, u=one, delta=one, B=one, C=one, dy=one, du=one, ddelta=one, dB=one,
                   dC=one, D=one) == 1
    assert _bwd_rc(A=one, dA=one, u=one, delta=one, B=one, C=one, dy=one, du=one, ddelta=one, dB=one,
                   dC=one, z=one) == 1


def test_product_path_does_not_import_oracle():
    """The package never imports, links or loads the oracle (test infrastructure)."""
    src_dir = os.path.join(ROOT, "selective_state_space_161_b300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "liboracle" not in text, f


def _ssd_rc(**kw):
    lib = ssm.load_library()
    args = dict(x=None, dt=None, A=None, B=None, C=None, D=None, z=None, bias=None, sp=1, y=None,
                last=None, batch=1, L=64, d_inner=128, heads=2, d_state=64, io=1, ws=None, ws_bytes=0,
                stream=None)
    args.update(kw)
    return lib.ssm_ssd_fwd(*args.values())


def test_ssd_host_validation_before_any_device_call():
    assert _ssd_rc(io=0) == 3                      # the chunked form is bf16 only
    assert _ssd_rc(d_state=48) == 2                # d_state in {16, 32, 64, 128}
    assert _ssd_rc(d_state=256) == 2
    assert _ssd_rc(d_inner=96) == 2                # head dimension is 64
    assert _ssd_rc(heads=0) == 2
    assert _ssd_rc(L=-1) == 2
    assert _ssd_rc(batch=0) == 0                   # empty problem
    assert _ssd_rc() == 1                          # A (and the tensors) missing
    # the chunk Gram matrices C B^T, shared by every head: 8 x 32 chunks x 64 x 64 fp32
    # status word, Gram matrices, one flag per (batch, head) in whole 256-byte blocks, and the
    # state handed from the first time half to the second
    assert ssm.ssm_ssd_fwd_workspace_size(8, 2048, 5120, 80, 128) == (
        256 + 8 * 32 * 64 * 64 * 4 + 5120 + 8 * 5120 * 128 * 4)
    assert ssm.ssm_ssd_fwd_workspace_size(8, 0, 5120, 80, 128) == 0
