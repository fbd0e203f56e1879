"""Float64 reference ("oracle") for the selective scan and its decode step.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path never
does.  The arithmetic lives in ``ssm_oracle.c`` (plain C, double precision,
sequential per channel, OpenMP across channels); this module only compiles it
and marshals numpy arrays.  See the header of ``ssm_oracle.c`` for the
equations and the pages they come from.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_scan_fwd.argtypes = [dp] * 8 + [ctypes.c_int, dp, dp, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_scan_fwd.restype = ctypes.c_int
        lib.oracle_scan_fwd_from_state.argtypes = ([dp] * 8 + [ctypes.c_int, dp, dp, dp, i64, i64,
                                                               i64, i64, ctypes.c_int])
        lib.oracle_scan_fwd_from_state.restype = ctypes.c_int
        lib.oracle_scan_bwd.argtypes = [dp] * 8 + [ctypes.c_int] + [dp] * 12 + [i64, i64, i64, i64]
        lib.oracle_scan_bwd.restype = ctypes.c_int
        lib.oracle_conv1d_silu.argtypes = [dp] * 5 + [i64, i64, i64, i64]
        lib.oracle_conv1d_silu.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = [dp] * 10 + [ctypes.c_int, i64, i64, i64, ctypes.c_int]
        lib.oracle_state_update.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def softplus(x: float) -> float:
    return float(_load().oracle_softplus(float(x)))


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus_flag=True,
             nthreads: int | None = None, initial_state=None):
    """y [batch, L, d_inner] and last_state [batch, d_inner, d_state], both float64.

    u, delta, z: [batch, L, d_inner]; B, C: [batch, L, d_state];
    A: [d_inner, d_state]; D, delta_bias: [d_inner] (None = absent);
    initial_state: [batch, d_inner, d_state] (None = start from zero).
    """
    u, delta, A, B, C, D, z, delta_bias = map(_f64, (u, delta, A, B, C, D, z, delta_bias))
    initial_state = _f64(initial_state)
    batch, L, d_inner = u.shape
    d_state = A.shape[1]
    assert A.shape == (d_inner, d_state)
    assert B.shape == (batch, L, d_state) and C.shape == (batch, L, d_state)
    assert delta.shape == u.shape and (z is None or z.shape == u.shape)
    for t in (u, delta, A, B, C, D, z, delta_bias):
        assert t is None or np.all(np.isfinite(t)), "oracle inputs must be finite"
    assert initial_state is None or initial_state.shape == (batch, d_inner, d_state)
    y = np.zeros((batch, L, d_inner), dtype=np.float64)
    last = np.zeros((batch, d_inner, d_state), dtype=np.float64)
    if initial_state is None:
        rc = _load().oracle_scan_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(z), _ptr(delta_bias), int(bool(softplus_flag)), _ptr(y),
                                     _ptr(last), batch, L, d_inner, d_state,
                                     int(nthreads or max_threads()))
    else:
        rc = _load().oracle_scan_fwd_from_state(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                                _ptr(D), _ptr(z), _ptr(delta_bias),
                                                int(bool(softplus_flag)), _ptr(initial_state),
                                                _ptr(y), _ptr(last), batch, L, d_inner, d_state,
                                                int(nthreads or max_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_scan_fwd failed ({rc})")
    return y, last


def scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus_flag=True,
             initial_state=None, dlast=None):
    """Gradients of scan_fwd for given dL/dy (and dL/dlast_state).  Returns a dict with
    du, ddelta, dA, dB, dC, and dD / dz / ddelta_bias / dinitial_state where those operands
    exist, all float64."""
    u, delta, A, B, C, D, z, delta_bias, initial_state, dy, dlast = map(
        _f64, (u, delta, A, B, C, D, z, delta_bias, initial_state, dy, dlast))
    batch, L, d_inner = u.shape
    d_state = A.shape[1]
    out = dict(du=np.zeros_like(u), ddelta=np.zeros_like(u), dA=np.zeros_like(A),
               dB=np.zeros_like(B), dC=np.zeros_like(C))
    out["dD"] = np.zeros(d_inner) if D is not None else None
    out["dz"] = np.zeros_like(u) if z is not None else None
    out["ddelta_bias"] = np.zeros(d_inner) if delta_bias is not None else None
    out["dinitial_state"] = np.zeros((batch, d_inner, d_state))
    rc = _load().oracle_scan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                 _ptr(delta_bias), int(bool(softplus_flag)), _ptr(initial_state),
                                 _ptr(dy), _ptr(dlast), _ptr(out["du"]), _ptr(out["ddelta"]),
                                 _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                                 _ptr(out["dz"]), _ptr(out["ddelta_bias"]),
                                 _ptr(out["dinitial_state"]), batch, L, d_inner, d_state)
    if rc != 0:
        raise RuntimeError(f"oracle_scan_bwd failed ({rc})")
    return {k: v for k, v in out.items() if v is not None}


def conv1d_silu(x, w, bias=None, x_prev=None):
    """silu(causal depthwise conv1d(x)) [batch, L, d_inner], float64.

    x: [batch, L, d_inner]; w: [d_inner, d_conv]; bias: [d_inner] or None;
    x_prev: [batch, d_inner, d_conv - 1], the inputs before t = 0 (None = zeros)."""
    x, w, bias, x_prev = map(_f64, (x, w, bias, x_prev))
    batch, L, d_inner = x.shape
    d_conv = w.shape[1]
    assert w.shape == (d_inner, d_conv)
    assert x_prev is None or x_prev.shape == (batch, d_inner, d_conv - 1)
    u = np.zeros_like(x)
    rc = _load().oracle_conv1d_silu(_ptr(x), _ptr(w), _ptr(bias), _ptr(x_prev), _ptr(u), batch, L,
                                    d_inner, d_conv)
    if rc != 0:
        raise RuntimeError(f"oracle_conv1d_silu failed ({rc})")
    return u


def state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus_flag=True,
                 nthreads: int | None = None):
    """One decode step.  Returns (y [batch, d_inner], new_state [batch, d_inner, d_state])."""
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    u, delta, A, B, C, D, z, delta_bias = map(_f64, (u, delta, A, B, C, D, z, delta_bias))
    batch, d_inner = u.shape
    d_state = A.shape[1]
    assert st.shape == (batch, d_inner, d_state) and B.shape == (batch, d_state)
    y = np.zeros((batch, d_inner), dtype=np.float64)
    rc = _load().oracle_state_update(_ptr(st), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                     _ptr(D), _ptr(z), _ptr(y), _ptr(delta_bias),
                                     int(bool(softplus_flag)), batch, d_inner, d_state,
                                     int(nthreads or max_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_state_update failed ({rc})")
    return y, st
