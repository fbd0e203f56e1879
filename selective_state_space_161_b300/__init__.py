"""Python binding of libssm, the B300 (sm_103a) selective-scan library.

The functions named like the C ABI (``ssm_scan_fwd``, ``ssm_state_update``,
``ssm_scan_fwd_workspace_size``, ``ssm_status_string``) only marshal
arguments: every step of the computation runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.  There is no fallback: if the
compiled library is missing or cannot be loaded, every call raises.

``selective_scan`` is the convenience entry a user calls: it allocates the
outputs and the scratch workspace with PyTorch and accepts either CUDA tensors
or host tensors (which it copies to the current device and back).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH, build

__all__ = ["SsmError", "ssm_scan_fwd", "ssm_scan_fwd_from_state", "ssm_scan_fwd_conv",
           "ssm_scan_fwd_noalloc", "ssm_state_update", "ssm_state_update_conv", "ssm_scan_bwd",
           "ssm_scan_bwd_workspace_size", "ssm_scan_bwd_launches", "selective_scan_backward", "ssm_ssd_fwd",
           "ssm_ssd_fwd_workspace_size", "selective_scan_ssd",
           "ssm_scan_fwd_workspace_size", "ssm_get_status",
           "ssm_status_string", "ssm_version", "selective_scan", "selective_state_update",
           "load_library", "build", "SSM_F32", "SSM_BF16", "EXPORTED_SYMBOLS"]

SSM_F32, SSM_BF16 = 0, 1
EXPORTED_SYMBOLS = ("ssm_scan_fwd_workspace_size", "ssm_scan_fwd", "ssm_scan_fwd_from_state",
                    "ssm_scan_fwd_conv", "ssm_scan_fwd_noalloc", "ssm_state_update",
                    "ssm_state_update_conv", "ssm_scan_bwd", "ssm_scan_bwd_workspace_size",
                    "ssm_scan_bwd_launches",
                    "ssm_ssd_fwd", "ssm_ssd_fwd_workspace_size", "ssm_get_status",
                    "ssm_status_string", "ssm_version")
SSM_ERR_LOOKBACK_TIMEOUT, SSM_ERR_SCRATCH_LIMIT = 7, 8
SSM_NOALLOC_SCRATCH_BYTES = 8 << 20

_lib = None


class SsmError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: status {status} ({ssm_status_string(status)})")


def load_library() -> ctypes.CDLL:
    """Load the compiled library (building it first if the sources are newer)."""
    global _lib
    if _lib is None:
        path = build()
        if not os.path.exists(path):
            raise RuntimeError(f"libssm not found at {path}")
        lib = ctypes.CDLL(path)
        vp, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.ssm_scan_fwd_workspace_size.argtypes = [i64, i64, i64, c_int, c_int]
        lib.ssm_scan_fwd_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_fwd.argtypes = [vp] * 8 + [c_int, vp, vp, i64, i64, i64, c_int, c_int, vp,
                                              ctypes.c_size_t, vp]
        lib.ssm_scan_fwd.restype = c_int
        lib.ssm_scan_fwd_from_state.argtypes = [vp] * 8 + [c_int, vp, vp, vp, i64, i64, i64, c_int,
                                                          c_int, vp, ctypes.c_size_t, vp]
        lib.ssm_scan_fwd_from_state.restype = c_int
        lib.ssm_scan_fwd_conv.argtypes = ([vp, vp, vp, c_int] + [vp] * 7 + [c_int, vp, vp, vp, vp, i64,
                                                                         i64, i64, c_int, c_int, vp,
                                                                         ctypes.c_size_t, vp])
        lib.ssm_scan_fwd_conv.restype = c_int
        lib.ssm_state_update_conv.argtypes = ([vp] * 5 + [c_int] + [vp] * 8 + [c_int, i64, i64, c_int,
                                                                              c_int, vp])
        lib.ssm_state_update_conv.restype = c_int
        lib.ssm_scan_bwd_workspace_size.argtypes = [i64, i64, i64, c_int, c_int]
        lib.ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_bwd_launches.argtypes = [i64, i64, i64, c_int, c_int]
        lib.ssm_scan_bwd_launches.restype = c_int
        lib.ssm_scan_bwd.argtypes = [vp] * 8 + [c_int] + [vp] * 12 + [i64, i64, i64, c_int, c_int, vp,
                                                                   ctypes.c_size_t, vp]
        lib.ssm_scan_bwd.restype = c_int
        lib.ssm_ssd_fwd_workspace_size.argtypes = [i64, i64, i64, c_int, c_int]
        lib.ssm_ssd_fwd_workspace_size.restype = ctypes.c_size_t
        lib.ssm_ssd_fwd.argtypes = [vp] * 8 + [c_int, vp, vp, i64, i64, i64, c_int, c_int, c_int, vp,
                                              ctypes.c_size_t, vp]
        lib.ssm_ssd_fwd.restype = c_int
        lib.ssm_scan_fwd_noalloc.argtypes = [vp] * 8 + [c_int, vp, vp, i64, i64, i64, c_int, c_int,
                                                       vp]
        lib.ssm_scan_fwd_noalloc.restype = c_int
        lib.ssm_state_update.argtypes = [vp] * 10 + [c_int, i64, i64, c_int, c_int, vp]
        lib.ssm_state_update.restype = c_int
        lib.ssm_get_status.argtypes = [vp, vp]
        lib.ssm_get_status.restype = c_int
        lib.ssm_status_string.argtypes = [c_int]
        lib.ssm_status_string.restype = ctypes.c_char_p
        lib.ssm_version.restype = c_int
        _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _io_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"I/O tensors must be float32 or bfloat16, got {t.dtype}")


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_dev(name, t, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def ssm_status_string(status: int) -> str:
    return load_library().ssm_status_string(int(status)).decode()


def ssm_version() -> int:
    return int(load_library().ssm_version())


def ssm_scan_fwd_workspace_size(batch: int, L: int, d_inner: int, d_state: int, io: int) -> int:
    return int(load_library().ssm_scan_fwd_workspace_size(batch, L, d_inner, d_state, io))


def ssm_get_status(workspace=None, stream=None) -> int:
    """C-ABI ``ssm_get_status``: waits for ``stream`` and returns the device-side status of the
    latest forward scan, backward pass or chunked SSD call that used ``workspace`` (None: the
    no-allocation entry point's scratch): 0 (SSM_OK), SSM_ERR_LOOKBACK_TIMEOUT or SSM_ERR_CUDA."""
    _check_dev("workspace", workspace)
    return int(load_library().ssm_get_status(_ptr(workspace), _stream_handle(stream)))


def ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                 workspace=None, stream=None) -> None:
    """C-ABI ``ssm_scan_fwd`` on CUDA tensors (shapes as documented in include/ssm.h)."""
    _scan_call("ssm_scan_fwd", u, delta, A, B, C, D, z, delta_bias, softplus_flag, None, y,
               last_state, workspace, stream)


def ssm_scan_fwd_from_state(u, delta, A, B, C, D, z, delta_bias, softplus_flag, initial_state, y,
                            last_state, workspace=None, stream=None) -> None:
    """C-ABI ``ssm_scan_fwd_from_state``: the scan continuing from ``initial_state``."""
    _scan_call("ssm_scan_fwd_from_state", u, delta, A, B, C, D, z, delta_bias, softplus_flag,
               initial_state, y, last_state, workspace, stream)


def ssm_scan_fwd_conv(x, conv_weight, conv_bias, delta, A, B, C, D, z, delta_bias,
                      softplus_flag, initial_state, y, last_state, u_out=None, workspace=None,
                      stream=None) -> None:
    """C-ABI ``ssm_scan_fwd_conv``: u = silu(causal depthwise conv1d(x)) fused in front of the
    scan; ``conv_weight`` is [d_inner, d_conv] (d_conv <= 4), ``u_out`` optionally receives u."""
    _scan_call("ssm_scan_fwd_conv", x, delta, A, B, C, D, z, delta_bias, softplus_flag,
               initial_state, y, last_state, workspace, stream,
               conv=(conv_weight, conv_bias, u_out))


def _scan_call(func, u, delta, A, B, C, D, z, delta_bias, softplus_flag, initial_state, y,
               last_state, workspace, stream, conv=None):
    batch, L, d_inner = u.shape
    d_state = A.shape[1]
    io = _io_code(u)
    dt = u.dtype
    for name, t, shp in (("u", u, (batch, L, d_inner)), ("delta", delta, (batch, L, d_inner)),
                         ("z", z, (batch, L, d_inner)), ("y", y, (batch, L, d_inner)),
                         ("B", B, (batch, L, d_state)), ("C", C, (batch, L, d_state))):
        _check_dev(name, t, dt, shp)
    _check_dev("A", A, torch.float32, (d_inner, d_state))
    _check_dev("D", D, torch.float32, (d_inner,))
    _check_dev("delta_bias", delta_bias, torch.float32, (d_inner,))
    _check_dev("last_state", last_state, torch.float32, (batch, d_inner, d_state))
    _check_dev("initial_state", initial_state, torch.float32, (batch, d_inner, d_state))
    _check_dev("workspace", workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load_library()
    head = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(softplus_flag)))
    tail = (_ptr(y), _ptr(last_state), batch, L, d_inner, d_state, io, _ptr(workspace), ws_bytes,
            _stream_handle(stream))
    if func == "ssm_scan_fwd":
        rc = lib.ssm_scan_fwd(*head, *tail)
    elif func == "ssm_scan_fwd_from_state":
        rc = lib.ssm_scan_fwd_from_state(*head, _ptr(initial_state), *tail)
    else:
        cw, cb, u_out = conv
        _check_dev("conv_weight", cw, torch.float32)
        if cw.dim() != 2 or cw.shape[0] != d_inner:
            raise ValueError("conv_weight must be [d_inner, d_conv]")
        _check_dev("conv_bias", cb, torch.float32, (d_inner,))
        _check_dev("u_out", u_out, u.dtype, (batch, L, d_inner))
        rc = lib.ssm_scan_fwd_conv(_ptr(u), _ptr(cw), _ptr(cb), int(cw.shape[1]), *head[1:],
                                   _ptr(initial_state), _ptr(y), _ptr(last_state), _ptr(u_out),
                                   *tail[2:])
    if rc != 0:
        raise SsmError(func, rc)


def ssm_scan_fwd_noalloc(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                         stream=None) -> None:
    """C-ABI ``ssm_scan_fwd_noalloc``: ``ssm_scan_fwd`` with the library's own fixed scratch
    instead of a caller workspace, for callers that cannot allocate device memory where they
    call it.  Calls that overlap on the GPU share that scratch and must be serialised."""
    batch, L, d_inner = u.shape
    d_state = A.shape[1]
    io = _io_code(u)
    dt = u.dtype
    for name, t, shp in (("u", u, (batch, L, d_inner)), ("delta", delta, (batch, L, d_inner)),
                         ("z", z, (batch, L, d_inner)), ("y", y, (batch, L, d_inner)),
                         ("B", B, (batch, L, d_state)), ("C", C, (batch, L, d_state))):
        _check_dev(name, t, dt, shp)
    _check_dev("A", A, torch.float32, (d_inner, d_state))
    _check_dev("D", D, torch.float32, (d_inner,))
    _check_dev("delta_bias", delta_bias, torch.float32, (d_inner,))
    _check_dev("last_state", last_state, torch.float32, (batch, d_inner, d_state))
    rc = load_library().ssm_scan_fwd_noalloc(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                             _ptr(D), _ptr(z), _ptr(delta_bias),
                                             int(bool(softplus_flag)), _ptr(y), _ptr(last_state),
                                             batch, L, d_inner, d_state, io,
                                             _stream_handle(stream))
    if rc != 0:
        raise SsmError("ssm_scan_fwd_noalloc", rc)


def ssm_scan_bwd_workspace_size(batch: int, L: int, d_inner: int, d_state: int, io: int) -> int:
    return int(load_library().ssm_scan_bwd_workspace_size(batch, L, d_inner, d_state, io))


def ssm_scan_bwd_launches(batch: int, L: int, d_inner: int, d_state: int, io: int) -> int:
    return int(load_library().ssm_scan_bwd_launches(batch, L, d_inner, d_state, io))


def ssm_scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, initial_state, dy,
                 dlast_state, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, dinitial_state,
                 workspace, stream=None) -> None:
    """C-ABI ``ssm_scan_bwd`` on CUDA tensors (shapes as documented in include/ssm.h)."""
    batch, L, d_inner = u.shape
    d_state = A.shape[1]
    io = _io_code(u)
    dt = u.dtype
    for name, t, shp, ty in (("u", u, (batch, L, d_inner), dt), ("delta", delta, (batch, L, d_inner), dt),
                             ("z", z, (batch, L, d_inner), dt), ("dy", dy, (batch, L, d_inner), dt),
                             ("du", du, (batch, L, d_inner), dt), ("ddelta", ddelta, (batch, L, d_inner), dt),
                             ("dz", dz, (batch, L, d_inner), dt), ("B", B, (batch, L, d_state), dt),
                             ("C", C, (batch, L, d_state), dt),
                             ("dB", dB, (batch, L, d_state), torch.float32),
                             ("dC", dC, (batch, L, d_state), torch.float32),
                             ("A", A, (d_inner, d_state), torch.float32),
                             ("dA", dA, (d_inner, d_state), torch.float32),
                             ("D", D, (d_inner,), torch.float32), ("dD", dD, (d_inner,), torch.float32),
                             ("delta_bias", delta_bias, (d_inner,), torch.float32),
                             ("ddelta_bias", ddelta_bias, (d_inner,), torch.float32),
                             ("initial_state", initial_state, (batch, d_inner, d_state), torch.float32),
                             ("dlast_state", dlast_state, (batch, d_inner, d_state), torch.float32),
                             ("dinitial_state", dinitial_state, (batch, d_inner, d_state), torch.float32)):
        _check_dev(name, t, ty, shp)
    _check_dev("workspace", workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().ssm_scan_bwd(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        int(bool(softplus_flag)), _ptr(initial_state), _ptr(dy), _ptr(dlast_state), _ptr(du),
        _ptr(ddelta), _ptr(dA), _ptr(dB), _ptr(dC), _ptr(dD), _ptr(dz), _ptr(ddelta_bias),
        _ptr(dinitial_state), batch, L, d_inner, d_state, io, _ptr(workspace), ws_bytes,
        _stream_handle(stream))
    if rc != 0:
        raise SsmError("ssm_scan_bwd", rc)


def selective_scan_backward(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=True,
                            initial_state=None, dlast_state=None, stream=None):
    """Gradients of ``selective_scan`` (CUDA tensors).  Returns a dict with du, ddelta, dA, dB,
    dC and, where those inputs were given, dD, dz, ddelta_bias, dinitial_state."""
    batch, L, d_inner = u.shape
    d_state = A.shape[1]
    dev = u.device
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(du=torch.empty_like(u), ddelta=torch.empty_like(u), dA=torch.empty((d_inner, d_state), **f32),
             dB=torch.empty((batch, L, d_state), **f32), dC=torch.empty((batch, L, d_state), **f32))
    g["dD"] = torch.empty(d_inner, **f32) if D is not None else None
    g["dz"] = torch.empty_like(u) if z is not None else None
    g["ddelta_bias"] = torch.empty(d_inner, **f32) if delta_bias is not None else None
    g["dinitial_state"] = torch.empty((batch, d_inner, d_state), **f32)
    nbytes = ssm_scan_bwd_workspace_size(batch, L, d_inner, d_state, _io_code(u))
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    ssm_scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, initial_state, dy, dlast_state,
                 g["du"], g["ddelta"], g["dA"], g["dB"], g["dC"], g["dD"], g["dz"], g["ddelta_bias"],
                 g["dinitial_state"], ws, stream)
    return {k: v for k, v in g.items() if v is not None}


def ssm_ssd_fwd_workspace_size(batch: int, L: int, d_inner: int, n_heads: int, d_state: int) -> int:
    return int(load_library().ssm_ssd_fwd_workspace_size(batch, L, d_inner, n_heads, d_state))


def ssm_ssd_fwd(x, dt, A_head, B, C, D, z, dt_bias, softplus_flag, y, last_state, workspace,
                stream=None) -> None:
    """C-ABI ``ssm_ssd_fwd``: the chunked tensor-core form for one A and one step size per head
    (bf16 I/O, heads of 64 channels; see include/ssm.h)."""
    batch, L, d_inner = x.shape
    n_heads = dt.shape[2]
    d_state = B.shape[2]
    bf = torch.bfloat16
    for name, t, shp, ty in (("x", x, (batch, L, d_inner), bf), ("z", z, (batch, L, d_inner), bf),
                             ("y", y, (batch, L, d_inner), bf), ("dt", dt, (batch, L, n_heads), bf),
                             ("B", B, (batch, L, d_state), bf), ("C", C, (batch, L, d_state), bf),
                             ("A_head", A_head, (n_heads,), torch.float32),
                             ("dt_bias", dt_bias, (n_heads,), torch.float32),
                             ("D", D, (d_inner,), torch.float32),
                             ("last_state", last_state, (batch, d_inner, d_state), torch.float32)):
        _check_dev(name, t, ty, shp)
    _check_dev("workspace", workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().ssm_ssd_fwd(_ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D),
                                    _ptr(z), _ptr(dt_bias), int(bool(softplus_flag)), _ptr(y),
                                    _ptr(last_state), batch, L, d_inner, n_heads, d_state, SSM_BF16,
                                    _ptr(workspace), ws_bytes, _stream_handle(stream))
    if rc != 0:
        raise SsmError("ssm_ssd_fwd", rc)


def selective_scan_ssd(x, dt, A_head, B, C, D=None, z=None, dt_bias=None, softplus=True,
                       stream=None):
    """Chunked SSD scan on CUDA bf16 tensors; returns (y, last_state)."""
    batch, L, d_inner = x.shape
    d_state = B.shape[2]
    y = torch.empty_like(x)
    last = torch.empty((batch, d_inner, d_state), dtype=torch.float32, device=x.device)
    nbytes = ssm_ssd_fwd_workspace_size(batch, L, d_inner, dt.shape[2], d_state)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device) if nbytes else None
    ssm_ssd_fwd(x, dt, A_head, B, C, D, z, dt_bias, softplus, y, last, ws, stream)
    return y, last


def ssm_state_update_conv(state, conv_state, x, conv_weight, conv_bias, delta, A, B, C, D, z, y,
                          delta_bias, softplus_flag, stream=None) -> None:
    """C-ABI ``ssm_state_update_conv``: one decode step with conv1d + SiLU in front;
    ``conv_state`` [batch, d_inner, d_conv - 1] fp32 is shifted in place."""
    batch, d_inner = x.shape
    d_state = A.shape[1]
    io = _io_code(x)
    _check_dev("state", state, torch.float32, (batch, d_inner, d_state))
    _check_dev("conv_weight", conv_weight, torch.float32)
    d_conv = int(conv_weight.shape[1])
    _check_dev("conv_state", conv_state, torch.float32, (batch, d_inner, d_conv - 1))
    _check_dev("conv_bias", conv_bias, torch.float32, (d_inner,))
    for name, t, shp in (("x", x, (batch, d_inner)), ("delta", delta, (batch, d_inner)),
                         ("z", z, (batch, d_inner)), ("y", y, (batch, d_inner)),
                         ("B", B, (batch, d_state)), ("C", C, (batch, d_state))):
        _check_dev(name, t, x.dtype, shp)
    _check_dev("A", A, torch.float32, (d_inner, d_state))
    _check_dev("D", D, torch.float32, (d_inner,))
    _check_dev("delta_bias", delta_bias, torch.float32, (d_inner,))
    rc = load_library().ssm_state_update_conv(
        _ptr(state), _ptr(conv_state) if d_conv > 1 else None, _ptr(x), _ptr(conv_weight),
        _ptr(conv_bias), d_conv, _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(y),
        _ptr(delta_bias), int(bool(softplus_flag)), batch, d_inner, d_state, io,
        _stream_handle(stream))
    if rc != 0:
        raise SsmError("ssm_state_update_conv", rc)


def ssm_state_update(state, u, delta, A, B, C, D, z, y, delta_bias, softplus_flag,
                     stream=None) -> None:
    """C-ABI ``ssm_state_update`` on CUDA tensors; ``state`` is updated in place."""
    batch, d_inner = u.shape
    d_state = A.shape[1]
    io = _io_code(u)
    dt = u.dtype
    _check_dev("state", state, torch.float32, (batch, d_inner, d_state))
    for name, t, shp in (("u", u, (batch, d_inner)), ("delta", delta, (batch, d_inner)),
                         ("z", z, (batch, d_inner)), ("y", y, (batch, d_inner)),
                         ("B", B, (batch, d_state)), ("C", C, (batch, d_state))):
        _check_dev(name, t, dt, shp)
    _check_dev("A", A, torch.float32, (d_inner, d_state))
    _check_dev("D", D, torch.float32, (d_inner,))
    _check_dev("delta_bias", delta_bias, torch.float32, (d_inner,))
    rc = load_library().ssm_state_update(_ptr(state), _ptr(u), _ptr(delta), _ptr(A), _ptr(B),
                                         _ptr(C), _ptr(D), _ptr(z), _ptr(y), _ptr(delta_bias),
                                         int(bool(softplus_flag)), batch, d_inner, d_state, io,
                                         _stream_handle(stream))
    if rc != 0:
        raise SsmError("ssm_state_update", rc)


def _to_device(t, device):
    if t is None:
        return None
    return t if t.is_cuda else t.to(device, non_blocking=True)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                   return_last_state=True, stream=None, initial_state=None, conv_weight=None,
                   conv_bias=None):
    """Selective scan forward.  Returns (y, last_state) on the inputs' device.

    ``initial_state`` [batch, d_inner, d_state] continues from a saved state (None: zero).
    With ``conv_weight`` [d_inner, d_conv] the first operand is the block input x and
    u = silu(causal depthwise conv1d(x) + conv_bias) is computed inside the scan.
    Host tensors (pinned for asynchronous copies) are copied to the current
    CUDA device, processed there, and the results copied back."""
    on_host = not u.is_cuda
    device = torch.device("cuda", torch.cuda.current_device()) if on_host else u.device
    ins = [_to_device(t, device) for t in (u, delta, A, B, C, D, z, delta_bias, initial_state,
                                            conv_weight, conv_bias)]
    u_d, delta_d, A_d, B_d, C_d, D_d, z_d, bias_d, h0_d, cw_d, cb_d = ins
    batch, L, d_inner = u_d.shape
    d_state = A_d.shape[1]
    y = torch.empty_like(u_d)
    last = (torch.empty((batch, d_inner, d_state), dtype=torch.float32, device=device)
            if return_last_state else None)
    nbytes = ssm_scan_fwd_workspace_size(batch, L, d_inner, d_state, _io_code(u_d))
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device) if nbytes else None
    if cw_d is not None:
        ssm_scan_fwd_conv(u_d, cw_d, cb_d, delta_d, A_d, B_d, C_d, D_d, z_d, bias_d, softplus, h0_d,
                          y, last, None, ws, stream)
    elif h0_d is None:
        ssm_scan_fwd(u_d, delta_d, A_d, B_d, C_d, D_d, z_d, bias_d, softplus, y, last, ws, stream)
    else:
        ssm_scan_fwd_from_state(u_d, delta_d, A_d, B_d, C_d, D_d, z_d, bias_d, softplus, h0_d, y,
                                last, ws, stream)
    if on_host:
        y = y.to("cpu", non_blocking=False)
        last = last.to("cpu") if last is not None else None
    return y, last


def selective_state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                           softplus=True, stream=None):
    """One decode step on CUDA tensors; updates ``state`` in place and returns y."""
    y = torch.empty_like(u)
    ssm_state_update(state, u, delta, A, B, C, D, z, y, delta_bias, softplus, stream)
    return y
