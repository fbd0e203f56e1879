"""Seeded synthetic inputs for the selective-scan workloads.

This package is shared by the tests (which feed the oracle) and the benchmark
(which feeds the CUDA library).  It holds none of the selective-scan
arithmetic: it only draws numbers.  Values are bit-identical whether drawn on
the host (``libssm_inputgen_host.so``, plain C) or filled on the GPU
(``libssm_inputgen_cuda.so``), so the oracle can check any sampled element of a
tensor that was generated on the device.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_HOST_SRC = [os.path.join(_CSRC, "gen_host.c"), os.path.join(_CSRC, "gen_core.h")]
_DEV_SRC = [os.path.join(_CSRC, "gen_fill.cu"), os.path.join(_CSRC, "gen_core.h")]
_HOST_LIB = os.path.join(_HERE, "libssm_inputgen_host.so")
_DEV_LIB = os.path.join(_HERE, "libssm_inputgen_cuda.so")
_host = None
_dev = None

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _stale(lib, srcs):
    return not os.path.exists(lib) or any(os.path.getmtime(lib) < os.path.getmtime(s) for s in srcs)


def build(force: bool = False, device: bool = True) -> None:
    """Compile the host generator (gcc) and, if requested, the device fill (nvcc)."""
    if force or _stale(_HOST_LIB, _HOST_SRC):
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                        "-o", _HOST_LIB + ".tmp", _HOST_SRC[0], "-lm"], check=True)
        os.replace(_HOST_LIB + ".tmp", _HOST_LIB)
    if device and (force or _stale(_DEV_LIB, _DEV_SRC)):
        subprocess.run([NVCC, "-O3", "--fmad=false", "-shared", "-Xcompiler", "-fPIC",
                        "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
                        "-o", _DEV_LIB + ".tmp", _DEV_SRC[0]], check=True)
        os.replace(_DEV_LIB + ".tmp", _DEV_LIB)


def _host_lib():
    global _host
    if _host is None:
        build(device=False)
        lib = ctypes.CDLL(_HOST_LIB)
        u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.gen_normal_f32.argtypes = [u64, u64, f64, f64, i64, i64, vp]
        lib.gen_normal_bf16.argtypes = [u64, u64, f64, f64, i64, i64, vp]
        lib.gen_normal_f32_at.argtypes = [u64, u64, f64, f64, vp, i64, vp]
        lib.gen_normal_bf16_at.argtypes = [u64, u64, f64, f64, vp, i64, vp]
        lib.gen_uniform_f64.argtypes = [u64, u64, i64, i64, vp]
        lib.gen_delta_bias_f32.argtypes = [u64, u64, f64, f64, i64, vp]
        lib.gen_bf16_to_f32.argtypes = [vp, i64, vp]
        for f in (lib.gen_normal_f32, lib.gen_normal_bf16, lib.gen_normal_f32_at,
                  lib.gen_normal_bf16_at, lib.gen_uniform_f64, lib.gen_delta_bias_f32,
                  lib.gen_bf16_to_f32):
            f.restype = None
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        build(device=True)
        lib = ctypes.CDLL(_DEV_LIB)
        lib.gen_dev_fill_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                            ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.gen_dev_fill_normal.restype = ctypes.c_int
        _dev = lib
    return _dev


def normal(seed: int, tensor_id: int, mean: float, sd: float, start: int, count: int,
           bf16: bool) -> np.ndarray:
    """Draws for flat indices [start, start+count): float32, or uint16 bfloat16 bits."""
    out = np.empty(count, dtype=np.uint16 if bf16 else np.float32)
    f = _host_lib().gen_normal_bf16 if bf16 else _host_lib().gen_normal_f32
    f(seed, tensor_id, mean, sd, start, count, out.ctypes.data)
    return out


def normal_at(seed: int, tensor_id: int, mean: float, sd: float, idx: np.ndarray,
              bf16: bool) -> np.ndarray:
    """Draws at the given flat indices (same values as the full tensor holds there)."""
    idx = np.ascontiguousarray(idx, dtype=np.int64).ravel()
    out = np.empty(idx.size, dtype=np.uint16 if bf16 else np.float32)
    f = _host_lib().gen_normal_bf16_at if bf16 else _host_lib().gen_normal_f32_at
    f(seed, tensor_id, mean, sd, idx.ctypes.data, idx.size, out.ctypes.data)
    return out


def uniform(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float64)
    _host_lib().gen_uniform_f64(seed, tensor_id, start, count, out.ctypes.data)
    return out


def delta_bias(seed: int, tensor_id: int, dt_min: float, dt_max: float, count: int) -> np.ndarray:
    """fp32 biases whose softplus is log-uniform on [dt_min, dt_max]."""
    out = np.empty(count, dtype=np.float32)
    _host_lib().gen_delta_bias_f32(seed, tensor_id, dt_min, dt_max, count, out.ctypes.data)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).reshape(bits.shape)


def dev_fill_normal(seed: int, tensor_id: int, mean: float, sd: float, start: int, count: int,
                    bf16: bool, dev_ptr: int, stream: int = 0) -> None:
    """Fill a device buffer (raw pointer) with the same draws ``normal`` returns."""
    rc = _dev_lib().gen_dev_fill_normal(seed, tensor_id, mean, sd, start, count, int(bf16),
                                        ctypes.c_void_p(dev_ptr), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"gen_dev_fill_normal failed ({rc})")
