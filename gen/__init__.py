"""Seeded synthetic inputs for the quantized MoE expert layer.

This module is shared by the oracle's tests and by the CUDA path's tests and
benchmark.  It produces the layer's inputs only -- activations x (bf16),
router weights (bf16), router bias (fp32) and the fp32 expert weights before
quantisation -- and holds none of the layer's arithmetic.  Every element is a
pure function of (workload seed, tensor, expert, matrix, index), computed by
the same C header (``moe_gen.h``) on the host and on the device, so a slice
generated on either side is bit-identical.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import WORKLOADS, Workload, get_workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libmoegen_host.so")
DEV_LIB = os.path.join(_HERE, "libmoegen_dev.so")
_lock = threading.Lock()
_host = None
_dev = None

T_X, T_ROUTER, T_WEIGHT, T_ZIPF, T_BIAS = 1, 2, 3, 4, 5
WEIGHT_SIGMA = 0.02
ROUTER_SIGMA = 0.02


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build(device: bool = True) -> None:
    """Compile the host generator (gcc) and, if asked, the device one (nvcc, sm_103a)."""
    hdr = os.path.join(_HERE, "moe_gen.h")
    src = os.path.join(_HERE, "gen_host.c")
    if _stale(HOST_LIB, [hdr, src]):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", src, "-o", HOST_LIB + ".tmp", "-lm"])
        os.replace(HOST_LIB + ".tmp", HOST_LIB)
    if device:
        dsrc = os.path.join(_HERE, "gen_device.cu")
        if _stale(DEV_LIB, [hdr, dsrc]):
            subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                                   "-Xcompiler", "-fPIC", "-shared", dsrc, "-o", DEV_LIB + ".tmp"])
            os.replace(DEV_LIB + ".tmp", DEV_LIB)


def _host_lib():
    global _host
    with _lock:
        if _host is None:
            build(device=False)
            lib = ctypes.CDLL(HOST_LIB)
            lib.moe_gen_stream_key.restype = ctypes.c_uint64
            lib.moe_gen_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                               ctypes.c_uint32]
            for name in ("moe_gen_fill_f32", "moe_gen_fill_bf16"):
                f = getattr(lib, name)
                f.restype = None
                f.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                              ctypes.c_uint64, ctypes.c_int]
            lib.moe_gen_zipf_bias.restype = None
            lib.moe_gen_zipf_bias.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                              ctypes.c_double, ctypes.c_double]
            _host = lib
    return _host


def _dev_lib():
    global _dev
    with _lock:
        if _dev is None:
            if not os.path.exists(DEV_LIB):
                raise RuntimeError("device generator not built: call gen.build(device=True)")
            lib = ctypes.CDLL(DEV_LIB)
            for name in ("moe_gen_fill_f32_dev", "moe_gen_fill_bf16_dev"):
                f = getattr(lib, name)
                f.restype = ctypes.c_int
                f.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                              ctypes.c_uint64, ctypes.c_void_p]
            _dev = lib
    return _dev


def key(seed: int, tensor: int, a: int = 0, b: int = 0) -> int:
    return int(_host_lib().moe_gen_stream_key(seed, tensor, a, b))


def _threads():
    return max(1, min(64, os.cpu_count() or 1))


def normal_f32(k: int, n: int, sigma: float, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _host_lib().moe_gen_fill_f32(out.ctypes.data, n, k, sigma, offset, _threads())
    return out


def normal_bf16(k: int, n: int, sigma: float, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _host_lib().moe_gen_fill_bf16(out.ctypes.data, n, k, sigma, offset, _threads())
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- workload tensors
def matrix_shape(w: Workload, matrix: int):
    """(rows, K) of an expert matrix: 0 gate [I x H], 1 up [I x H], 2 down [H x I]."""
    return (w.I, w.H) if matrix in (0, 1) else (w.H, w.I)


def x_tokens(w: Workload, T: int | None = None, first: int = 0) -> np.ndarray:
    """Activations x[first:first+T] as bf16 bits, shape [T, H]."""
    T = w.T if T is None else T
    flat = normal_bf16(key(w.seed, T_X), T * w.H, 1.0, offset=first * w.H)
    return flat.reshape(T, w.H)


def router_weights(w: Workload) -> np.ndarray:
    """Router weights Wr as bf16 bits, shape [E, H]."""
    return normal_bf16(key(w.seed, T_ROUTER), w.E * w.H, ROUTER_SIGMA).reshape(w.E, w.H)


def router_bias(w: Workload):
    """Router bias as fp32 [E], or None when the workload has none."""
    if w.bias == "none":
        return None
    out = np.empty(w.E, dtype=np.float32)
    if w.bias == "zipf":
        _host_lib().moe_gen_zipf_bias(out.ctypes.data, w.E, key(w.seed, T_ZIPF), w.bias_param,
                                      w.bias_scale)
        return out
    if w.bias == "normal":
        return normal_f32(key(w.seed, T_BIAS), w.E, w.bias_scale)
    raise ValueError(w.bias)


def expert_weight(w: Workload, expert: int, matrix: int) -> np.ndarray:
    """fp32 weights of one expert matrix before quantisation (expert == E: shared expert)."""
    rows, K = matrix_shape(w, matrix)
    return normal_f32(key(w.seed, T_WEIGHT, expert, matrix), rows * K, WEIGHT_SIGMA).reshape(rows, K)


# ---------------------------------------------------------------- device fills
def fill_expert_weight_dev(w: Workload, expert: int, matrix: int, dev_ptr: int, stream: int = 0,
                           seed: int | None = None) -> None:
    """Same values as expert_weight(), written to a device buffer of rows*K fp32."""
    rows, K = matrix_shape(w, matrix)
    s = w.seed if seed is None else seed
    rc = _dev_lib().moe_gen_fill_f32_dev(dev_ptr, rows * K, key(s, T_WEIGHT, expert, matrix),
                                         WEIGHT_SIGMA, 0, stream)
    if rc != 0:
        raise RuntimeError("device generator launch failed")


def fill_normal_dev(k: int, n: int, sigma: float, dev_ptr: int, bf16: bool, stream: int = 0,
                    offset: int = 0) -> None:
    f = _dev_lib().moe_gen_fill_bf16_dev if bf16 else _dev_lib().moe_gen_fill_f32_dev
    if f(dev_ptr, n, k, sigma, offset, stream) != 0:
        raise RuntimeError("device generator launch failed")
