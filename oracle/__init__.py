"""Oracle of the quantized MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Python binding of ``moe_oracle.cpp``, a plain, slow CPU reference (fp64
accumulation, fp32 quantisation decisions) of the whole layer: NVFP4 and FP6
e2m3 quantise / dequantise, router logits, softmax / top-k / renormalise,
expert-sorted dispatch, SwiGLU experts and the gate-weighted combine.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never uses it and shares
no code with it; the two meet only through the seeded inputs of ``gen``.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
published code tables, library routines (torch's e4m3 conversion, numpy
matmul / sort / bincount, scipy's softmax) and invariants.  The whole-layer
values have no worked example on the pages; beyond those pins they are
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "libmoe_oracle.so")
SRC = os.path.join(_HERE, "moe_oracle.cpp")
_lock = threading.Lock()
_lib = None

FMT_NVFP4 = 1
FMT_FP6 = 2
FMT_MXFP4 = 3


def build() -> None:
    """Compile the oracle with g++ (no fast-math, no FMA contraction)."""
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-pthread", SRC, "-o", LIB + ".tmp"])
    os.replace(LIB + ".tmp", LIB)


class _Layer(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("E", ctypes.c_int), ("k", ctypes.c_int), ("shared", ctypes.c_int),
                ("codes", ctypes.POINTER(ctypes.c_void_p)),
                ("scales", ctypes.POINTER(ctypes.c_void_p)),
                ("tscales", ctypes.c_void_p), ("router", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("act_fp4", ctypes.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            sig = {
                "orc_e2m1_value": (ctypes.c_double, [I]),
                "orc_e2m3_value": (ctypes.c_double, [I]),
                "orc_e4m3_value": (ctypes.c_double, [I]),
                "orc_ue8m0_value": (ctypes.c_double, [I]),
                "orc_e2m1_rne": (I, [F]),
                "orc_e2m3_rne": (I, [F]),
                "orc_e4m3_rne": (I, [F]),
                "orc_quantize_nvfp4": (I, [P, I, I, P, P, P]),
                "orc_quantize_fp6": (I, [P, I, I, P, P]),
                "orc_quantize_mxfp4": (I, [P, I, I, P, P]),
                "orc_dequant_mxfp4": (I, [P, P, I, I, P]),
                "orc_dequant_nvfp4": (I, [P, P, F, I, I, P]),
                "orc_dequant_fp6": (I, [P, P, I, I, P]),
                "orc_router_logits": (I, [P, P, I, P]),
                "orc_topk_gates": (I, [P, I, I, I, P, P]),
                "orc_topk_gates_sigmoid": (I, [P, P, I, I, I, P, P]),
                "orc_dispatch": (I, [P, I, I, I, P, P, P]),
                "orc_combine": (I, [P, P, I, P, P, P, I]),
                "orc_moe_forward": (I, [P, P, I, P, P, P, P, I]),
                "orc_expert_ffn": (I, [P, I, P, I, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with {rc}")


# ---------------------------------------------------------------- code tables / rounding
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e2m3_value(code: int) -> float:
    return lib().orc_e2m3_value(code)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def ue8m0_value(b: int) -> float:
    return lib().orc_ue8m0_value(b)


def e2m1_rne(v: float) -> int:
    return lib().orc_e2m1_rne(v)


def e2m3_rne(v: float) -> int:
    return lib().orc_e2m3_rne(v)


def e4m3_rne(v: float) -> int:
    return lib().orc_e4m3_rne(v)


# ---------------------------------------------------------------- quantise / dequantise
def quantize_nvfp4(W: np.ndarray):
    """fp32 [rows x K] -> (codes u8 [rows x K/2], scales u8 [rows x K/16], tscale float)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, K = W.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 16), np.uint8)
    ts = np.zeros(1, np.float32)
    _check(lib().orc_quantize_nvfp4(_p(W), rows, K, _p(codes), _p(scales), _p(ts)), "quantize")
    return codes, scales, float(ts[0])


def quantize_fp6(W: np.ndarray):
    """fp32 [rows x K] -> (codes u8 [rows x K], exps u8 [rows x K/128])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, K = W.shape
    codes = np.zeros((rows, K), np.uint8)
    exps = np.zeros((rows, K // 128), np.uint8)
    _check(lib().orc_quantize_fp6(_p(W), rows, K, _p(codes), _p(exps)), "quantize")
    return codes, exps


def quantize_mxfp4(W: np.ndarray):
    """fp32 [rows x K] -> (codes u8 [rows x K/2], exps u8 [rows x K/32])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, K = W.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    exps = np.zeros((rows, K // 32), np.uint8)
    _check(lib().orc_quantize_mxfp4(_p(W), rows, K, _p(codes), _p(exps)), "quantize")
    return codes, exps


def dequant_mxfp4(codes, exps, rows, K) -> np.ndarray:
    out = np.empty((rows, K), np.float32)
    _check(lib().orc_dequant_mxfp4(_p(codes), _p(exps), rows, K, _p(out)), "dequant")
    return out


def dequant_nvfp4(codes, scales, tscale, rows, K) -> np.ndarray:
    out = np.empty((rows, K), np.float32)
    _check(lib().orc_dequant_nvfp4(_p(codes), _p(scales), tscale, rows, K, _p(out)), "dequant")
    return out


def dequant_fp6(codes, exps, rows, K) -> np.ndarray:
    out = np.empty((rows, K), np.float32)
    _check(lib().orc_dequant_fp6(_p(codes), _p(exps), rows, K, _p(out)), "dequant")
    return out


# ---------------------------------------------------------------- the layer
class Layer:
    """Canonical (quantised) weights of one layer, as the oracle sees them.

    ``mats[(expert, matrix)] = (codes, scales, tscale)``; expert == E is the
    shared expert; matrices a call does not touch may be absent.
    """

    def __init__(self, fmt, H, I, E, k, shared, router_bf16, bias=None, act_fp4=False):
        """act_fp4: W4A4 (R20), every product's activations quantised to NVFP4
        per row (x per token, a per token and expert) before it."""
        self.fmt, self.H, self.I, self.E, self.k, self.shared = fmt, H, I, E, k, int(bool(shared))
        self.act_fp4 = bool(act_fp4)
        self.router = np.ascontiguousarray(router_bf16, dtype=np.uint16)
        self.bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        self.mats = {}

    def n_total(self):
        return self.E + self.shared

    def shape(self, matrix):
        return (self.I, self.H) if matrix in (0, 1) else (self.H, self.I)

    def set_matrix(self, expert, matrix, codes, scales, tscale=1.0):
        self.mats[(expert, matrix)] = (np.ascontiguousarray(codes), np.ascontiguousarray(scales),
                                       float(tscale))

    def quantize_matrix(self, expert, matrix, W):
        if self.fmt == FMT_NVFP4:
            c, s, ts = quantize_nvfp4(W)
        elif self.fmt == FMT_MXFP4:
            (c, s), ts = quantize_mxfp4(W), 1.0
        else:
            (c, s), ts = quantize_fp6(W), 1.0
        self.set_matrix(expert, matrix, c, s, ts)
        return self.mats[(expert, matrix)]

    def dequant(self, expert, matrix):
        c, s, ts = self.mats[(expert, matrix)]
        rows, K = self.shape(matrix)
        if self.fmt == FMT_NVFP4:
            return dequant_nvfp4(c, s, ts, rows, K)
        if self.fmt == FMT_MXFP4:
            return dequant_mxfp4(c, s, rows, K)
        return dequant_fp6(c, s, rows, K)

    def _struct(self):
        n = self.n_total() * 3
        codes = (ctypes.c_void_p * n)()
        scales = (ctypes.c_void_p * n)()
        ts = np.ones(n, np.float32)
        for (e, m), (c, s, t) in self.mats.items():
            codes[e * 3 + m] = c.ctypes.data
            scales[e * 3 + m] = s.ctypes.data
            ts[e * 3 + m] = t
        st = _Layer(self.fmt, self.H, self.I, self.E, self.k, self.shared,
                    ctypes.cast(codes, ctypes.POINTER(ctypes.c_void_p)),
                    ctypes.cast(scales, ctypes.POINTER(ctypes.c_void_p)),
                    ts.ctypes.data, self.router.ctypes.data,
                    None if self.bias is None else self.bias.ctypes.data, int(self.act_fp4))
        return st, (codes, scales, ts)  # keep the arrays alive with the struct

    def _need(self, experts):
        for e in set(int(v) for v in np.asarray(experts).ravel()):
            for m in range(3):
                if (e, m) not in self.mats:
                    raise KeyError(f"oracle layer lacks expert {e} matrix {m}")

    # -- steps
    def logits(self, x_bf16: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        T = x.shape[0]
        out = np.empty((T, self.E), np.float32)
        st, keep = self._struct()
        _check(lib().orc_router_logits(ctypes.byref(st), _p(x), T, _p(out)), "router")
        return out

    def topk(self, logits: np.ndarray):
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        T = lg.shape[0]
        idx = np.empty((T, self.k), np.int32)
        gates = np.empty((T, self.k), np.float32)
        _check(lib().orc_topk_gates(_p(lg), T, self.E, self.k, _p(idx), _p(gates)), "topk")
        return idx, gates

    def dispatch(self, idx: np.ndarray):
        return dispatch(idx, self.E)

    def combine(self, x_bf16, idx, gates, threads=None) -> np.ndarray:
        x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gates = np.ascontiguousarray(gates, dtype=np.float32)
        self._need(list(idx.ravel()) + ([self.E] if self.shared else []))
        T = x.shape[0]
        out = np.empty((T, self.H), np.float32)
        st, keep = self._struct()
        th = threads or min(T, os.cpu_count() or 1)
        _check(lib().orc_combine(ctypes.byref(st), _p(x), T, _p(idx), _p(gates), _p(out), th),
               "combine")
        return out

    def forward(self, x_bf16, threads=None):
        """Whole layer: returns (logits, idx, gates, out)."""
        lg = self.logits(x_bf16)
        idx, gates = self.topk(lg)
        return lg, idx, gates, self.combine(x_bf16, idx, gates, threads)

    def expert_ffn(self, expert, x_bf16) -> np.ndarray:
        x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        self._need([expert])
        T = x.shape[0]
        out = np.empty((T, self.H), np.float32)
        st, keep = self._struct()
        _check(lib().orc_expert_ffn(ctypes.byref(st), expert, _p(x), T, _p(out)), "expert_ffn")
        return out


def topk_gates_sigmoid(logits: np.ndarray, bias, k: int):
    """The sigmoid router (R19): logits [T x E] without the bias, bias [E] or
    None; returns (idx [T x k], gates [T x k])."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    idx = np.empty((T, k), np.int32)
    gates = np.empty((T, k), np.float32)
    _check(lib().orc_topk_gates_sigmoid(_p(lg), None if b is None else _p(b), T, E, k, _p(idx),
                                        _p(gates)), "topk sigmoid")
    return idx, gates


def dispatch(idx: np.ndarray, E: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    _check(lib().orc_dispatch(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm)), "dispatch")
    return counts, offsets, perm


def layer_for_workload(w, experts=None) -> Layer:
    """Oracle layer of a workload: router from the generator, the listed experts
    (all when None; E means the shared expert) quantised by the oracle itself."""
    import gen
    L = Layer(w.fmt, w.H, w.I, w.E, w.k, w.shared, gen.router_weights(w), gen.router_bias(w))
    if experts is None:
        experts = range(w.n_experts_total)
    jobs = [(int(e), m) for e in experts for m in range(3)]

    def one(job):  # the C calls release the GIL, so matrices quantise in parallel
        e, m = job
        return job, L_quantize(w, e, m)

    def L_quantize(w_, e, m):
        W = gen.expert_weight(w_, e, m)
        if w_.fmt == FMT_NVFP4:
            return quantize_nvfp4(W)
        if w_.fmt == FMT_MXFP4:
            c, s = quantize_mxfp4(W)
            return c, s, 1.0
        c, s = quantize_fp6(W)
        return c, s, 1.0

    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        for (e, m), (c, s, ts) in ex.map(one, jobs):
            L.set_matrix(e, m, c, s, ts)
    return L
