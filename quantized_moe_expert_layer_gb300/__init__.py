"""Quantized MoE expert layer for GB300 (sm_103a): Python binding of the C ABI.

Thin ctypes marshalling over ``libmoe_gb300.so`` (``include/moe.h``).  Every
step of the layer runs in the library's CUDA kernels; torch is used here only
to hold device memory and streams.  If the library is missing the import of
``lib()`` raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
CSRC = os.path.join(_HERE, "csrc")
BUILD = os.path.join(_HERE, "_build")
LIB = os.path.join(_HERE, "libmoe_gb300.so")
HEADER = os.path.join(_ROOT, "include", "moe.h")
SOURCES = ["layer.cu", "quant_pack.cu", "route.cu", "expert.cu", "noalloc.cu", "tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-cudart", "shared"]

FMT_NVFP4 = 1
FMT_FP6 = 2
FMT_MXFP4 = 3
GATE, UP, DOWN = 0, 1, 2
ROUTER_SOFTMAX, ROUTER_SIGMOID = 0, 1
ACT_BF16, ACT_NVFP4 = 0, 1
PATH_DECODE, PATH_STREAM, PATH_TC_F16, PATH_TC_FP4 = 0, 1, 2, 3
HOST, DEVICE = 0, 1

OK, EINVAL, ENOMEM, ECUDA, ESTATE, ETIMEOUT, ERANGE = 0, -1, -2, -3, -4, -5, -6

# every symbol include/moe.h declares
EXPORTS = [
    "moe_layer_create", "moe_layer_reserve", "moe_layer_destroy", "moe_last_error",
    "moe_layer_status", "moe_layer_info", "moe_set_router", "moe_pack_matrix",
    "moe_pack_weights", "moe_set_router_mode", "moe_quantize_nvfp4", "moe_quantize_fp6", "moe_quantize_mxfp4", "moe_forward",
    "moe_forward_host", "moe_forward_routed", "moe_debug_dequant", "moe_debug_routing",
    "moe_debug_run_phase", "moe_route_noalloc", "moe_forward_launches", "moe_forward_path",
    "moe_place_experts",
    "moe_layer_placement", "moe_set_wait_budget", "moe_debug_fail_alloc",
    "moe_debug_check_workspace", "moe_set_act_format", "moe_quantize_act_nvfp4"
]

_lock = threading.Lock()
_lib = None


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [HEADER]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources for sm_103a (in parallel) and link the shared library."""
    deps = _deps()
    if not force and os.path.exists(LIB) and all(
            os.path.getmtime(LIB) >= os.path.getmtime(d) for d in deps):
        return LIB
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = ["nvcc", *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = LIB + ".tmp"
    subprocess.check_call(["nvcc", *ARCH, "-shared", "-cudart", "shared", "-o", tmp,
                           *[o for o, _ in results]])
    os.replace(tmp, LIB)
    return LIB


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"{LIB} is missing: run __graft_entry__.build() "
                                   "(the layer has no CPU fallback)")
            L = ctypes.CDLL(LIB)
            P, I, F, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64
            sig = {
                "moe_layer_create": (I, [I, I, I, I, I, I, ctypes.POINTER(P)]),
                "moe_layer_reserve": (I, [P, I]),
                "moe_layer_destroy": (None, [P]),
                "moe_last_error": (ctypes.c_char_p, []),
                "moe_layer_status": (I, [P, I, ctypes.POINTER(I)]),
                "moe_layer_info": (I, [P, ctypes.POINTER(U64), ctypes.POINTER(U64)]),
                "moe_set_router": (I, [P, P, P, I]),
                "moe_pack_matrix": (I, [P, I, I, P, P, P, I, P]),
                "moe_pack_weights": (I, [P, P, P, P]),
                "moe_quantize_nvfp4": (I, [P, I, I, P, P, P, P]),
                "moe_quantize_fp6": (I, [P, I, I, P, P, P]),
                "moe_quantize_mxfp4": (I, [P, I, I, P, P, P]),
                "moe_set_router_mode": (I, [P, I]),
                "moe_forward": (I, [P, P, I, P, P]),
                "moe_forward_host": (I, [P, P, I, P, P]),
                "moe_forward_routed": (I, [P, P, I, P, P, P, P]),
                "moe_debug_dequant": (I, [P, I, I, P, P]),
                "moe_debug_routing": (I, [P, P, P, P, P, P, P, P]),
                "moe_debug_run_phase": (I, [P, I, P, I, P, P]),
                "moe_route_noalloc": (I, [P, I, I, P, P, I, I, P, P, P, P]),
                "moe_forward_launches": (I, [P, I]),
                "moe_forward_path": (I, [P, I]),
                "moe_place_experts": (I, [P, P]),
                "moe_layer_placement": (I, [P, P, ctypes.POINTER(U64), ctypes.POINTER(U64)]),
                "moe_set_wait_budget": (I, [P, ctypes.c_int64]),
                "moe_debug_fail_alloc": (I, [I]),
                "moe_debug_check_workspace": (I, [P, ctypes.POINTER(I)]),
                "moe_set_act_format": (I, [P, I]),
                "moe_quantize_act_nvfp4": (I, [P, I, I, I, P, P, P, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def check(rc: int) -> int:
    if rc < 0:
        raise MoeError(rc, lib().moe_last_error().decode())
    return rc


def _ptr(t):
    """Device (or host) address of a torch tensor / numpy array / None."""
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


class MoeLayer:
    """One quantized MoE layer on the current CUDA device (see include/moe.h)."""

    def __init__(self, fmt, H, I, E, k, shared):
        self.fmt, self.H, self.I, self.E, self.k, self.shared = fmt, H, I, E, k, int(shared)
        h = ctypes.c_void_p()
        check(lib().moe_layer_create(fmt, H, I, E, k, int(shared), ctypes.byref(h)))
        self.h = h

    def close(self):
        if self.h:
            lib().moe_layer_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reserve(self, T_max):
        check(lib().moe_layer_reserve(self.h, T_max))


    def launches(self, T):
        """Kernels one forward of T tokens launches."""
        return check(lib().moe_forward_launches(self.h, T))

    def path(self, T):
        """The expert path a forward of T tokens takes: PATH_DECODE, PATH_STREAM,
        PATH_TC_F16 or PATH_TC_FP4."""
        return check(lib().moe_forward_path(self.h, T))

    def info(self):
        a, e = ctypes.c_uint64(), ctypes.c_uint64()
        check(lib().moe_layer_info(self.h, ctypes.byref(a), ctypes.byref(e)))
        return a.value, e.value

    def place_experts(self, in_hbm):
        """Per expert (routed ones, then the shared one): True = an HBM slot,
        False = the pinned host mirror the kernels read over the CPU-GPU link."""
        import numpy as np
        m = np.ascontiguousarray(np.asarray(in_hbm, dtype=np.uint8).reshape(-1))
        if m.size != self.E + self.shared:
            raise ValueError(f"place_experts: {m.size} flags for {self.E + self.shared} experts")
        check(lib().moe_place_experts(self.h, _ptr(m)))

    def placement(self):
        """(in_hbm flags as a numpy bool array, HBM bytes, host-mirror bytes)."""
        import numpy as np
        m = np.zeros(self.E + self.shared, np.uint8)
        a, b = ctypes.c_uint64(), ctypes.c_uint64()
        check(lib().moe_layer_placement(self.h, _ptr(m), ctypes.byref(a), ctypes.byref(b)))
        return m.astype(bool), a.value, b.value

    def status(self, reset=False):
        """The device status word (0 or a negative moe_status a kernel recorded)."""
        v = ctypes.c_int()
        check(lib().moe_layer_status(self.h, int(reset), ctypes.byref(v)))
        return v.value

    def set_wait_budget(self, cycles):
        """Budget (clock64 cycles) of each bounded wait in the tensor-core
        kernels; 0 restores the default (about one second)."""
        check(lib().moe_set_wait_budget(self.h, int(cycles)))

    def set_act_format(self, fmt):
        """ACT_BF16 (W4A16, default) or ACT_NVFP4 (W4A4: activations quantised per row)."""
        check(lib().moe_set_act_format(self.h, fmt))

    def check_workspace(self):
        """Guard bytes of the workspace that a kernel overwrote (0 = none)."""
        v = ctypes.c_int()
        check(lib().moe_debug_check_workspace(self.h, ctypes.byref(v)))
        return v.value

    def pack_weights(self, router, bias, mats):
        """Whole layer from host memory (moe_pack_weights): router bf16 bits
        [E x H], bias fp32 [E] or None, mats[(expert, matrix)] = (codes,
        scales, tscale) numpy arrays in the canonical format for every expert
        in [0, E + shared) and matrix 0..2."""
        import numpy as np
        n = self.E + self.shared
        arr = (_CanonicalMatrix * (3 * n))()
        keep = []
        for e in range(n):
            for m in range(3):
                c, sc, ts = mats[(e, m)]
                c = np.ascontiguousarray(c, dtype=np.uint8)
                sc = np.ascontiguousarray(sc, dtype=np.uint8)
                keep += [c, sc]
                arr[3 * e + m].codes = c.ctypes.data
                arr[3 * e + m].scales = sc.ctypes.data
                arr[3 * e + m].tscale = float(ts)
        wr = np.ascontiguousarray(router, dtype=np.uint16)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        check(lib().moe_pack_weights(self.h, _ptr(wr), _ptr(b), ctypes.cast(arr, ctypes.c_void_p)))

    def set_router(self, wr, bias=None, where=None):
        where = _where(wr) if where is None else where
        check(lib().moe_set_router(self.h, _ptr(wr), _ptr(bias), where))

    def set_router_mode(self, mode):
        """ROUTER_SOFTMAX (default) or ROUTER_SIGMOID (selection-only bias)."""
        check(lib().moe_set_router_mode(self.h, mode))

    def pack_matrix(self, expert, matrix, codes, scales, tscale=None, stream=None):
        """codes/scales (+ tscale) as torch device tensors or numpy host arrays."""
        where = _where(codes)
        if where == HOST:
            import numpy as np
            ts = None if tscale is None else np.array([tscale], np.float32)
            check(lib().moe_pack_matrix(self.h, expert, matrix, _ptr(codes), _ptr(scales),
                                        _ptr(ts), HOST, None))
        else:
            check(lib().moe_pack_matrix(self.h, expert, matrix, _ptr(codes), _ptr(scales),
                                        _ptr(tscale), DEVICE, _stream(stream)))

    def forward(self, x, out, T=None, stream=None):
        T = x.shape[0] if T is None else T
        check(lib().moe_forward(self.h, _ptr(x), T, _ptr(out), _stream(stream)))

    def forward_host(self, x_host, out_host, T=None, stream=None):
        T = x_host.shape[0] if T is None else T
        check(lib().moe_forward_host(self.h, _ptr(x_host), T, _ptr(out_host), _stream(stream)))

    def forward_routed(self, x, idx, gates, out, stream=None):
        check(lib().moe_forward_routed(self.h, _ptr(x), x.shape[0], _ptr(idx), _ptr(gates),
                                       _ptr(out), _stream(stream)))

    def run_phase(self, phase, x, out, T=None, stream=None):
        T = x.shape[0] if T is None else T
        check(lib().moe_debug_run_phase(self.h, phase, _ptr(x), T, _ptr(out), _stream(stream)))

    def debug_dequant(self, expert, matrix, out, stream=None):
        check(lib().moe_debug_dequant(self.h, expert, matrix, _ptr(out), _stream(stream)))

    def debug_routing(self, logits=None, idx=None, gates=None, counts=None, offsets=None,
                      perm=None, stream=None):
        check(lib().moe_debug_routing(self.h, _ptr(logits), _ptr(idx), _ptr(gates), _ptr(counts),
                                      _ptr(offsets), _ptr(perm), _stream(stream)))


class _CanonicalMatrix(ctypes.Structure):
    """moe_canonical_matrix of include/moe.h."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tscale", ctypes.c_float)]


def fail_alloc(n):
    """Test hook: the n-th following allocation of the library fails (0 = none)."""
    check(lib().moe_debug_fail_alloc(int(n)))


def _where(t):
    return DEVICE if (hasattr(t, "is_cuda") and t.is_cuda) else HOST


def quantize_nvfp4(W, codes, scales, tscale, stream=None):
    rows, K = W.shape
    check(lib().moe_quantize_nvfp4(_ptr(W), rows, K, _ptr(codes), _ptr(scales), _ptr(tscale),
                                   _stream(stream)))


def quantize_fp6(W, codes, exps, stream=None):
    rows, K = W.shape
    check(lib().moe_quantize_fp6(_ptr(W), rows, K, _ptr(codes), _ptr(exps), _stream(stream)))


def quantize_mxfp4(W, codes, exps, stream=None):
    rows, K = W.shape
    check(lib().moe_quantize_mxfp4(_ptr(W), rows, K, _ptr(codes), _ptr(exps), _stream(stream)))


def quantize_act_nvfp4(A, codes, scales, tscale, stream=None):
    """Activation rows A [rows x K] (bf16 bits as int16/uint16, or fp32) to
    canonical NVFP4 with one tensor scale per row."""
    import torch
    rows, K = A.shape
    in_bf16 = 1 if A.dtype in (torch.int16, torch.bfloat16) else 0
    check(lib().moe_quantize_act_nvfp4(_ptr(A), in_bf16, rows, K, _ptr(codes), _ptr(scales),
                                       _ptr(tscale), _stream(stream)))


def route_noalloc(x, wr, bias, E, k, logits, idx, gates, stream=None):
    """Router logits + top-k with no device allocation (see moe_route_noalloc):
    x [T x H] and wr [E x H] bf16 bits, bias [E] fp32 or None, outputs on the device."""
    T, H = x.shape
    check(lib().moe_route_noalloc(_ptr(x), T, H, _ptr(wr), _ptr(bias), E, k, _ptr(logits),
                                  _ptr(idx), _ptr(gates), _stream(stream)))
