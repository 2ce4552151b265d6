"""CPU oracle for the weight-quantized SwiGLU MLP -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The library's product path never calls it: there
is no CPU fallback anywhere in ``weight_quantized_swiglu_gb300``.

The arithmetic lives in ``qmlp_oracle.c`` (plain C, fp64, table decode); this
module builds it with gcc and marshals numpy arrays through ctypes.

Pinned functions (see ``tests/test_oracle_pins.py``): E2M1/E4M3 tables,
bf16/fp16 rounding, NVFP4/FP8/AWQ decode, projection dot products, the dense
SwiGLU forward and the routed-expert forward. No function is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmlp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

NVFP4, FP8 = 1, 2


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
            _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.check_call(base[:1] + ["-fopenmp"] + base[1:], cwd=_HERE)
    except subprocess.CalledProcessError:
        subprocess.check_call(base, cwd=_HERE)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class _Proj(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("global_scale", ctypes.c_float)]


def _p(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.qo_e2m1.restype = ctypes.c_double
            L.qo_e2m1.argtypes = [ctypes.c_int]
            L.qo_e4m3.restype = ctypes.c_double
            L.qo_e4m3.argtypes = [ctypes.c_int]
            L.qo_bf16_rne.restype = ctypes.c_uint16
            L.qo_bf16_rne.argtypes = [ctypes.c_double]
            L.qo_fp16_rne.restype = ctypes.c_uint16
            L.qo_fp16_rne.argtypes = [ctypes.c_double]
            L.qo_bf16_value.restype = ctypes.c_double
            L.qo_bf16_value.argtypes = [ctypes.c_uint16]
            L.qo_fp16_value.restype = ctypes.c_double
            L.qo_fp16_value.argtypes = [ctypes.c_uint16]
            L.qo_num_threads.restype = ctypes.c_int
            for name in ("qo_bf16_rne_array", "qo_fp16_rne_array"):
                getattr(L, name).argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            L.qo_decode_proj.argtypes = [ctypes.c_int, ctypes.POINTER(_Proj), ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p]
            L.qo_project.argtypes = [ctypes.c_int, ctypes.POINTER(_Proj), ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
            L.qo_dense_forward.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(_Proj),
                                           ctypes.POINTER(_Proj), ctypes.POINTER(_Proj), ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p]
            L.qo_awq_decode.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
            L.qo_moe_m1_forward.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 5 + [
                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 4
            _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().qo_num_threads())


# ---------------------------------------------------------------- scalars
def e2m1(code: int) -> float:
    return float(lib().qo_e2m1(code))


def e4m3(byte: int) -> float:
    return float(lib().qo_e4m3(byte))


def bf16_rne(v: float) -> int:
    return int(lib().qo_bf16_rne(v))


def fp16_rne(v: float) -> int:
    return int(lib().qo_fp16_rne(v))


def bf16_value(bits: int) -> float:
    return float(lib().qo_bf16_value(bits))


def fp16_value(bits: int) -> float:
    return float(lib().qo_fp16_value(bits))


def bf16_rne_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().qo_bf16_rne_array(_p(v), v.size, _p(out))
    return out


def fp16_rne_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().qo_fp16_rne_array(_p(v), v.size, _p(out))
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> exact double (bf16 is the top half of an fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def fp16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# ---------------------------------------------------------------- dense path
def _proj(p) -> _Proj:
    return _Proj(p.w.ctypes.data, p.scale.ctypes.data, float(p.global_scale))


def _fmt(fmt) -> int:
    return NVFP4 if fmt in ("nvfp4", NVFP4) else FP8


def decode_proj(p) -> np.ndarray:
    """Decoded weights [N, K] in fp64 without the global/per-channel factor."""
    out = np.empty((p.N, p.K), dtype=np.float64)
    pr = _proj(p)
    lib().qo_decode_proj(_fmt(p.fmt), ctypes.byref(pr), p.N, p.K, _p(out))
    return out


def project(p, x_bits: np.ndarray, rows=None) -> np.ndarray:
    """x[rows] . decode(W)^T in fp64 (no channel factor); x is bf16 bits [M, K]."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M = x_bits.shape[0]
    rows = np.arange(M, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    y = np.empty((rows.size, p.N), dtype=np.float64)
    pr = _proj(p)
    lib().qo_project(_fmt(p.fmt), ctypes.byref(pr), p.N, p.K, _p(x_bits), rows.size, _p(rows), _p(y))
    return y


def dense_forward(case, rows=None, want_pre: bool = False):
    """SwiGLU MLP on token rows `rows` of case.x. Returns dict with 'out' (bf16
    bits [r, K]) and 'act' (bf16 bits [r, I]); with want_pre also 'g', 'u'
    (fp64 pre-activations [r, I]) and 'out_pre' (fp64 [r, K])."""
    x = np.ascontiguousarray(case.x, dtype=np.uint16)
    M = x.shape[0]
    rows = np.arange(M, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    R = rows.size
    out = np.empty((R, case.K), dtype=np.uint16)
    act = np.empty((R, case.I), dtype=np.uint16)
    g = np.empty((R, case.I), dtype=np.float64) if want_pre else None
    u = np.empty((R, case.I), dtype=np.float64) if want_pre else None
    op = np.empty((R, case.K), dtype=np.float64) if want_pre else None
    pg, pu, pd = _proj(case.gate), _proj(case.up), _proj(case.down)
    lib().qo_dense_forward(_fmt(case.fmt), case.K, case.I, _p(x), R, _p(rows), ctypes.byref(pg),
                           ctypes.byref(pu), ctypes.byref(pd), _p(out), _p(act), _p(g), _p(u), _p(op))
    res = {"out": out, "act": act}
    if want_pre:
        res.update(g=g, u=u, out_pre=op)
    return res


# ---------------------------------------------------------------- AWQ MoE path
def awq_decode(w: np.ndarray, meta: np.ndarray, meta_bytes: int, e: int) -> np.ndarray:
    """Decoded fp16-valued weights (as fp64) of expert e: [N, Kr]."""
    E, N, half = w.shape
    Kr = half * 2
    w = np.ascontiguousarray(w)
    meta = np.ascontiguousarray(meta)
    out = np.empty((N, Kr), dtype=np.float64)
    lib().qo_awq_decode(_p(w), _p(meta), meta_bytes, E, N, Kr, e, _p(out))
    return out


def moe_m1_forward(case, meta_bytes: int = 4, x_dtype: str = "fp16", ids=None, rw=None,
                   want_stages: bool = False):
    """Routed-expert M=1 forward. Returns dict with 'out' (fp16 bits [K]) and,
    with want_stages, 'gu' [topk, 2I], 'act' [topk, I], 'y' [topk, K] (fp16
    bits) plus 'valid' [topk] booleans."""
    ids = np.ascontiguousarray(case.ids if ids is None else ids, dtype=np.int32)
    rw = np.ascontiguousarray(case.router_w if rw is None else rw, dtype=np.float32)
    topk = ids.size
    m13 = case.w13_meta4 if meta_bytes == 4 else case.w13_meta3
    m2 = case.w2_meta4 if meta_bytes == 4 else case.w2_meta3
    x = case.x_fp16 if x_dtype == "fp16" else case.x_bf16
    out = np.empty(case.K, dtype=np.uint16)
    gu = np.zeros((topk, 2 * case.I), dtype=np.uint16) if want_stages else None
    act = np.zeros((topk, case.I), dtype=np.uint16) if want_stages else None
    y = np.zeros((topk, case.K), dtype=np.uint16) if want_stages else None
    lib().qo_moe_m1_forward(case.E, case.K, case.I, meta_bytes, _p(np.ascontiguousarray(case.w13)),
                            _p(np.ascontiguousarray(m13)), _p(np.ascontiguousarray(case.w2)),
                            _p(np.ascontiguousarray(m2)), _p(np.ascontiguousarray(x)),
                            1 if x_dtype == "bf16" else 0, _p(ids), _p(rw), topk, _p(out), _p(gu),
                            _p(act), _p(y))
    res = {"out": out}
    if want_stages:
        res.update(gu=gu, act=act, y=y, valid=(ids >= 0) & (ids < case.E))
    return res
