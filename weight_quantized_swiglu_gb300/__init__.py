"""Weight-quantized SwiGLU MLP for GB300 (sm_103a): thin Python binding.

Every step of the computation runs in the CUDA kernels of ``libqmlp.so``
(built in-tree by ``weight_quantized_swiglu_gb300.build``); this module only
marshals arguments through the C ABI declared in ``include/qmlp.h``. There is
no CPU fallback: if the library is missing or fails to load, every call
raises ``RuntimeError``, and a failed call raises ``QmlpError`` (a
``RuntimeError``) carrying the library's status.

Module-level functions carry the C names (``qmlp_create``, ``qmlp_forward``,
...); ``QuantMLP`` and ``MoeAWQ`` wrap the handles for convenience. Device
buffers are passed as torch CUDA tensors (or raw integer addresses); streams
as ``torch.cuda.Stream`` (or raw handles, 0 = legacy default stream).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libqmlp.so")

QMLP_OK = 0
STATUS = {0: "QMLP_OK", 1: "QMLP_ERR_INVALID_ARG", 2: "QMLP_ERR_ALIGNMENT", 3: "QMLP_ERR_ALIAS",
          4: "QMLP_ERR_SHAPE", 5: "QMLP_ERR_UNSUPPORTED_ARCH", 6: "QMLP_ERR_OOM", 7: "QMLP_ERR_CUDA",
          8: "QMLP_ERR_DEVICE_TIMEOUT", 9: "QMLP_ERR_DEVICE_BOUNDS"}
FMT_NVFP4, FMT_FP8_PC = 1, 2
DT_BF16, DT_FP16 = 1, 2
META_3B, META_4B = 3, 4
PATH_AUTO, PATH_GEMV, PATH_GEMM, PATH_GEMM_PAIR, PATH_GEMM_DQ = 0, 1, 2, 3, 4


class QmlpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class qmlp_proj(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("global_scale", ctypes.c_float)]


class qmlp_desc(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("K", ctypes.c_int), ("I", ctypes.c_int), ("max_M", ctypes.c_int),
                ("gate", qmlp_proj), ("up", qmlp_proj), ("down", qmlp_proj)]


class qmlp_moe_desc(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("K", ctypes.c_int), ("I", ctypes.c_int), ("meta", ctypes.c_int),
                ("w13", ctypes.c_void_p), ("w13_meta", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_meta", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None

_VP = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "qmlp_create": ([ctypes.POINTER(_VP), ctypes.POINTER(qmlp_desc), _VP], _I),
    "qmlp_destroy": ([_VP], None),
    "qmlp_forward": ([_VP, _VP, _I, _VP, _VP], _I),
    "qmlp_forward_path": ([_VP, _I, _VP, _I, _VP, _VP], _I),
    "qmlp_forward_host": ([_VP, _VP, _I, _VP, _VP], _I),
    "qmlp_forward_stage": ([_VP, _I, _I, _VP, _I, _VP, _VP], _I),
    "qmlp_forward_debug": ([_VP, _I, _VP, _I, _VP, _VP, _VP], _I),
    "qmlp_debug_project": ([_VP, _I, _I, _VP, _I, _VP, _VP], _I),
    "qmlp_check": ([_VP, _VP], _I),
    "qmlp_debug_split": ([_VP, _VP, _VP, _I, _VP, _VP, _VP, _VP], _I),
    "qmlp_debug_set_wait": ([_VP, ctypes.c_uint64, _I], _I),
    "qmlp_debug_bounds_enabled": ([], _I),
    "qmlp_debug_bounds": ([ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_ulonglong)], _I),
    "qmlp_debug_bounds_limit": ([_VP, ctypes.c_size_t], _I),
    "qmlp_create_shard": ([ctypes.POINTER(_VP), ctypes.POINTER(qmlp_desc), _I, _I, _VP], _I),
    "qmlp_forward_partial": ([_VP, _VP, _I, _VP, _VP], _I),
    "qmlp_shard_combine": ([_VP, _VP, _I, _I, _VP, _VP], _I),
    "qmlp_shard_info": ([_VP, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)], _I),
    "qmlp_decode_ctas": ([_VP], _I),
    "qmlp_moe_create": ([ctypes.POINTER(_VP), ctypes.POINTER(qmlp_moe_desc), _VP], _I),
    "qmlp_moe_destroy": ([_VP], None),
    "qmlp_moe_m1_forward": ([_VP, _VP, _I, _VP, _VP, _I, _VP, _VP], _I),
    "qmlp_moe_debug_stages": ([_VP, _VP, _I, _VP, _VP, _I, _VP, _VP, _VP, _VP, _VP], _I),
    "qmlp_moe_check": ([_VP, _VP], _I),
    "qmlp_moe_reserve": ([_VP, _I, _VP], _I),
    "qmlp_moe_forward": ([_VP, _VP, _I, _VP, _VP, _I, _I, _VP, _VP], _I),
    "qmlp_moe_m1_forward_noalloc": ([ctypes.POINTER(qmlp_moe_desc), _VP, _I, _VP, _VP, _I, _VP, _VP], _I),
    "qmlp_status_str": ([_I], ctypes.c_char_p),
    "qmlp_abi_version": ([], _I),
}


def lib(path: str | None = None):
    """Load libqmlp.so (raises QmlpError-compatible RuntimeError if absent).
    QMLP_LIB in the environment names another build of it to load instead
    (the index-checking build, lib/libqmlp_bounds.so)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or os.environ.get("QMLP_LIB") or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libqmlp.so not built ({p}); run weight_quantized_swiglu_gb300.build.build()")
            L = ctypes.CDLL(p)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _chk(st: int, where: str):
    if st != QMLP_OK:
        raise QmlpError(st, where)


# ---- C-named thin wrappers --------------------------------------------------
def qmlp_status_str(st: int) -> str:
    return lib().qmlp_status_str(st).decode()


def qmlp_abi_version() -> int:
    return lib().qmlp_abi_version()


def qmlp_create(desc: qmlp_desc, stream=None) -> int:
    h = ctypes.c_void_p()
    st = lib().qmlp_create(ctypes.byref(h), ctypes.byref(desc), _stream(stream))
    _chk(st, "qmlp_create")
    return h.value


def qmlp_destroy(h: int):
    lib().qmlp_destroy(h)


def qmlp_forward(h, x, M, out, stream=None) -> int:
    return lib().qmlp_forward(h, _ptr(x), M, _ptr(out), _stream(stream))


def qmlp_forward_path(h, path, x, M, out, stream=None) -> int:
    return lib().qmlp_forward_path(h, path, _ptr(x), M, _ptr(out), _stream(stream))


def qmlp_forward_stage(h, stage, path, x, M, out, stream=None) -> int:
    return lib().qmlp_forward_stage(h, stage, path, _ptr(x), M, _ptr(out), _stream(stream))


def qmlp_forward_host(h, x_host, M, out_host, stream=None) -> int:
    return lib().qmlp_forward_host(h, _ptr(x_host), M, _ptr(out_host), _stream(stream))


def qmlp_forward_debug(h, path, x, M, act, out, stream=None) -> int:
    return lib().qmlp_forward_debug(h, path, _ptr(x), M, _ptr(act), _ptr(out), _stream(stream))


def qmlp_debug_project(h, which, path, x, M, y, stream=None) -> int:
    return lib().qmlp_debug_project(h, which, path, _ptr(x), M, _ptr(y), _stream(stream))


def qmlp_check(h, stream=None) -> int:
    return lib().qmlp_check(h, _stream(stream))


def qmlp_debug_split(h, x, act_in, M, g, u, out_f32, stream=None) -> int:
    return lib().qmlp_debug_split(h, _ptr(x), _ptr(act_in), M, _ptr(g), _ptr(u), _ptr(out_f32), _stream(stream))


def qmlp_debug_set_wait(h, limit_ns: int, withhold_last_step: bool) -> int:
    return lib().qmlp_debug_set_wait(h, limit_ns, 1 if withhold_last_step else 0)


def qmlp_debug_bounds_enabled() -> int:
    return lib().qmlp_debug_bounds_enabled()


def qmlp_debug_bounds():
    """(status, site, index) of the first failed index check since the last
    call (a checking build; see include/qmlp.h)."""
    site, index = ctypes.c_int(0), ctypes.c_ulonglong(0)
    st = lib().qmlp_debug_bounds(ctypes.byref(site), ctypes.byref(index))
    return st, site.value, index.value


def qmlp_debug_bounds_limit(h, gate_up_bank_bytes: int) -> int:
    return lib().qmlp_debug_bounds_limit(h, gate_up_bank_bytes)


def qmlp_create_shard(desc: qmlp_desc, rank: int, nranks: int, stream=None) -> int:
    h = ctypes.c_void_p()
    st = lib().qmlp_create_shard(ctypes.byref(h), ctypes.byref(desc), rank, nranks, _stream(stream))
    _chk(st, "qmlp_create_shard")
    return h.value


def qmlp_forward_partial(h, x, M, partial, stream=None) -> int:
    return lib().qmlp_forward_partial(h, _ptr(x), M, _ptr(partial), _stream(stream))


def qmlp_shard_combine(h, partials, nranks, M, out, stream=None) -> int:
    return lib().qmlp_shard_combine(h, _ptr(partials), nranks, M, _ptr(out), _stream(stream))


def qmlp_shard_info(h):
    """(rank, nranks, I of the handle)"""
    r, n, i = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    if not lib().qmlp_shard_info(h, ctypes.byref(r), ctypes.byref(n), ctypes.byref(i)):
        raise QmlpError(1, "qmlp_shard_info")
    return r.value, n.value, i.value


def qmlp_decode_ctas(h) -> int:
    return lib().qmlp_decode_ctas(h)


def qmlp_moe_create(desc: qmlp_moe_desc, stream=None) -> int:
    h = ctypes.c_void_p()
    st = lib().qmlp_moe_create(ctypes.byref(h), ctypes.byref(desc), _stream(stream))
    _chk(st, "qmlp_moe_create")
    return h.value


def qmlp_moe_destroy(h: int):
    lib().qmlp_moe_destroy(h)


def qmlp_moe_m1_forward(h, x, xdt, ids, rw, topk, out, stream=None) -> int:
    return lib().qmlp_moe_m1_forward(h, _ptr(x), xdt, _ptr(ids), _ptr(rw), topk, _ptr(out), _stream(stream))


def qmlp_moe_debug_stages(h, x, xdt, ids, rw, topk, out, gu, act, y, stream=None) -> int:
    return lib().qmlp_moe_debug_stages(h, _ptr(x), xdt, _ptr(ids), _ptr(rw), topk, _ptr(out), _ptr(gu),
                                       _ptr(act), _ptr(y), _stream(stream))


def qmlp_moe_reserve(h, max_tokens, stream=None) -> int:
    return lib().qmlp_moe_reserve(h, max_tokens, _stream(stream))


def qmlp_moe_forward(h, x, xdt, ids, rw, topk, M, out, stream=None) -> int:
    return lib().qmlp_moe_forward(h, _ptr(x), xdt, _ptr(ids), _ptr(rw), topk, M, _ptr(out), _stream(stream))


def qmlp_moe_check(h, stream=None) -> int:
    return lib().qmlp_moe_check(h, _stream(stream))


def qmlp_moe_m1_forward_noalloc(banks: qmlp_moe_desc, x, xdt, ids, rw, topk, out, stream=None) -> int:
    """Routed-expert step on caller-owned device banks; allocates nothing."""
    return lib().qmlp_moe_m1_forward_noalloc(ctypes.byref(banks), _ptr(x), xdt, _ptr(ids), _ptr(rw), topk,
                                             _ptr(out), _stream(stream))


# ---- convenience handles ------------------------------------------------------
def _host_or_dev(a):
    """Keep numpy arrays (host) alive and return (address, owner)."""
    if isinstance(a, np.ndarray):
        a = np.ascontiguousarray(a)
        return a.ctypes.data, a
    return _ptr(a), a


class QuantMLP:
    """Dense weight-quantized SwiGLU MLP handle (NVFP4 or FP8 per-channel).

    Weights may be numpy arrays (host) or torch CUDA tensors; they are copied
    into handle-owned device memory at construction."""

    def __init__(self, fmt: str, K: int, I: int, max_M: int, gate, up, down, stream=None, shard=None):
        """shard = (rank, nranks): this rank's tensor-parallel shard of the
        whole layer described by the arguments (qmlp_create_shard)."""
        self.fmt = FMT_NVFP4 if fmt == "nvfp4" else FMT_FP8_PC
        self.K, self.I, self.max_M = K, I, max_M
        keep = []
        projs = []
        for p in (gate, up, down):
            w, o1 = _host_or_dev(p.w)
            s, o2 = _host_or_dev(p.scale)
            keep += [o1, o2]
            projs.append(qmlp_proj(w, s, float(p.global_scale)))
        d = qmlp_desc(self.fmt, K, I, max_M, *projs)
        if shard is None:
            self.h = qmlp_create(d, stream)
        else:
            self.h = qmlp_create_shard(d, shard[0], shard[1], stream)
            self.I = I // shard[1]
        self.rank, self.nranks, _ = qmlp_shard_info(self.h)

    @classmethod
    def from_case(cls, case, max_M=None, stream=None, shard=None):
        return cls(case.fmt, case.K, case.I, max_M or case.M, case.gate, case.up, case.down, stream, shard)

    def forward_partial(self, x, partial, M=None, stream=None):
        """fp32 [M, K] partial of a tensor-parallel shard (no down factor)."""
        M = x.shape[0] if M is None else M
        _chk(qmlp_forward_partial(self.h, x, M, partial, stream), "qmlp_forward_partial")
        return partial

    def combine(self, partials, out, M=None, stream=None):
        """out = bf16(sigma_d * rank-ordered sum of partials [nranks, M, K])."""
        M = partials.shape[1] if M is None else M
        _chk(qmlp_shard_combine(self.h, partials, self.nranks, M, out, stream), "qmlp_shard_combine")
        return out

    def debug_split(self, x, act_in, g, u, out_f32, M=None, stream=None):
        M = x.shape[0] if M is None else M
        _chk(qmlp_debug_split(self.h, x, act_in, M, g, u, out_f32, stream), "qmlp_debug_split")

    def set_wait(self, limit_ns: int, withhold_last_step: bool = False):
        _chk(qmlp_debug_set_wait(self.h, limit_ns, withhold_last_step), "qmlp_debug_set_wait")

    def bounds_limit(self, gate_up_bank_bytes: int):
        _chk(qmlp_debug_bounds_limit(self.h, gate_up_bank_bytes), "qmlp_debug_bounds_limit")

    def forward(self, x, out, M=None, path=PATH_AUTO, stream=None):
        M = x.shape[0] if M is None else M
        _chk(qmlp_forward_path(self.h, path, x, M, out, stream), "qmlp_forward")
        return out

    def forward_stage(self, stage, x, out, M, path=PATH_AUTO, stream=None):
        _chk(qmlp_forward_stage(self.h, stage, path, x, M, out, stream), "qmlp_forward_stage")

    def forward_debug(self, x, act, out, M=None, path=PATH_AUTO, stream=None):
        M = x.shape[0] if M is None else M
        _chk(qmlp_forward_debug(self.h, path, x, M, act, out, stream), "qmlp_forward_debug")
        return act, out

    def forward_host(self, x_host, out_host, M=None, stream=None):
        M = x_host.shape[0] if M is None else M
        _chk(qmlp_forward_host(self.h, x_host, M, out_host, stream), "qmlp_forward_host")
        return out_host

    def debug_project(self, which, x, y, M=None, path=PATH_AUTO, stream=None):
        M = x.shape[0] if M is None else M
        _chk(qmlp_debug_project(self.h, which, path, x, M, y, stream), "qmlp_debug_project")
        return y

    def check(self, stream=None):
        _chk(qmlp_check(self.h, stream), "qmlp_check")

    def decode_ctas(self):
        """CTAs of the I-partitioned single-launch decode kernel (0: not used)."""
        return qmlp_decode_ctas(self.h)

    def close(self):
        if getattr(self, "h", None):
            qmlp_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoeAWQ:
    """Routed-expert AWQ int4 g32 handle (one token; M tokens after reserve())."""

    def __init__(self, E, K, I, meta_bytes, w13, w13_meta, w2, w2_meta, stream=None):
        self.E, self.K, self.I, self.meta = E, K, I, meta_bytes
        ptrs = [_host_or_dev(a) for a in (w13, w13_meta, w2, w2_meta)]
        d = qmlp_moe_desc(E, K, I, meta_bytes, *[p for p, _ in ptrs])
        self.h = qmlp_moe_create(d, stream)

    @classmethod
    def from_case(cls, case, meta_bytes=4, stream=None):
        m13 = case.w13_meta4 if meta_bytes == 4 else case.w13_meta3
        m2 = case.w2_meta4 if meta_bytes == 4 else case.w2_meta3
        return cls(case.E, case.K, case.I, meta_bytes, case.w13, m13, case.w2, m2, stream)

    def forward(self, x, xdt, ids, rw, out, topk=None, stream=None):
        topk = ids.shape[0] if topk is None else topk
        _chk(qmlp_moe_m1_forward(self.h, x, xdt, ids, rw, topk, out, stream), "qmlp_moe_m1_forward")
        return out

    def reserve(self, max_tokens, stream=None):
        _chk(qmlp_moe_reserve(self.h, max_tokens, stream), "qmlp_moe_reserve")

    def forward_tokens(self, x, xdt, ids, rw, out, stream=None):
        """M tokens: x [M, K], ids / rw [M, topk], out [M, K]."""
        M, topk = ids.shape
        _chk(qmlp_moe_forward(self.h, x, xdt, ids, rw, topk, M, out, stream), "qmlp_moe_forward")
        return out

    def debug_stages(self, x, xdt, ids, rw, out, gu=None, act=None, y=None, topk=None, stream=None):
        topk = ids.shape[0] if topk is None else topk
        _chk(qmlp_moe_debug_stages(self.h, x, xdt, ids, rw, topk, out, gu, act, y, stream),
             "qmlp_moe_debug_stages")

    def check(self, stream=None):
        _chk(qmlp_moe_check(self.h, stream), "qmlp_moe_check")

    def close(self):
        if getattr(self, "h", None):
            qmlp_moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
