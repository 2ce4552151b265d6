"""C-ABI library checks that need no GPU: it builds for sm_103a, loads, and
exports every symbol include/qmlp.h declares; host-side validation rejects
bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import build as qbuild


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "qmlp.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(qmlp_[a-z0-9_]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return q.lib()


def test_header_declares_the_three_entry_points():
    syms = declared_symbols()
    for s in ("qmlp_create", "qmlp_forward", "qmlp_moe_m1_forward"):
        assert s in syms


def test_library_exports_every_declared_symbol(L):
    syms = declared_symbols()
    assert len(syms) >= 15
    missing = [s for s in syms if not hasattr(L, s)]
    assert not missing, missing


def test_binding_signatures_cover_the_header():
    assert set(declared_symbols()) == set(q._SIGS)


def header_enum(prefix):
    txt = open(os.path.join(ROOT, "include", "qmlp.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return {k: int(v) for k, v in re.findall(r"\b(" + prefix + r"[A-Z0-9_]+)\s*=\s*(\d+)", txt)}


def test_binding_constants_match_the_header():
    """Every kernel-family path and status value the binding names is the
    header's own (a path added on one side only would call another kernel)."""
    paths = header_enum("QMLP_PATH_")
    assert paths == {"QMLP_PATH_AUTO": q.PATH_AUTO, "QMLP_PATH_GEMV": q.PATH_GEMV, "QMLP_PATH_GEMM": q.PATH_GEMM,
                     "QMLP_PATH_GEMM_PAIR": q.PATH_GEMM_PAIR, "QMLP_PATH_GEMM_DQ": q.PATH_GEMM_DQ}
    status = {k: v for k, v in header_enum("QMLP_").items() if k.startswith(("QMLP_OK", "QMLP_ERR_"))}
    assert status == {name: code for code, name in q.STATUS.items()}


def test_status_strings(L):
    assert q.qmlp_status_str(0) == "QMLP_OK"
    assert q.qmlp_status_str(8) == "QMLP_ERR_DEVICE_TIMEOUT"
    assert q.qmlp_abi_version() == 104


def test_null_arguments_are_rejected_without_a_device(L):
    assert L.qmlp_forward(None, None, 1, None, None) == 1
    assert L.qmlp_moe_m1_forward(None, None, 1, None, None, 1, None, None) == 1
    h = ctypes.c_void_p()
    assert L.qmlp_create(ctypes.byref(h), None, None) == 1
    assert L.qmlp_create(None, None, None) == 1
    L.qmlp_destroy(None)
    L.qmlp_moe_destroy(None)


def test_bad_shapes_are_rejected_before_the_device(L):
    h = ctypes.c_void_p()
    dummy = (ctypes.c_uint8 * 64)()
    p = q.qmlp_proj(ctypes.addressof(dummy), ctypes.addressof(dummy), 1.0)
    for K, I, M in ((24, 32, 1), (32, 40, 1), (32, 32, 0), (8, 32, 1)):
        d = q.qmlp_desc(q.FMT_NVFP4, K, I, M, p, p, p)
        assert L.qmlp_create(ctypes.byref(h), ctypes.byref(d), None) == 4, (K, I, M)
    d = q.qmlp_desc(7, 32, 32, 1, p, p, p)
    assert L.qmlp_create(ctypes.byref(h), ctypes.byref(d), None) == 1
    m = q.qmlp_moe_desc(4, 100, 160, 4, ctypes.addressof(dummy), ctypes.addressof(dummy),
                        ctypes.addressof(dummy), ctypes.addressof(dummy))
    assert L.qmlp_moe_create(ctypes.byref(h), ctypes.byref(m), None) == 4
    m = q.qmlp_moe_desc(4, 2560, 160, 5, ctypes.addressof(dummy), ctypes.addressof(dummy),
                        ctypes.addressof(dummy), ctypes.addressof(dummy))
    assert L.qmlp_moe_create(ctypes.byref(h), ctypes.byref(m), None) == 1


def test_library_is_built_for_sm_103a_only():
    assert qbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_noalloc_rejects_out_overlapping_the_banks_without_a_device(L):
    """The allocation-free routed-expert call reads the caller's banks in
    place, so an output that overlaps any of them is an alias error; the
    check is pointer arithmetic only and runs before any device call."""
    E, K, I, meta = 4, 64, 32, 4
    sizes = [E * 2 * I * (K // 2), E * 2 * I * (K // 32) * meta, E * K * (I // 2), E * K * (I // 32) * meta]
    base = 1 << 32
    addr, pos = [], base
    for n in sizes:  # four disjoint, 256-byte aligned fake device ranges
        addr.append(pos)
        pos += (n + 255) // 256 * 256 + 4096
    x, ids, rw = pos, pos + 4096, pos + 8192
    desc = q.qmlp_moe_desc(E, K, I, meta, *addr)
    for a, n in zip(addr, sizes):
        for out in (a, a + (n // 32) * 16):  # start of a bank, and inside it
            assert q.qmlp_moe_m1_forward_noalloc(desc, x, q.DT_FP16, ids, rw, 4, out, 0) == 3, hex(out)
    # an output just past the last bank passes the alias checks and then
    # needs the device: anything but ALIAS (no GPU here)
    out = addr[3] + (sizes[3] + 15) // 16 * 16 + 1024
    assert q.qmlp_moe_m1_forward_noalloc(desc, x, q.DT_FP16, ids, rw, 4, out, 0) != 3
