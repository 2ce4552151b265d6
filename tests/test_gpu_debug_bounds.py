"""The index-checking build (QMLP_DEBUG_BOUNDS; include/qmlp.h, "Index
checks"): compute-sanitizer cannot run here, so every kernel can be built to
check the index of each computed global access against its buffer and to
record the first bad one instead of making it.

* Every kernel family runs in a checking build (a child process with QMLP_LIB
  naming lib/libqmlp_bounds.so) on the workloads of tests/bounds_cases.py:
  no check fails, and every output is bit-identical to the default build's
  (the checks change no arithmetic).
* A planted failure that faults nothing: the decode kernel is told that its
  gate/up banks are half as long as they are, so the copies of its later
  weight steps fail their check (and are taken from the bank start, which
  exists); qmlp_debug_bounds reports site 1 with an index past the cut, once,
  and the same handle is clean again when the limit is lifted.
The CPU part (test_abi-like): the checking build loads and says so."""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
BOUNDS = 9
assert q.STATUS[BOUNDS] == "QMLP_ERR_DEVICE_BOUNDS"


def test_checking_build_loads_and_reports_itself():
    """No GPU needed: both builds load side by side and answer."""
    lib_default = ctypes.CDLL(build.build())
    lib_check = ctypes.CDLL(build.build(bounds=True))
    assert lib_default.qmlp_debug_bounds_enabled() == 0
    assert lib_check.qmlp_debug_bounds_enabled() == 1
    # the default build has nothing to shrink
    assert lib_default.qmlp_debug_bounds_limit(None, ctypes.c_size_t(0)) == 1


@pytest.mark.gpu
def test_checking_build_is_clean_and_bit_identical(cuda_available, tmp_path):
    import bounds_cases
    build.build()
    lib_check = build.build(bounds=True)
    q.lib()
    out = str(tmp_path / "bounds.npz")
    env = dict(os.environ, QMLP_LIB=lib_check)
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_cases.py"), out], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    got = np.load(out)
    info = json.load(open(out + ".json"))
    for name, rep in info["reports"].items():
        assert rep == [0, 0, 0], (name, rep)
    ref, _ = bounds_cases.run(False)
    assert set(ref) <= set(got.files)
    for name, b in ref.items():
        assert np.array_equal(got[name], b), name
    # the planted cut: site 1 (the decode kernel's gate/up copies), an index
    # past the allowed bytes, reported once; clean after the limit is lifted
    status, site, index = info["cut"]
    assert (status, site) == (BOUNDS, 1), info["cut"]
    assert index >= info["half"]
    assert info["after"] == [0, 0, 0]
    assert np.array_equal(got["planted_out"], ref["nvfp4_decode_m1"])
