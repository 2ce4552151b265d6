"""Bit-exact weight decode through the single-launch decode kernel's own
layouts (the I-partitioned gemv_split kernel that serves the 27B-class decode
calls), through the C ABI (qmlp_debug_split): its gate/up records in the
CTA-interleaved order and its CTA-sliced copy of the down projection.

With one-hot x the raw gate/up outputs are single decoded weights, and with a
one-hot act the raw down output is a single decoded down weight from the one
CTA whose slice holds that column (every other CTA adds an exact zero):
each must equal the oracle's decoded weight bit for bit (Qwen3.8-27B-NVFP4,
"NVFP4 numerics as implemented"; vllm.cpp issue, "Mechanism on the tp>1 path"
for e4m3fn). Also: the E4M3 / e4m3fn NaN codes 0x7F and 0xFF decode to NaN on
every kernel family, as the oracle's table says."""
import numpy as np
import pytest

import oracle
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from helpers import to_dev

pytestmark = pytest.mark.gpu

K, I = gen.DENSE_K, gen.DENSE_I


@pytest.fixture(scope="module")
def torch_cuda(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    q.lib()
    return torch


def one_hot(n, positions):
    x = np.zeros((len(positions), n), dtype=np.uint16)
    for r, k in enumerate(positions):
        x[r, k] = 0x3F80  # bf16 1.0
    return x


def run_split(torch, mlp, x_bits, act_bits):
    M = x_bits.shape[0]
    g = torch.full((M, mlp.I), float("nan"), dtype=torch.float32, device="cuda")
    u = torch.full((M, mlp.I), float("nan"), dtype=torch.float32, device="cuda")
    o = torch.full((M, mlp.K), float("nan"), dtype=torch.float32, device="cuda")
    mlp.debug_split(to_dev(x_bits), to_dev(act_bits), g, u, o)
    torch.cuda.synchronize()
    mlp.check()
    return (g.cpu().numpy().astype(np.float64), u.cpu().numpy().astype(np.float64),
            o.cpu().numpy().astype(np.float64))


# k of x (gate/up) and i of act (down) probed per call: scale-group, chunk and
# record boundaries, and -- for the down columns -- the edges of several CTAs'
# 128-column slices (136 CTAs x 8 row tiles at this shape)
X_SETS = [[0, 15, 16, 31, 63, 64, K - 1], [1, 100, 1000, 2559, 2560, 4095, 5103]]
A_SETS = [[0, 15, 16, 31, 63, 64, I - 1], [127, 128, 128 * 67 + 5, 8703, 8704, 128 * 135, I - 17]]


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("M", [1, 7])
def test_split_kernel_one_hot_is_bit_exact(torch_cuda, fmt, M):
    """M = 1 runs the one-token instance (NVFP4: the in-kernel ticket
    reduction), M = 7 the multi-token one with the separate reduce kernel."""
    torch = torch_cuda
    case = gen.gen_dense_case(fmt, K, I, 1, seed=301 if fmt == "nvfp4" else 302)
    mlp = q.QuantMLP.from_case(case, max_M=8)
    assert mlp.decode_ctas() == 136
    if M > 1:
        calls = list(zip(X_SETS, A_SETS))
    else:  # one position per call: every third pair of the two sets
        calls = [([k], [i]) for k, i in zip(X_SETS[0] + X_SETS[1], A_SETS[0] + A_SETS[1])][::3]
    for kx, ia in calls:
        xb, ab = one_hot(K, kx), one_hot(I, ia)
        g, u, o = run_split(torch, mlp, xb, ab)
        # the oracle's dot of a one-hot row is the decoded weight itself
        assert np.array_equal(g, oracle.project(case.gate, xb)), (fmt, kx)
        assert np.array_equal(u, oracle.project(case.up, xb)), (fmt, kx)
        assert np.array_equal(o, oracle.project(case.down, ab)), (fmt, ia)
    mlp.close()


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_split_kernel_raw_dot_products(torch_cuda, fmt):
    """Random x and act through the same raw epilogues: fp32 sums against the
    oracle's fp64 dots (relative L2 below 1e-5)."""
    torch = torch_cuda
    case = gen.gen_dense_case(fmt, K, I, 1, seed=303)
    mlp = q.QuantMLP.from_case(case, max_M=8)
    xb = gen.gen_x_only(304, 5, K)
    ab = gen.gen_x_only(305, 5, I)
    g, u, o = run_split(torch, mlp, xb, ab)
    for got, ref in ((g, oracle.project(case.gate, xb)), (u, oracle.project(case.up, xb)),
                     (o, oracle.project(case.down, ab))):
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-5
    mlp.close()


def _nan_case(fmt):
    """The tiny shape (K=256, I=512: a 4-CTA partition, and GEMM tiles) with
    NaN codes planted: NVFP4 E4M3 scale bytes 0x7F / 0xFF, FP8 weight bytes
    0x7F / 0xFF, in gate (rows 3, 5) and down (row 7)."""
    case = gen.gen_dense_case(fmt, gen.TINY_K, gen.TINY_I, 1, seed=310)
    if fmt == "nvfp4":
        case.gate.scale[3, 2] = 0x7F
        case.gate.scale[5, 0] = 0xFF
        case.down.scale[7, 1] = 0x7F
    else:
        case.gate.w[3, 33] = 0x7F
        case.gate.w[5, 200] = 0xFF
        case.down.w[7, 17] = 0xFF
    return case


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_nan_codes_decode_to_nan_on_every_path(torch_cuda, fmt):
    torch = torch_cuda
    case = _nan_case(fmt)
    ks = [0, 16, 33, 40, 200, 255]
    xb = one_hot(case.K, ks)
    ab = one_hot(case.I, [0, 17, 20, 300, 511, 256])
    ref_g, ref_u, ref_d = oracle.project(case.gate, xb), oracle.project(case.up, xb), oracle.project(case.down, ab)
    # the oracle's table decodes the planted codes to NaN, so the rows that
    # hold one are NaN for every x (0 * NaN = NaN), and only those rows
    assert np.isnan(ref_g[:, 3]).all() and np.isnan(ref_g[:, 5]).all() and np.isnan(ref_d[:, 7]).all()
    assert np.isnan(ref_g).any(axis=0).sum() == 2 and np.isnan(ref_d).any(axis=0).sum() == 1
    assert not np.isnan(ref_u).any()
    mlp = q.QuantMLP.from_case(case, max_M=64)
    for path in (q.PATH_GEMV, q.PATH_GEMM):
        for which, proj, x, ref in ((0, case.gate, xb, ref_g), (1, case.up, xb, ref_u), (2, case.down, ab, ref_d)):
            y = torch.empty((x.shape[0], proj.N), dtype=torch.float32, device="cuda")
            mlp.debug_project(which, to_dev(x), y, path=path)
            torch.cuda.synchronize()
            got = y.cpu().numpy().astype(np.float64)
            assert np.array_equal(got, ref, equal_nan=True), (path, which)
    assert mlp.decode_ctas() > 0
    g, u, o = run_split(torch, mlp, xb, ab)
    assert np.array_equal(g, ref_g, equal_nan=True)
    assert np.array_equal(u, ref_u, equal_nan=True)
    assert np.array_equal(o, ref_d, equal_nan=True)
    mlp.close()
