"""GPU parity of the decode kernel that partitions the intermediate
dimension across CTAs (each CTA: gate/up for its slice of I, then the down
projection over that slice; partial outputs added in a fixed order, after a
grid barrier inside the kernel for one NVFP4 token, else by a reduce kernel
launched after it), against the CPU oracle."""
import numpy as np
import pytest

import oracle
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from helpers import bits_from_dev, compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    q.lib()
    return torch


def run_forward(torch, mlp, x_bits, path=q.PATH_GEMV):
    M = x_bits.shape[0]
    out = torch.empty((M, mlp.K), dtype=torch.int16, device="cuda")
    act = torch.empty((M, mlp.I), dtype=torch.int16, device="cuda")
    mlp.forward_debug(to_dev(x_bits), act, out, path=path)
    torch.cuda.synchronize()
    mlp.check()
    return bits_from_dev(out), bits_from_dev(act)


def sm_count(torch):
    return torch.cuda.get_device_properties(0).multi_processor_count


def test_plan_of_the_27b_shape(torch_cuda):
    """K=5120, I=17408 on a 152-SM GB300: 136 CTAs x 8 gate/up row tiles."""
    if sm_count(torch_cuda) != 152:
        pytest.skip("the expected partition is for a 152-SM device")
    case = gen.workload_case("dense_nvfp4_decode", 0)
    mlp = q.QuantMLP.from_case(case)
    assert mlp.decode_ctas() == 136
    mlp.close()


# (K, I): tiles of 4 CTA-local gate/up tiles spanning 4 warps each (1024,
# 7680 -> 120 CTAs); down tiles split at warp boundaries with padding records
# (1536, 23040 -> 120 CTAs, 3 down chunks per CTA, 20 records per warp).
SHAPES = [(1024, 7680), (1536, 23040)]


@pytest.mark.parametrize("fmt,M", [("nvfp4", 1), ("nvfp4", 4), ("fp8", 1), ("fp8", 8)])
def test_small_mlp_runs_on_a_few_ctas(torch_cuda, fmt, M):
    """K=256, I=512 (~0.2 MB of weights): fixed costs bound the call, so the
    partition uses a few CTAs (NVFP4: 4 of 8 gate/up row tiles each, FP8: 8
    of 4); both reduction schedules against the oracle."""
    case = gen.gen_dense_case(fmt, 256, 512, M, seed=340 + M)
    mlp = q.QuantMLP.from_case(case)
    assert mlp.decode_ctas() == (4 if fmt == "nvfp4" else 8)
    out, act = run_forward(torch_cuda, mlp, case.x)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    mlp.close()


@pytest.mark.parametrize("K,I", SHAPES)
@pytest.mark.parametrize("fmt,M", [("nvfp4", 1), ("nvfp4", 2), ("nvfp4", 3), ("nvfp4", 8), ("fp8", 1), ("fp8", 2),
                                   ("fp8", 4), ("fp8", 5)])
def test_split_parity(torch_cuda, K, I, fmt, M):
    """Every instance of the decode kernel: one token (each format's
    schedule), the token counts fixed at compile time (2, 4, 8) and the
    general one (3, 5)."""
    case = gen.gen_dense_case(fmt, K, I, M, seed=310 + M + K // 512)
    mlp = q.QuantMLP.from_case(case)
    if mlp.decode_ctas() == 0:
        pytest.skip("no I partition for this shape on this device")
    out, act = run_forward(torch_cuda, mlp, case.x)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    out2, act2 = run_forward(torch_cuda, mlp, case.x)
    assert np.array_equal(out, out2) and np.array_equal(act, act2)
    mlp.close()


def test_split_many_back_to_back_calls(torch_cuda):
    """200 back-to-back calls (each call's streaming CTAs start while the
    previous call's reduce kernel runs) give the same bits as the first,
    with changing inputs in between."""
    torch = torch_cuda
    K, I = SHAPES[0]
    case = gen.gen_dense_case("nvfp4", K, I, 2, seed=320)
    mlp = q.QuantMLP.from_case(case)
    if mlp.decode_ctas() == 0:
        pytest.skip("no I partition for this shape on this device")
    first, _ = run_forward(torch, mlp, case.x)
    x2 = gen.gen_x_only(321, 2, K)
    xd, x2d = to_dev(case.x), to_dev(x2)
    out = torch.empty((2, K), dtype=torch.int16, device="cuda")
    for i in range(200):
        mlp.forward(x2d if i % 2 else xd, out)
    torch.cuda.synchronize()
    mlp.check()
    last, _ = run_forward(torch, mlp, case.x)
    assert np.array_equal(first, last)
    mlp.close()


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M", [1, 3])
def test_split_host_buffers_match_device(torch_cuda, pinned, M):
    """qmlp_forward_host on the I-partitioned kernel: pinned buffers are read
    and written in place by the kernel (one token: the compact staging reads
    x in host memory), pageable ones go through the staging copies; both give
    the device-buffer result bit for bit."""
    torch = torch_cuda
    K, I = SHAPES[0]
    case = gen.gen_dense_case("nvfp4", K, I, M, seed=330 + M)
    mlp = q.QuantMLP.from_case(case)
    if mlp.decode_ctas() == 0:
        pytest.skip("no I partition for this shape on this device")
    dev, _ = run_forward(torch, mlp, case.x)
    xh = torch.from_numpy(case.x.view(np.int16).copy())
    oh = torch.zeros((M, K), dtype=torch.int16)
    if pinned:
        xh, oh = xh.pin_memory(), oh.pin_memory()
    mlp.forward_host(xh, oh)
    assert np.array_equal(oh.numpy().view(np.uint16), dev)
    mlp.close()


@pytest.mark.parametrize("M", [9, 13, 16])
def test_fp8_sixteen_token_launch(torch_cuda, M):
    """FP8 at 9..16 tokens on the 27B-class shape: one launch of the
    I-partitioned kernel with two 8-token column tiles and x staged in two
    halves (the second tile ragged below 16 tokens); every row against the
    oracle, the same bytes on a second call, and the automatic path is this
    kernel (not the GEMM)."""
    case = gen.gen_dense_case("fp8", gen.DENSE_K, gen.DENSE_I, M, seed=330 + M)
    mlp = q.QuantMLP.from_case(case, max_M=16)
    out, act = run_forward(torch_cuda, mlp, case.x, path=q.PATH_AUTO)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    out2, _ = run_forward(torch_cuda, mlp, case.x, path=q.PATH_AUTO)
    assert np.array_equal(out, out2)
    gemv, _ = run_forward(torch_cuda, mlp, case.x, path=q.PATH_GEMV)
    assert np.array_equal(out, gemv)
    mlp.close()
