"""Tensor-parallel shards over the intermediate dimension, all on one GPU
(vllm.cpp issue "tp>1 fp8w tail-MLP shard host-dequantizes every layer",
"Proposed fix": gate/up row slices, down column slices, one sum over the
ranks). N = 2, 4 and 8 shard handles of the 27B-class layer each write their
fp32 partial into slot r of one rank-major buffer -- what the all-gather of a
multi-GPU run delivers -- and qmlp_shard_combine adds them in rank order,
applies the down factor and rounds to bf16. The result is compared with the
oracle of the WHOLE layer (the shards change only the fp32 summation order),
through the C ABI."""
import numpy as np
import pytest

import oracle
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from weight_quantized_swiglu_gb300 import tp
from helpers import bits_from_dev, compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    q.lib()
    return torch


_REF = {}


def reference(case, key):
    if key not in _REF:
        _REF[key] = oracle.dense_forward(case)["out"]
    return _REF[key]


def run_shards(torch, case, n, max_M=None):
    M = case.M
    x = to_dev(case.x)
    partials = torch.full((n, M, case.K), float("nan"), dtype=torch.float32, device="cuda")
    shards = [q.QuantMLP.from_case(case, max_M=max_M, shard=(r, n)) for r in range(n)]
    for r, s in enumerate(shards):
        assert (s.rank, s.nranks, s.I) == (r, n, case.I // n)
        assert tp.shard_range(case.I, r, n) == (r * s.I, (r + 1) * s.I)
        s.forward_partial(x, partials[r])
    out = torch.empty((M, case.K), dtype=torch.int16, device="cuda")
    shards[0].combine(partials, out)
    out2 = torch.empty_like(out)
    shards[-1].combine(partials, out2)  # any rank's handle: the same bytes
    torch.cuda.synchronize()
    for s in shards:
        s.check()
        s.close()
    assert np.array_equal(bits_from_dev(out), bits_from_dev(out2))
    return bits_from_dev(out), partials


@pytest.mark.parametrize("n", [2, 4, 8])
@pytest.mark.parametrize("variant", [0, 1])
def test_nvfp4_decode_shards(torch_cuda, n, variant):
    """M = 1 and 4 tokens: at n = 2 each shard runs the I-partitioned decode
    kernel (fp32 output mode); at n = 4 and 8 the shard's slice has no
    partition and runs the stream-K kernels with the raw down epilogue."""
    case = gen.workload_case("dense_nvfp4_decode", variant)
    got, _ = run_shards(torch_cuda, case, n)
    compare(got, reference(case, ("nvfp4", variant)), what=f"n={n}")


@pytest.mark.parametrize("n,variant", [(2, 0), (4, 0), (2, 1)])
def test_fp8_shards(torch_cuda, n, variant):
    """FP8 per-channel: the down factor is the full per-output-channel scale
    vector (down rows are not sharded); M = 16 runs each shard's GEMM with
    the raw epilogue."""
    case = gen.workload_case("dense_fp8_decode", variant)
    got, _ = run_shards(torch_cuda, case, n)
    compare(got, reference(case, ("fp8", variant)), what=f"n={n}")


def test_prefill_shards_on_the_gemm(torch_cuda):
    """M = 200 tokens (two token tiles, the second ragged) on the tensor-core
    GEMM of each of two shards."""
    case = gen.gen_dense_case("nvfp4", gen.DENSE_K, gen.DENSE_I, 200, seed=320)
    got, _ = run_shards(torch_cuda, case, 2)
    rows = np.arange(0, 200, 7, dtype=np.int32)
    ref = oracle.dense_forward(case, rows=rows)["out"]
    compare(got[rows], ref, what="prefill n=2")


def test_shard_partials_sum_to_the_whole_layer_partial(torch_cuda):
    """The ranks' fp32 partials add up (in fp64, any order) to the whole
    layer's unscaled down output: a one-rank 'shard' of the same layer. The
    two layouts split gate/up tiles between warps at other k, so a few act
    values round to the other bf16 neighbour (one ulp, 2^-8 relative): the
    sums agree to ~1e-5, checked at 2e-4."""
    torch = torch_cuda
    case = gen.workload_case("dense_nvfp4_decode", 0)
    _, parts = run_shards(torch, case, 2)
    _, whole = run_shards(torch, case, 1)
    p = parts.cpu().numpy().astype(np.float64)
    w = whole.cpu().numpy().astype(np.float64)[0]
    assert np.linalg.norm(p.sum(axis=0) - w) / np.linalg.norm(w) < 2e-4


def test_shard_argument_rejection(torch_cuda):
    case = gen.workload_case("tiny_nvfp4", 0)
    for rank, n in ((2, 2), (-1, 2), (0, 0)):
        with pytest.raises(q.QmlpError) as e:
            q.QuantMLP.from_case(case, shard=(rank, n))
        assert e.value.status == 1  # QMLP_ERR_INVALID_ARG
    with pytest.raises(q.QmlpError) as e:
        q.QuantMLP.from_case(case, shard=(0, 3))  # 512 does not split in 3
    assert e.value.status == 4  # QMLP_ERR_SHAPE
    s = q.QuantMLP.from_case(case, shard=(0, 2))
    torch = torch_cuda
    parts = torch.zeros((2, 1, case.K), dtype=torch.float32, device="cuda")
    out = torch.empty((1, case.K), dtype=torch.int16, device="cuda")
    assert q.qmlp_shard_combine(s.h, parts, 3, 1, out) == 1  # wrong rank count
    assert q.qmlp_shard_combine(s.h, parts, 2, 1, parts) == 3  # out overlaps the partials
    s.close()
