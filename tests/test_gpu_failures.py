"""Failure detection without a GPU fault (vllm.cpp issue "tp>1 fp8w tail-MLP
shard ...", "Risks": a failure returns a status, never a silent fallback).

* Allocation failures, injected on the host (QMLP_FAULT_INJECT=alloc or
  alloc:N): create returns QMLP_ERR_OOM, hands back no handle and releases
  every allocation it had made.
* Launch failures, injected on the host (QMLP_FAULT_INJECT=launch): the
  forward calls return QMLP_ERR_CUDA, launch nothing and leave the output as
  it was.
* Bounded waits that run out: a test-only knob (qmlp_debug_set_wait) gives the
  decode and GEMM kernels a 20 ms wait limit and makes their producers
  withhold their last weight step, so the consumers' waits expire. The
  kernels record it and leave normally (no trap, no hang); qmlp_check reports
  QMLP_ERR_DEVICE_TIMEOUT once, and the next normal call on the same handle
  is bit-identical to one made before the failure.
"""
import os

import numpy as np
import pytest

import oracle
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from helpers import bits_from_dev, compare, to_dev

pytestmark = pytest.mark.gpu

OOM, CUDA, TIMEOUT = 6, 7, 8
assert (q.STATUS[OOM], q.STATUS[CUDA], q.STATUS[TIMEOUT]) == ("QMLP_ERR_OOM", "QMLP_ERR_CUDA",
                                                                "QMLP_ERR_DEVICE_TIMEOUT")


@pytest.fixture(scope="module")
def torch_cuda(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    q.lib()
    return torch


class inject:
    """QMLP_FAULT_INJECT set for the duration of a with-block."""

    def __init__(self, what):
        self.what = what

    def __enter__(self):
        os.environ["QMLP_FAULT_INJECT"] = self.what

    def __exit__(self, *exc):
        os.environ.pop("QMLP_FAULT_INJECT", None)


def free_bytes(torch):
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def test_allocation_failure_returns_oom_and_leaks_nothing(torch_cuda):
    """The 27B-class shape: the first two allocations (tens of MB of weight
    copies) succeed before the injected failure in most of these runs, and
    each failed create must give them back."""
    torch = torch_cuda
    case = gen.workload_case("dense_nvfp4_decode", 0)
    before = free_bytes(torch)
    for what in ["alloc"] + [f"alloc:{n}" for n in (1, 2, 3, 5, 8, 12)] * 3:
        with inject(what):
            with pytest.raises(q.QmlpError) as e:
                q.QuantMLP.from_case(case)
        assert e.value.status == OOM, what
    assert free_bytes(torch) >= before - (64 << 20)
    # the same for the routed-expert handle
    c = gen.gen_moe_case(401, E=32)
    before = free_bytes(torch)
    for n in (1, 2, 3, 4, 5, 6) * 3:
        with inject(f"alloc:{n}"):
            with pytest.raises(q.QmlpError) as e:
                q.MoeAWQ.from_case(c, 4)
        assert e.value.status == OOM
    assert free_bytes(torch) >= before - (64 << 20)
    # and once the variable is gone, create works
    q.QuantMLP.from_case(case).close()


def test_launch_failure_launches_nothing(torch_cuda):
    torch = torch_cuda
    case = gen.workload_case("tiny_nvfp4", 1)
    mlp = q.QuantMLP.from_case(case, max_M=64)
    x = to_dev(case.x)
    out = torch.full((case.M, case.K), 0x1357, dtype=torch.int16, device="cuda")
    y = torch.full((case.M, case.I), 7.0, dtype=torch.float32, device="cuda")
    c = gen.gen_moe_case(402, E=16)
    moe = q.MoeAWQ.from_case(c, 4)
    mx = to_dev(c.x_fp16)
    ids = torch.from_numpy(c.ids).cuda()
    rw = torch.from_numpy(c.router_w).cuda()
    mout = torch.full((c.K,), 0x1357, dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    with inject("launch"):
        for path in (q.PATH_AUTO, q.PATH_GEMV, q.PATH_GEMM):
            assert q.qmlp_forward_path(mlp.h, path, x, case.M, out) == CUDA
        assert q.qmlp_debug_project(mlp.h, 0, q.PATH_AUTO, x, case.M, y) == CUDA
        assert q.qmlp_moe_m1_forward(moe.h, mx, q.DT_FP16, ids, rw, c.topk, mout) == CUDA
    torch.cuda.synchronize()
    assert np.all(bits_from_dev(out) == 0x1357)
    assert np.all(y.cpu().numpy() == 7.0)
    assert np.all(bits_from_dev(mout) == 0x1357)
    mlp.forward(x, out)  # nothing was left half-done
    torch.cuda.synchronize()
    mlp.check()
    compare(bits_from_dev(out), oracle.dense_forward(case)["out"], what="after")
    mlp.close()
    moe.close()


def _timeout_then_recover(torch, mlp, x_bits, path):
    M = x_bits.shape[0]
    x = to_dev(x_bits)
    good = torch.empty((M, mlp.K), dtype=torch.int16, device="cuda")
    mlp.forward(x, good, path=path)
    torch.cuda.synchronize()
    mlp.check()
    # 20 ms limit, last weight step withheld: every consumer's wait for it runs out
    mlp.set_wait(20_000_000, True)
    bad = torch.empty_like(good)
    mlp.forward(x, bad, path=path)  # the launch itself succeeds
    with pytest.raises(q.QmlpError) as e:
        mlp.check()
    assert e.value.status == TIMEOUT
    mlp.check()  # reported once, then cleared
    # normal waits again: the same bytes as before the failure
    mlp.set_wait(0, False)
    again = torch.empty_like(good)
    for _ in range(2):
        mlp.forward(x, again, path=path)
    torch.cuda.synchronize()
    mlp.check()
    assert np.array_equal(bits_from_dev(again), bits_from_dev(good))


@pytest.mark.parametrize("fmt,variant", [("nvfp4", 0), ("nvfp4", 1), ("fp8", 0)])
def test_decode_kernel_wait_runs_out_and_recovers(torch_cuda, fmt, variant):
    """The single-launch decode kernel: one NVFP4 token (in-kernel ticket
    barrier, which every CTA still passes exactly once), four NVFP4 tokens and
    one FP8 token (separate reduce kernel)."""
    name = "dense_nvfp4_decode" if fmt == "nvfp4" else "dense_fp8_decode"
    case = gen.workload_case(name, variant)
    mlp = q.QuantMLP.from_case(case)
    assert mlp.decode_ctas() > 0
    _timeout_then_recover(torch_cuda, mlp, case.x, q.PATH_AUTO)
    mlp.close()


@pytest.mark.parametrize("path", [q.PATH_GEMM, q.PATH_GEMM_PAIR, q.PATH_GEMM_DQ])
@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_gemm_wait_runs_out_and_recovers(torch_cuda, fmt, path):
    """The tensor-core GEMM (both launches of a forward), single-CTA, on CTA
    pairs and dequantise-once: the MMA and decoder warps give up on the
    withheld step, raise the CTA's abort flag, the other roles leave their
    loops, issued MMAs are waited for, both CTAs of a pair meet at the
    cluster barrier and TMEM is freed."""
    case = gen.gen_dense_case(fmt, 1024, 2048, 300, seed=403)
    mlp = q.QuantMLP.from_case(case, max_M=768 if path == q.PATH_GEMM_DQ else None)
    _timeout_then_recover(torch_cuda, mlp, case.x, path)
    mlp.close()
