"""GPU parity of the routed-expert entry points at their limits, through the
C ABI: 16 routes per token (the largest top-k they accept) on the smallest
shapes they accept (K = 64, I = 32), for the one-token step and for M tokens
-- with 8-route groups (M = 3) and with 16-route groups (M = 9: 144 routes
over 16 experts). At K = 64 one of the ten K-split warps of W13 holds the
only 64-k chunk and the others add zeros; at I = 32 W2 has two k16 groups.
Each token's 16 routes are 14 distinct ids, a duplicate and an invalid id."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from helpers import bits_from_dev, compare, to_dev

pytestmark = pytest.mark.gpu

E, K, I, TOPK = 16, 64, 32, 16


@pytest.fixture(scope="module")
def torch_cuda(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    q.lib()
    return torch


def _dt(xdt):
    return q.DT_FP16 if xdt == "fp16" else q.DT_BF16


def _one_token(torch, moe, x_bits, ids, rw, xdt):
    x = to_dev(x_bits.copy())
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    d_rw = torch.from_numpy(np.ascontiguousarray(rw, dtype=np.float32)).cuda()
    out = torch.empty(K, dtype=torch.int16, device="cuda")
    moe.forward(x, _dt(xdt), d_ids, d_rw, out)
    torch.cuda.synchronize()
    moe.check()
    return bits_from_dev(out)


@pytest.mark.parametrize("meta", [4, 3])
@pytest.mark.parametrize("xdt", ["fp16", "bf16"])
def test_one_token_top16_smallest_shape(torch_cuda, meta, xdt):
    c = gen.gen_moe_case(900 + meta, E=E, K=K, I=I, topk=TOPK)
    assert c.ids.size == TOPK and np.count_nonzero(c.ids == E) == 1
    moe = q.MoeAWQ.from_case(c, meta)
    got = _one_token(torch_cuda, moe, c.x_fp16 if xdt == "fp16" else c.x_bf16, c.ids, c.router_w, xdt)
    compare(got, oracle.moe_m1_forward(c, meta, xdt)["out"], "fp16", "out")
    moe.close()


@pytest.mark.parametrize("xdt", ["fp16", "bf16"])
@pytest.mark.parametrize("M", [3, 9])
def test_tokens_top16_smallest_shape(torch_cuda, xdt, M):
    torch = torch_cuda
    tok = gen.gen_moe_tokens(950 + M, M, E=E, K=K, I=I, topk=TOPK)
    moe = q.MoeAWQ.from_case(tok.case, 4)
    moe.reserve(M)
    xb = tok.x16 if xdt == "fp16" else tok.xb
    x = to_dev(xb)
    d_ids = torch.from_numpy(np.ascontiguousarray(tok.ids)).cuda()
    d_rw = torch.from_numpy(np.ascontiguousarray(tok.rw)).cuda()
    out = torch.empty((M, K), dtype=torch.int16, device="cuda")
    moe.forward_tokens(x, _dt(xdt), d_ids, d_rw, out)
    torch.cuda.synchronize()
    moe.check()
    got = bits_from_dev(out)
    for t in range(M):
        c = replace(tok.case, x_fp16=tok.x16[t], x_bf16=tok.xb[t])
        ref = oracle.moe_m1_forward(c, 4, xdt, ids=tok.ids[t], rw=tok.rw[t])["out"]
        compare(got[t], ref, "fp16", f"token {t}")
        # the same bytes as the one-token kernels (same k splits, MMA order, router-order sum)
        assert np.array_equal(got[t], _one_token(torch, moe, xb[t], tok.ids[t], tok.rw[t], xdt)), t
    moe.close()
