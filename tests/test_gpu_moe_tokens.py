"""GPU parity of the multi-token routed-expert path (qmlp_moe_forward, M > 1)
through the C ABI. Tokens do not interact: the reference for token t is the
one-token oracle on token t's x and routes, and the grouped kernels must give
the same bytes as the one-token GPU kernels token by token (the same k
splits, MMA order and router-order sum)."""
from dataclasses import replace

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


def _dt(xdt):
    return q.DT_FP16 if xdt == "fp16" else q.DT_BF16


def run_tokens(torch, moe, tok, xdt, ids=None):
    ids = tok.ids if ids is None else ids
    x = to_dev(tok.x16 if xdt == "fp16" else tok.xb)
    d_ids = torch.from_numpy(np.ascontiguousarray(ids)).cuda()
    d_rw = torch.from_numpy(np.ascontiguousarray(tok.rw)).cuda()
    out = torch.empty((ids.shape[0], tok.case.K), dtype=torch.int16, device="cuda")
    moe.forward_tokens(x, _dt(xdt), d_ids, d_rw, out)
    torch.cuda.synchronize()
    moe.check()
    return bits_from_dev(out)


def run_one_token(torch, moe, tok, xdt, t):
    x = to_dev((tok.x16 if xdt == "fp16" else tok.xb)[t].copy())
    d_ids = torch.from_numpy(tok.ids[t].copy()).cuda()
    d_rw = torch.from_numpy(tok.rw[t].copy()).cuda()
    out = torch.empty(tok.case.K, dtype=torch.int16, device="cuda")
    moe.forward(x, _dt(xdt), d_ids, d_rw, out)
    torch.cuda.synchronize()
    moe.check()
    return bits_from_dev(out)


def oracle_tokens(tok, meta, xdt, rows, ids=None):
    ids = tok.ids if ids is None else ids
    outs = []
    for t in rows:
        c = replace(tok.case, x_fp16=tok.x16[t], x_bf16=tok.xb[t])
        outs.append(oracle.moe_m1_forward(c, meta, xdt, ids=ids[t], rw=tok.rw[t])["out"])
    return np.stack(outs)


@pytest.mark.parametrize("meta", [4, 3])
@pytest.mark.parametrize("xdt", ["fp16", "bf16"])
@pytest.mark.parametrize("M", [2, 9, 13, 37])
def test_tokens_small_bank_heavy_sharing(torch_cuda, meta, xdt, M):
    """E = 16: most experts carry many routes, so groups fill, experts spread
    over several groups and a token's duplicate shares a group with its
    original; every token also has one invalid id. Groups hold 8 routes up
    to M = 12 and 16 routes (two MMA column sets) from M = 13, where the
    M x 10 routes reach 8 per expert."""
    tok = gen.gen_moe_tokens(400 + M, M, E=16, K=512, I=160)
    moe = q.MoeAWQ.from_case(tok.case, meta)
    moe.reserve(M)
    got = run_tokens(torch_cuda, moe, tok, xdt)
    compare(got, oracle_tokens(tok, meta, xdt, range(M)), "fp16", "out")
    for t in range(M):
        assert np.array_equal(got[t], run_one_token(torch_cuda, moe, tok, xdt, t)), t
    moe.close()


@pytest.fixture(scope="module")
def big_tokens():
    # the routed-expert bank of the one-token workload (E=512, K=2560, I=160,
    # top-10) with 512 tokens: ~10 routes per expert, the prefill regime
    return gen.gen_moe_tokens(gen.seed_for(6, 0), 512)


@pytest.mark.parametrize("M", [16, 512])
def test_tokens_e512(torch_cuda, big_tokens, M):
    tok = gen.MoeTokens(big_tokens.case, big_tokens.x16[:M], big_tokens.xb[:M], big_tokens.ids[:M],
                        big_tokens.rw[:M])
    moe = q.MoeAWQ.from_case(tok.case, 4)
    moe.reserve(M)
    got = run_tokens(torch_cuda, moe, tok, "fp16")
    rng = np.random.default_rng(600 + M)
    rows = np.arange(M) if M <= 16 else np.unique(np.concatenate([[0, 1, M - 1], rng.choice(M, 29, replace=False)]))
    compare(got[rows], oracle_tokens(tok, 4, "fp16", rows), "fp16", "out")
    for t in rows[:4]:
        assert np.array_equal(got[t], run_one_token(torch_cuda, moe, tok, "fp16", t)), t
    # the same bytes every call (the grouping order inside an expert varies)
    assert np.array_equal(got, run_tokens(torch_cuda, moe, tok, "fp16"))
    moe.close()


def test_tokens_with_no_valid_route_give_zero(torch_cuda):
    tok = gen.gen_moe_tokens(450, 5, E=16, K=256, I=160)
    ids = tok.ids.copy()
    ids[1, :] = 16    # every id >= E
    ids[3, :] = -1    # every id < 0
    moe = q.MoeAWQ.from_case(tok.case, 4)
    moe.reserve(5)
    got = run_tokens(torch_cuda, moe, tok, "fp16", ids=ids)
    assert not got[1].any() and not got[3].any()
    compare(got, oracle_tokens(tok, 4, "fp16", range(5), ids=ids), "fp16", "out")
    moe.close()


def test_tokens_graph_replay_with_changing_routes(torch_cuda):
    """The routing runs on the device: a captured graph replayed after the
    ids change on the device gives the new routes' result."""
    torch = torch_cuda
    tok = gen.gen_moe_tokens(460, 12, E=32, K=512, I=160)
    moe = q.MoeAWQ.from_case(tok.case, 4)
    moe.reserve(12)
    x = to_dev(tok.x16)
    d_ids = torch.from_numpy(tok.ids.copy()).cuda()
    d_rw = torch.from_numpy(tok.rw.copy()).cuda()
    out = torch.empty((12, tok.case.K), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    moe.forward_tokens(x, q.DT_FP16, d_ids, d_rw, out, stream=s)  # warm (outside capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.forward_tokens(x, q.DT_FP16, d_ids, d_rw, out, stream=s)
    rng = np.random.default_rng(461)
    for call in range(3):
        # fresh routes in [-2, 40): duplicates, and ids < 0 or >= 32 invalid
        ids = rng.integers(-2, 40, size=tok.ids.shape).astype(np.int32)
        d_ids.copy_(torch.from_numpy(ids))
        g.replay()
        torch.cuda.synchronize()
        moe.check()
        compare(bits_from_dev(out), oracle_tokens(tok, 4, "fp16", range(12), ids=ids), "fp16", f"replay {call}")
    moe.close()


def test_tokens_argument_rejection(torch_cuda):
    torch = torch_cuda
    tok = gen.gen_moe_tokens(470, 4, E=16, K=256, I=160)
    moe = q.MoeAWQ.from_case(tok.case, 4)
    L = q.lib()
    cs = torch.cuda.current_stream().cuda_stream
    x = to_dev(tok.x16)
    ids = torch.from_numpy(tok.ids.copy()).cuda()
    rw = torch.from_numpy(tok.rw.copy()).cuda()
    out = torch.full((4, tok.case.K), 0x1234, dtype=torch.int16, device="cuda")
    args = lambda M, o=out.data_ptr(), xx=x.data_ptr(): (moe.h, xx, q.DT_FP16, ids.data_ptr(), rw.data_ptr(), 10, M,
                                                        o, cs)
    assert L.qmlp_moe_forward(*args(4)) == 4   # not reserved yet: max_tokens = 1
    moe.reserve(4)
    assert L.qmlp_moe_forward(*args(5)) == 4   # M > max_tokens
    assert L.qmlp_moe_forward(*args(0)) == 4   # M = 0
    assert L.qmlp_moe_forward(*args(4, o=out.data_ptr() + 2)) == 2   # misaligned out
    assert L.qmlp_moe_forward(*args(4, o=x.data_ptr())) == 3         # out aliases x
    assert L.qmlp_moe_forward(moe.h, x.data_ptr(), q.DT_FP16, ids.data_ptr(), rw.data_ptr(), 17, 4,
                              out.data_ptr(), cs) == 4                # topk > 16
    assert L.qmlp_moe_forward(moe.h, x.data_ptr(), 9, ids.data_ptr(), rw.data_ptr(), 10, 4,
                              out.data_ptr(), cs) == 1                # bad dtype
    assert L.qmlp_moe_reserve(moe.h, 0, cs) == 4
    torch.cuda.synchronize()
    assert bool((out == 0x1234).all())
    moe.close()
