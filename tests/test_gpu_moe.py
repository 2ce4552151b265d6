"""GPU parity of the routed-expert AWQ int4 g32 M=1 path against the CPU
oracle, through the C ABI: the E=512/top-10 workload with an invalid and a
duplicate id, both metadata layouts, fp16 and bf16 x, per-stage checks,
one-hot decode exactness, CUDA-graph replay with changing ids, rejection."""
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


@pytest.fixture(scope="module")
def big_case():
    return gen.gen_moe_case(gen.seed_for(4, 0))


def dev_inputs(torch, c, x_dtype, ids=None, rw=None):
    x = to_dev(c.x_fp16 if x_dtype == "fp16" else c.x_bf16)
    ids = torch.from_numpy(np.ascontiguousarray(c.ids if ids is None else ids, dtype=np.int32)).cuda()
    rw = torch.from_numpy(np.ascontiguousarray(c.router_w if rw is None else rw, dtype=np.float32)).cuda()
    return x, ids, rw


def run_stages(torch, moe, c, x_dtype, ids=None, rw=None):
    x, ids_d, rw_d = dev_inputs(torch, c, x_dtype, ids, rw)
    topk = ids_d.shape[0]
    out = torch.empty(c.K, dtype=torch.int16, device="cuda")
    gu = torch.zeros((topk, 2 * c.I), dtype=torch.int16, device="cuda")
    act = torch.zeros((topk, c.I), dtype=torch.int16, device="cuda")
    y = torch.zeros((topk, c.K), dtype=torch.int16, device="cuda")
    xdt = q.DT_FP16 if x_dtype == "fp16" else q.DT_BF16
    moe.debug_stages(x, xdt, ids_d, rw_d, out, gu, act, y)
    torch.cuda.synchronize()
    moe.check()
    return {k: bits_from_dev(v) for k, v in (("out", out), ("gu", gu), ("act", act), ("y", y))}


@pytest.mark.parametrize("meta_bytes,x_dtype", [(4, "fp16"), (3, "fp16"), (4, "bf16"), (3, "bf16")])
def test_parity_moe_e512_top10(torch_cuda, big_case, meta_bytes, x_dtype):
    c = big_case
    moe = q.MoeAWQ.from_case(c, meta_bytes)
    got = run_stages(torch_cuda, moe, c, x_dtype)
    ref = oracle.moe_m1_forward(c, meta_bytes, x_dtype, want_stages=True)
    valid = ref["valid"]
    assert valid.sum() == c.topk - 1  # one invalid id in the workload
    compare(got["out"], ref["out"], "fp16", "out")
    compare(got["gu"][valid], ref["gu"][valid], "fp16", "gate/up")
    compare(got["act"][valid], ref["act"][valid], "fp16", "act")
    compare(got["y"][valid], ref["y"][valid], "fp16", "y")
    moe.close()


def test_stage_pairs_within_fp16_rounding_bound(torch_cuda, big_case):
    """Each stage against fp64 given the GPU's own previous-stage output: the
    GPU value must be within half an fp16 ulp plus an fp32 accumulation bound
    of the exact value (1Cat-vLLM PR, "Test plan and results": FP64 stage
    checks with an explicit FP16 rounding allowance)."""
    c = big_case
    moe = q.MoeAWQ.from_case(c, 4)
    got = run_stages(torch_cuda, moe, c, "fp16")
    x = oracle.fp16_bits_to_f64(c.x_fp16)
    for r, e in enumerate(c.ids):
        if not (0 <= e < c.E):
            continue
        w13 = oracle.awq_decode(c.w13, c.w13_meta4, 4, int(e))
        h = w13 @ x
        # fp32 sum of 8*ceil(K/256) terms per lane, then a 5-step butterfly
        bound = np.abs(w13) @ np.abs(x) * (8 * -(-c.K // 256) + 5) * 2.0 ** -24
        gu = oracle.fp16_bits_to_f64(got["gu"][r])
        ulp = np.spacing(np.maximum(np.abs(h), np.abs(gu)).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(gu - h) <= 0.5 * ulp + bound + 1e-12), r
        w2 = oracle.awq_decode(c.w2, c.w2_meta4, 4, int(e))
        a = oracle.fp16_bits_to_f64(got["act"][r])
        yv = w2 @ a
        yb = np.abs(w2) @ np.abs(a) * (8 * -(-c.I // 256) + 5) * 2.0 ** -24
        ygot = oracle.fp16_bits_to_f64(got["y"][r])
        yulp = np.spacing(np.maximum(np.abs(yv), np.abs(ygot)).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(ygot - yv) <= 0.5 * yulp + yb + 1e-12), r
    moe.close()


def test_one_hot_decode_is_bit_exact(torch_cuda):
    torch = torch_cuda
    c = gen.gen_moe_case(401, E=4, K=2560, I=160, topk=1, n_invalid=0, n_dup=0)
    for mb in (4, 3):
        moe = q.MoeAWQ.from_case(c, mb)
        m13 = c.w13_meta4 if mb == 4 else c.w13_meta3
        ref = oracle.awq_decode(c.w13, m13, mb, 2)
        for k in (0, 31, 32, 2559):
            x = np.zeros(c.K, dtype=np.float16)
            x[k] = 1.0
            c1 = gen.MoeCase(**{**c.__dict__, "x_fp16": x.view(np.uint16)})
            got = run_stages(torch, moe, c1, "fp16", ids=np.array([2], np.int32), rw=np.array([1.0], np.float32))
            assert np.array_equal(oracle.fp16_bits_to_f64(got["gu"][0]), ref[:, k]), (mb, k)
        moe.close()


def test_invalid_and_duplicate_routes(torch_cuda, big_case):
    torch = torch_cuda
    c = big_case
    moe = q.MoeAWQ.from_case(c, 4)
    ids = np.array([7, 7, 511, -3, 512, 100], np.int32)
    rw = np.array([0.3, 0.1, 0.2, 0.15, 0.15, 0.1], np.float32)
    got = run_stages(torch, moe, c, "fp16", ids, rw)
    assert np.array_equal(got["y"][0], got["y"][1])  # duplicate keeps identical stage outputs
    ref = oracle.moe_m1_forward(c, 4, "fp16", ids=ids, rw=rw)
    compare(got["out"], ref["out"], "fp16", "dup/invalid")
    # dropping the invalid routes changes nothing (bit-identical)
    keep = np.array([0, 1, 2, 5])
    got2 = run_stages(torch, moe, c, "fp16", ids[keep], rw[keep])
    assert np.array_equal(got["out"], got2["out"])
    moe.close()


def test_4b_and_3b_layouts_bit_identical(torch_cuda, big_case):
    c = big_case
    a = q.MoeAWQ.from_case(c, 4)
    b = q.MoeAWQ.from_case(c, 3)
    ga = run_stages(torch_cuda, a, c, "fp16")
    gb = run_stages(torch_cuda, b, c, "fp16")
    for k in ("out", "gu", "act", "y"):
        assert np.array_equal(ga[k], gb[k]), k
    a.close()
    b.close()


def test_graph_replay_with_changing_ids_and_weights(torch_cuda, big_case):
    torch = torch_cuda
    c = big_case
    moe = q.MoeAWQ.from_case(c, 4)
    x, ids, rw = dev_inputs(torch, c, "fp16")
    out = torch.empty(c.K, dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.forward(x, q.DT_FP16, ids, rw, out, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.forward(x, q.DT_FP16, ids, rw, out, stream=s)
    for call in (0, 7, 40):
        nid = gen.rotating_ids(call)
        nrw = np.full(10, 0.1, np.float32)
        ids.copy_(torch.from_numpy(nid).cuda())
        rw.copy_(torch.from_numpy(nrw).cuda())
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.moe_m1_forward(c, 4, "fp16", ids=nid, rw=nrw)
        compare(bits_from_dev(out), ref["out"], "fp16", f"replay {call}")
    moe.close()


def test_moe_argument_rejection(torch_cuda, big_case):
    torch = torch_cuda
    c = big_case
    moe = q.MoeAWQ.from_case(c, 4)
    x, ids, rw = dev_inputs(torch, c, "fp16")
    out = torch.full((c.K,), 0x1234, dtype=torch.int16, device="cuda")
    L = q.lib()
    cs = torch.cuda.current_stream().cuda_stream
    raw = torch.zeros(c.K + 16, dtype=torch.int16, device="cuda")
    assert L.qmlp_moe_m1_forward(moe.h, raw.data_ptr() + 2, 2, ids.data_ptr(), rw.data_ptr(), 10,
                                 out.data_ptr(), cs) == 2
    assert L.qmlp_moe_m1_forward(moe.h, x.data_ptr(), 2, ids.data_ptr(), rw.data_ptr(), 10,
                                 x.data_ptr(), cs) == 3
    assert L.qmlp_moe_m1_forward(moe.h, x.data_ptr(), 2, ids.data_ptr(), rw.data_ptr(), 17,
                                 out.data_ptr(), cs) == 4
    assert L.qmlp_moe_m1_forward(moe.h, x.data_ptr(), 9, ids.data_ptr(), rw.data_ptr(), 10,
                                 out.data_ptr(), cs) == 1
    assert L.qmlp_moe_m1_forward(moe.h, x.data_ptr(), 2, None, rw.data_ptr(), 10, out.data_ptr(), cs) == 1
    torch.cuda.synchronize()
    assert bool((out == 0x1234).all())
    moe.close()
