"""The allocation-free routed-expert entry point (qmlp_moe_m1_forward_noalloc).

Some callers cannot allocate device memory when they run the routed-expert
step: a runtime that owns the device allocator and forbids allocations from
libraries, or a program whose device memory is fixed once warm-up is over.
The entry point serves them by reading the caller's banks in place and
keeping its only scratch in a file-scope device array that every call
shares. Checked through the C ABI against the handle-based
qmlp_moe_m1_forward (and, at the array's size limit, the CPU oracle) on the
same inputs, twice in a row: the second call runs on the scratch the first
one left. This file sorts last so a stop-at-first-failure run has run every
other test.
"""
import numpy as np
import pytest

import oracle
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from helpers import bits_from_dev, compare, to_dev

pytestmark = pytest.mark.gpu

SHAPE = 4  # QMLP_ERR_SHAPE
assert q.STATUS[SHAPE] == "QMLP_ERR_SHAPE"


def _banks(torch, c, meta_bytes):
    m13 = c.w13_meta4 if meta_bytes == 4 else c.w13_meta3
    m2 = c.w2_meta4 if meta_bytes == 4 else c.w2_meta3
    dev = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (c.w13, m13, c.w2, m2)]
    return dev, q.qmlp_moe_desc(c.E, c.K, c.I, meta_bytes, *[t.data_ptr() for t in dev])


def _both(torch, c, moe, desc, x, xdt, ids_np, rw_np, topk):
    """One handle call and one allocation-free call on the same inputs."""
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    rw = torch.from_numpy(np.ascontiguousarray(rw_np, dtype=np.float32)).cuda()
    ref = torch.empty(c.K, dtype=torch.int16, device="cuda")
    got = torch.full((c.K,), 0x7E00, dtype=torch.int16, device="cuda")  # NaN until written
    moe.forward(x, xdt, ids, rw, ref, topk=topk)
    st = q.qmlp_moe_m1_forward_noalloc(desc, x, xdt, ids, rw, topk, got)
    assert st == q.QMLP_OK, q.STATUS.get(st, st)
    torch.cuda.synchronize()
    moe.check()
    return bits_from_dev(ref), bits_from_dev(got)


def test_noalloc_matches_handle_entry_point_twice(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    c = gen.gen_moe_case(gen.seed_for(4, 0), E=64, K=2560, I=160, topk=10)
    ids_all = [c.ids, gen.rotating_ids(3, n_experts=60)]
    for meta_bytes, xdt, xbits in ((4, q.DT_FP16, c.x_fp16), (3, q.DT_BF16, c.x_bf16)):
        banks_dev, desc = _banks(torch, c, meta_bytes)
        moe = q.MoeAWQ.from_case(c, meta_bytes)
        x = to_dev(xbits)
        for ids_np in ids_all:  # two calls in a row on the shared scratch
            r, g = _both(torch, c, moe, desc, x, xdt, ids_np, c.router_w, 10)
            compare(g, r, "fp16", "noalloc vs handle")
            assert np.array_equal(g, r)  # same kernels, same order: identical bits
        moe.close()


def test_noalloc_at_the_scratch_limit(cuda_available):
    """topk = 16 and I = 1024 fill the whole 16 x 1024 scratch array (its
    last row included), with an invalid and a duplicate id among the routes;
    K = 64 keeps the bank small. Bit-identical to the handle entry point,
    within tolerance of the oracle, on two calls in a row."""
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    c = gen.gen_moe_case(977, E=16, K=64, I=1024, topk=16)
    assert np.count_nonzero(c.ids == c.E) == 1 and len(set(c.ids.tolist())) == 15
    for meta_bytes, xdt, xname in ((4, q.DT_FP16, "fp16"), (3, q.DT_BF16, "bf16")):
        banks_dev, desc = _banks(torch, c, meta_bytes)
        moe = q.MoeAWQ.from_case(c, meta_bytes)
        x = to_dev(c.x_fp16 if xname == "fp16" else c.x_bf16)
        ids2 = np.roll(c.ids, 5)  # second call: the same routes in another order
        rw2 = np.roll(c.router_w, 5)
        for ids_np, rw_np in ((c.ids, c.router_w), (ids2, rw2)):
            r, g = _both(torch, c, moe, desc, x, xdt, ids_np, rw_np, 16)
            assert np.array_equal(g, r)
            ref = oracle.moe_m1_forward(c, meta_bytes, xname, ids=ids_np, rw=rw_np)["out"]
            compare(g, ref, "fp16", "noalloc vs oracle")
        moe.close()


def test_noalloc_rejects_sizes_beyond_the_scratch(cuda_available):
    """I above 1024 and topk above 16 return QMLP_ERR_SHAPE before any launch;
    the output buffer is left as it was."""
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    c = gen.gen_moe_case(978, E=16, K=64, I=1024, topk=16)
    banks_dev, desc = _banks(torch, c, 4)
    x = to_dev(c.x_fp16)
    ids = torch.zeros(32, dtype=torch.int32, device="cuda")
    rw = torch.full((32,), 1.0 / 32, dtype=torch.float32, device="cuda")
    out = torch.full((c.K,), 0x1234, dtype=torch.int16, device="cuda")
    big_i = q.qmlp_moe_desc(c.E, c.K, 2048, 4, *[t.data_ptr() for t in banks_dev])
    assert q.qmlp_moe_m1_forward_noalloc(big_i, x, q.DT_FP16, ids, rw, 16, out) == SHAPE
    assert q.qmlp_moe_m1_forward_noalloc(desc, x, q.DT_FP16, ids, rw, 17, out) == SHAPE
    torch.cuda.synchronize()
    assert np.all(bits_from_dev(out) == 0x1234)
