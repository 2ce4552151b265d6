"""The allocation-free routed-expert entry point (qmlp_moe_m1_forward_noalloc).

It serves callers that cannot allocate device memory when they run the step;
its scratch is a file-scope device array shared by all calls. Checked through
the C ABI against the handle-based qmlp_moe_m1_forward on the same inputs,
twice in a row (the second call runs on the scratch the first one left).
This file sorts last so a stop-at-first-failure run has run every other test.
"""
import numpy as np
import pytest

import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from helpers import bits_from_dev, compare, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_handle_entry_point_twice(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    c = gen.gen_moe_case(gen.seed_for(4, 0), E=64, K=2560, I=160, topk=10)
    ids_all = [c.ids, gen.rotating_ids(3, n_experts=60)]
    for meta_bytes, xdt, xbits in ((4, q.DT_FP16, c.x_fp16), (3, q.DT_BF16, c.x_bf16)):
        m13 = c.w13_meta4 if meta_bytes == 4 else c.w13_meta3
        m2 = c.w2_meta4 if meta_bytes == 4 else c.w2_meta3
        banks_dev = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (c.w13, m13, c.w2, m2)]
        desc = q.qmlp_moe_desc(c.E, c.K, c.I, meta_bytes, *[t.data_ptr() for t in banks_dev])
        moe = q.MoeAWQ.from_case(c, meta_bytes)
        x = to_dev(xbits)
        rw = torch.from_numpy(c.router_w).cuda()
        for ids_np in ids_all:  # two calls in a row on the shared scratch
            ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
            ref = torch.empty(c.K, dtype=torch.int16, device="cuda")
            got = torch.full((c.K,), 0x7E00, dtype=torch.int16, device="cuda")
            moe.forward(x, xdt, ids, rw, ref)
            st = q.qmlp_moe_m1_forward_noalloc(desc, x, xdt, ids, rw, 10, got)
            assert st == q.QMLP_OK, q.STATUS.get(st, st)
            torch.cuda.synchronize()
            r, g = bits_from_dev(ref), bits_from_dev(got)
            compare(g, r, "fp16", "noalloc vs handle")
            assert np.array_equal(g, r)  # same kernels, same order: identical bits
        moe.close()
        # sizes beyond the scratch array are rejected before any launch
        big = q.qmlp_moe_desc(c.E, c.K, 2048, meta_bytes, *[t.data_ptr() for t in banks_dev])
        assert q.qmlp_moe_m1_forward_noalloc(big, x, xdt, ids, rw, 10, got) == 4
        assert q.qmlp_moe_m1_forward_noalloc(desc, x, xdt, ids, rw, 17, got) == 4
