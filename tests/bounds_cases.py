"""Workloads run through the C ABI by the index-check test: once with the
default library (in the test process) and once with the checking build
(libqmlp_bounds.so, in a child process that sets QMLP_LIB). Every kernel
family runs at least once: the single-launch decode kernel under each of its
end-of-call schedules, the stream-K stage kernel, the tensor-core GEMM
(single-CTA, split-K, CTA-pair and dequantise-once), the one-token and grouped routed-expert
kernels (handle and allocation-free entry points) and the tensor-parallel
combine. Outputs are returned as raw bytes, so the two builds can be compared
bit for bit; with the checking build each case also records what
qmlp_debug_bounds reported after it.

Run as a script (the child): python bounds_cases.py OUT.npz
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import weight_quantized_swiglu_gb300 as q  # noqa: E402
from weight_quantized_swiglu_gb300 import inputs as gen  # noqa: E402


def _dev(torch, a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def _bytes(t):
    return t.detach().cpu().contiguous().numpy().view(np.uint8).copy()


def _dense(torch, case, path=q.PATH_AUTO, max_M=None, stages=False):
    mlp = q.QuantMLP.from_case(case, max_M=max_M)
    x = _dev(torch, case.x)
    out = torch.empty((case.M, case.K), dtype=torch.int16, device="cuda")
    if stages:
        mlp.forward_stage(0, x, None, case.M)
        mlp.forward_stage(1, None, out, case.M)
    else:
        for _ in range(2):  # a second call: the per-call counters and tags move on
            mlp.forward(x, out, path=path)
    torch.cuda.synchronize()
    mlp.check()
    mlp.close()
    return _bytes(out)


def _moe(torch, c, meta_bytes):
    moe = q.MoeAWQ.from_case(c, meta_bytes)
    x = _dev(torch, c.x_fp16)
    ids = torch.from_numpy(np.ascontiguousarray(c.ids)).cuda()
    rw = torch.from_numpy(np.ascontiguousarray(c.router_w)).cuda()
    out = torch.empty(c.K, dtype=torch.int16, device="cuda")
    moe.forward(x, q.DT_FP16, ids, rw, out)
    torch.cuda.synchronize()
    moe.check()
    moe.close()
    return _bytes(out)


def _noalloc(torch, c):
    banks = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (c.w13, c.w13_meta4, c.w2, c.w2_meta4)]
    desc = q.qmlp_moe_desc(c.E, c.K, c.I, 4, *[t.data_ptr() for t in banks])
    x = _dev(torch, c.x_fp16)
    ids = torch.from_numpy(np.ascontiguousarray(c.ids)).cuda()
    rw = torch.from_numpy(np.ascontiguousarray(c.router_w)).cuda()
    out = torch.empty(c.K, dtype=torch.int16, device="cuda")
    st = q.qmlp_moe_m1_forward_noalloc(desc, x, q.DT_FP16, ids, rw, c.topk, out)
    assert st == q.QMLP_OK, q.STATUS.get(st, st)
    torch.cuda.synchronize()
    return _bytes(out)


def _tokens(torch, M):
    tok = gen.gen_moe_tokens(gen.seed_for(6, 0), M)
    moe = q.MoeAWQ.from_case(tok.case, 4)
    moe.reserve(M)
    x = _dev(torch, tok.x16)
    ids = torch.from_numpy(np.ascontiguousarray(tok.ids)).cuda()
    rw = torch.from_numpy(np.ascontiguousarray(tok.rw)).cuda()
    out = torch.empty((M, tok.case.K), dtype=torch.int16, device="cuda")
    moe.forward_tokens(x, q.DT_FP16, ids, rw, out)
    torch.cuda.synchronize()
    moe.check()
    moe.close()
    return _bytes(out)


def _shards(torch, case, n):
    x = _dev(torch, case.x)
    partials = torch.zeros((n, case.M, case.K), dtype=torch.float32, device="cuda")
    shards = [q.QuantMLP.from_case(case, shard=(r, n)) for r in range(n)]
    for r, s in enumerate(shards):
        s.forward_partial(x, partials[r])
    out = torch.empty((case.M, case.K), dtype=torch.int16, device="cuda")
    shards[0].combine(partials, out)
    torch.cuda.synchronize()
    for s in shards:
        s.check()
        s.close()
    return _bytes(out)


def cases():
    """(name, runner(torch) -> bytes) for every workload."""
    small = lambda fmt, M, seed: gen.gen_dense_case(fmt, 1024, 2048, M, seed=seed)  # noqa: E731
    moe_case = gen.gen_moe_case(gen.seed_for(4, 0))
    return [
        ("nvfp4_decode_m1", lambda t: _dense(t, gen.workload_case("dense_nvfp4_decode", 0))),
        ("nvfp4_decode_m4", lambda t: _dense(t, gen.workload_case("dense_nvfp4_decode", 1))),
        ("fp8_decode_m1", lambda t: _dense(t, gen.workload_case("dense_fp8_decode", 0))),
        ("fp8_decode_m16", lambda t: _dense(t, gen.workload_case("dense_fp8_decode", 1))),
        ("tiny_m1", lambda t: _dense(t, gen.workload_case("tiny_nvfp4", 0))),
        ("stream_stages_m3", lambda t: _dense(t, small("nvfp4", 3, 501), stages=True)),
        ("gemm_splitk_m64", lambda t: _dense(t, small("nvfp4", 64, 502), path=q.PATH_GEMM)),
        ("gemm_m1024", lambda t: _dense(t, small("nvfp4", 1024, 503), path=q.PATH_GEMM)),
        ("gemm_fp8_m1024", lambda t: _dense(t, small("fp8", 1024, 504), path=q.PATH_GEMM)),
        ("gemm_pair_m1024", lambda t: _dense(t, small("nvfp4", 1024, 505), path=q.PATH_GEMM_PAIR)),
        ("gemm_dq_m1600", lambda t: _dense(t, small("nvfp4", 1600, 507), path=q.PATH_GEMM_DQ)),
        ("gemm_dq_fp8_m100", lambda t: _dense(t, small("fp8", 100, 508), max_M=768, path=q.PATH_GEMM_DQ)),
        ("moe_m1_4b", lambda t: _moe(t, moe_case, 4)),
        ("moe_m1_3b", lambda t: _moe(t, moe_case, 3)),
        ("moe_noalloc", lambda t: _noalloc(t, moe_case)),
        ("moe_tokens_m16", lambda t: _tokens(t, 16)),
        ("tp_shards_4", lambda t: _shards(t, small("fp8", 2, 506), 4)),
    ]


def run(checking: bool):
    """Every case's output bytes, and (checking build) its bounds report."""
    import torch
    outs, reports = {}, {}
    for name, fn in cases():
        outs[name] = fn(torch)
        if checking:
            reports[name] = list(q.qmlp_debug_bounds())
    return outs, reports


def planted(torch):
    """The decode kernel with its gate/up banks' allowed bytes cut to half:
    the report names site 1 and an index past the cut; after the limit is
    lifted the same call is clean again. Returns (report while cut, report
    after, bytes after)."""
    case = gen.workload_case("dense_nvfp4_decode", 0)
    mlp = q.QuantMLP.from_case(case)
    x = _dev(torch, case.x)
    out = torch.empty((case.M, case.K), dtype=torch.int16, device="cuda")
    half = case.I * case.K * 9 // 16 // 2  # half of one projection's bank: codes (K/2 B) + scales (K/16 B) a row
    mlp.bounds_limit(half)
    mlp.forward(x, out)
    cut = list(q.qmlp_debug_bounds())
    mlp.check()
    mlp.bounds_limit(0)
    mlp.forward(x, out)
    after = list(q.qmlp_debug_bounds())
    mlp.check()
    mlp.close()
    return cut, after, half, _bytes(out)


if __name__ == "__main__":
    import torch
    assert q.qmlp_debug_bounds_enabled() == 1, "QMLP_LIB does not name a checking build"
    outs, reports = run(True)
    cut, after, half, planted_out = planted(torch)
    np.savez(sys.argv[1], **outs, planted_out=planted_out)
    with open(sys.argv[1] + ".json", "w") as f:
        json.dump({"reports": reports, "cut": cut, "after": after, "half": half}, f)
    print("checking build: %d cases" % len(outs))
