"""The bench's multi-process host logic on CPU (gloo, world size 2): the
replicas-only launch (barrier, max over ranks) and the reference arm under
torchrun, where rank 0 alone works and prints. No GPU is involved."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    v = bench.max_over_ranks(w, 1.5 + r)  # each replica's own time
    bench.barrier(w)
    q.put((r, w, v, dist.get_backend()))
    dist.destroy_process_group()


def test_replicas_barrier_and_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 and o[3] == "gloo" for o in out)
    assert all(o[2] == 2.5 for o in out)  # the slowest replica's time, on every rank


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks: rank 0 times the oracle and prints one JSON line, rank 1
    exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0


def _tp_rank_main(rank, world, port, q):
    """One rank of the tensor-parallel exchange on CPU: its shard's partial
    output from the oracle (gate/up rows and down columns of its slice, fp64,
    down factor included -- linear, so the rank sum is the layer's), the
    all-gather, and the rank-ordered sum."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    from weight_quantized_swiglu_gb300 import inputs as gen
    from weight_quantized_swiglu_gb300 import tp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = gen.gen_dense_case("nvfp4", 128, 256, 3, seed=4242)
    i0, i1 = tp.shard_range(case.I, rank, world)
    P = gen.Proj
    sub = gen.DenseCase(case.fmt, case.K, i1 - i0, case.M, case.x,
                        P("nvfp4", i1 - i0, case.K, case.gate.w[i0:i1], case.gate.scale[i0:i1], case.gate.global_scale),
                        P("nvfp4", i1 - i0, case.K, case.up.w[i0:i1], case.up.scale[i0:i1], case.up.global_scale),
                        P("nvfp4", case.K, i1 - i0, np.ascontiguousarray(case.down.w[:, i0 // 2:i1 // 2]),
                          np.ascontiguousarray(case.down.scale[:, i0 // 16:i1 // 16]), case.down.global_scale))
    part = torch.from_numpy(oracle.dense_forward(sub, want_pre=True)["out_pre"])
    gathered = tp.gather_partials(part)
    total = gathered[0].clone()
    for r in range(1, world):
        total += gathered[r]
    q.put((rank, gathered.numpy().copy(), part.numpy().copy(), oracle.bf16_rne_array(total.numpy())))
    dist.destroy_process_group()


def test_tensor_parallel_gather_and_rank_ordered_sum_gloo():
    """World size 2 over gloo: every rank receives both partials in rank
    order, and their rank-ordered sum, rounded to bf16, is the whole layer's
    oracle output (the shard slicing covers I exactly once)."""
    import numpy as np
    import torch.multiprocessing as mp
    sys.path.insert(0, ROOT)
    import oracle
    from weight_quantized_swiglu_gb300 import inputs as gen
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    parts = [o[2] for o in out]
    for rank, gathered, _, _ in out:
        assert np.array_equal(gathered[0], parts[0]) and np.array_equal(gathered[1], parts[1]), rank
    assert np.array_equal(out[0][3], out[1][3])  # the same bytes on every rank
    full = oracle.dense_forward(gen.gen_dense_case("nvfp4", 128, 256, 3, seed=4242))["out"]
    assert np.array_equal(out[0][3], full)


def test_shard_range_tiles_the_intermediate_dimension():
    sys.path.insert(0, ROOT)
    from weight_quantized_swiglu_gb300 import tp
    for n in (1, 2, 4, 8):
        rs = [tp.shard_range(17408, r, n) for r in range(n)]
        assert rs[0][0] == 0 and rs[-1][1] == 17408
        assert all(rs[i][1] == rs[i + 1][0] for i in range(n - 1))
    with pytest.raises(ValueError):
        tp.shard_range(17408, 0, 3)
    with pytest.raises(ValueError):
        tp.shard_range(17408, 2, 2)
