"""GPU parity of the dense decode path (GEMV family, M <= 16) against the CPU
oracle, through the C ABI: decode bit-exactness, the tiny/27B-class NVFP4 and
FP8 workloads at their decode token counts, ragged tails, determinism, host
buffers, CUDA-graph replay and argument rejection."""
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


_CASES = {}


def case_of(name, variant):
    key = (name, variant)
    if key not in _CASES:
        _CASES[key] = gen.workload_case(name, variant)
    return _CASES[key]


def run_forward(torch, mlp, x_bits, path=q.PATH_AUTO):
    M = x_bits.shape[0]
    x = to_dev(x_bits)
    out = torch.empty((M, mlp.K), dtype=torch.int16, device="cuda")
    act = torch.empty((M, mlp.I), dtype=torch.int16, device="cuda")
    mlp.forward_debug(x, act, out, path=path)
    torch.cuda.synchronize()
    mlp.check()
    return bits_from_dev(out), bits_from_dev(act)


def one_hot_rows(K, ks):
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for r, k in enumerate(ks):
        x[r, k] = 0x3F80  # 1.0
    return x


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("M", [7, 12])
def test_decode_bit_exact_one_hot(torch_cuda, fmt, M):
    """One-hot x at k boundaries returns single dequantized weights exactly
    (E2M1*E4M3 for NVFP4, e4m3fn for FP8), for every projection."""
    torch = torch_cuda
    K, I = 336, 144  # K = 5 chunks of 64 + a ragged 16; I = 2 chunks + 16
    case = gen.gen_dense_case(fmt, K, I, 1, seed=101)
    mlp = q.QuantMLP.from_case(case, max_M=16)
    for which, proj in ((0, case.gate), (1, case.up), (2, case.down)):
        Kp = proj.K
        base = [0, 15, 16, 31, 63, 64, Kp - 1, Kp - 16, 17, 200 % Kp, 100 % Kp, 47]
        ks = base[:M]
        x = to_dev(one_hot_rows(Kp, ks))
        y = torch.empty((M, proj.N), dtype=torch.float32, device="cuda")
        mlp.debug_project(which, x, y, path=q.PATH_GEMV)
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        ref = oracle.decode_proj(proj)
        for r, k in enumerate(ks):
            assert np.array_equal(got[r], ref[:, k]), (fmt, which, k)
    mlp.close()


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_debug_project_matches_oracle_dot(torch_cuda, fmt):
    torch = torch_cuda
    case = gen.gen_dense_case(fmt, 512, 256, 5, seed=102)
    mlp = q.QuantMLP.from_case(case)
    for which, proj in ((0, case.gate), (2, case.down)):
        xb = gen.gen_x_only(103 + which, 5, proj.K)
        y = torch.empty((5, proj.N), dtype=torch.float32, device="cuda")
        mlp.debug_project(which, to_dev(xb), y)
        torch.cuda.synchronize()
        ref = oracle.project(proj, xb)
        got = y.cpu().numpy().astype(np.float64)
        err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert err < 1e-5, err
    mlp.close()


@pytest.mark.parametrize("variant", [0, 1])
def test_parity_tiny_nvfp4(torch_cuda, variant):
    case = case_of("tiny_nvfp4", variant)
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    mlp.close()


@pytest.mark.parametrize("variant", [0, 1])
def test_parity_dense_nvfp4_decode(torch_cuda, variant):
    case = case_of("dense_nvfp4_decode", variant)
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    # the same bytes through a second run: bit-identical (no atomics)
    out2, _ = run_forward(torch_cuda, mlp, case.x)
    assert np.array_equal(out, out2)
    mlp.close()


@pytest.mark.parametrize("path", [q.PATH_AUTO, q.PATH_GEMV, q.PATH_GEMM])
@pytest.mark.parametrize("variant", [0, 1])
def test_parity_dense_fp8_decode(torch_cuda, variant, path):
    """M = 1 and 16; at 16 tokens the automatic path is one launch of the
    I-partitioned decode kernel (two 8-token column tiles, x in two halves);
    the tensor-core GEMM at the same token counts is run explicitly (a handle
    with room for 17 tokens, so that it has GEMM tiles)."""
    case = case_of("dense_fp8_decode", variant)
    mlp = q.QuantMLP.from_case(case, max_M=17 if path == q.PATH_GEMM else None)
    out, act = run_forward(torch_cuda, mlp, case.x, path=path)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    mlp.close()


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("M", [1, 3, 9, 16, 20])
def test_ragged_tails(torch_cuda, fmt, M):
    """K and I that are multiples of 16 but not of the 64-k chunk; M that does
    not fill an 8-token MMA tile; M > 16 runs 16-token blocks."""
    case = gen.gen_dense_case(fmt, 336, 144, M, seed=110 + M)
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x, path=q.PATH_GEMV)
    ref = oracle.dense_forward(case)
    # a zero result must not pass: the reference is non-degenerate
    assert np.count_nonzero(oracle.bf16_bits_to_f64(ref["out"])) > 0.9 * ref["out"].size
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    mlp.close()


def test_tiny_x_magnitudes_keep_precision(torch_cuda):
    """Activations far below 1 (and a row of zeros) go through the per-token
    power-of-two staging without loss."""
    case = gen.gen_dense_case("nvfp4", 256, 512, 3, seed=120)
    x = case.x.copy()
    xf = oracle.bf16_bits_to_f64(x)
    xf[0] *= 2.0 ** -40
    xf[1] *= 2.0 ** 30
    xf[2] = 0.0
    case.x = oracle.bf16_rne_array(xf)
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x)
    ref = oracle.dense_forward(case)
    for r in range(2):
        compare(act[r:r + 1], ref["act"][r:r + 1], what=f"act row {r}")
    assert np.array_equal(oracle.bf16_bits_to_f64(act[2]), oracle.bf16_bits_to_f64(ref["act"][2]))
    mlp.close()


def test_forward_host_matches_device(torch_cuda):
    torch = torch_cuda
    case = case_of("tiny_nvfp4", 1)
    mlp = q.QuantMLP.from_case(case)
    out_dev, _ = run_forward(torch, mlp, case.x)
    xh = torch.from_numpy(case.x.view(np.int16)).pin_memory()
    oh = torch.empty((case.M, case.K), dtype=torch.int16).pin_memory()
    mlp.forward_host(xh, oh)
    assert np.array_equal(oh.numpy().view(np.uint16), out_dev)
    mlp.close()


def test_cuda_graph_replay_with_changing_inputs(torch_cuda):
    torch = torch_cuda
    case = case_of("tiny_nvfp4", 1)
    mlp = q.QuantMLP.from_case(case)
    x = to_dev(case.x)
    out = torch.empty((case.M, case.K), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mlp.forward(x, out, stream=s)  # warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mlp.forward(x, out, stream=s)
    for seed in (130, 131):
        xb = gen.gen_x_only(seed, case.M, case.K)
        x.copy_(to_dev(xb))
        g.replay()
        torch.cuda.synchronize()
        c2 = gen.DenseCase(**{**case.__dict__, "x": xb})
        compare(bits_from_dev(out), oracle.dense_forward(c2)["out"], what=f"graph seed {seed}")
    mlp.close()


def test_argument_rejection_launches_nothing(torch_cuda):
    torch = torch_cuda
    case = case_of("tiny_nvfp4", 1)
    mlp = q.QuantMLP.from_case(case)
    K, M = case.K, case.M
    x = to_dev(case.x)
    out = torch.full((M, K), 0x1234, dtype=torch.int16, device="cuda")
    raw = torch.zeros(M * K + 8, dtype=torch.int16, device="cuda")
    L = q.lib()
    cs = torch.cuda.current_stream().cuda_stream
    assert L.qmlp_forward(mlp.h, raw.data_ptr() + 2, M, out.data_ptr(), cs) == 2   # misaligned x
    assert L.qmlp_forward(mlp.h, x.data_ptr(), M, out.data_ptr() + 2, cs) == 2     # misaligned out
    assert L.qmlp_forward(mlp.h, x.data_ptr(), M, x.data_ptr(), cs) == 3           # out aliases x
    assert L.qmlp_forward(mlp.h, x.data_ptr(), 0, out.data_ptr(), cs) == 4         # M = 0
    assert L.qmlp_forward(mlp.h, x.data_ptr(), M + 1, out.data_ptr(), cs) == 4     # M > max_M
    assert L.qmlp_forward(mlp.h, None, M, out.data_ptr(), cs) == 1                 # null
    assert L.qmlp_forward_path(mlp.h, q.PATH_GEMM, x.data_ptr(), M, out.data_ptr(), cs) == 4
    assert L.qmlp_debug_project(mlp.h, 3, 0, x.data_ptr(), M, out.data_ptr(), cs) == 1
    torch.cuda.synchronize()
    assert bool((out == 0x1234).all())
    mlp.close()


def test_create_rejects_global_scale_zero_and_bad_fmt(torch_cuda):
    case = gen.gen_dense_case("nvfp4", 64, 32, 1, seed=140)
    case.gate.global_scale = np.float32(0.0)
    with pytest.raises(q.QmlpError) as e:
        q.QuantMLP.from_case(case)
    assert e.value.status == 1
