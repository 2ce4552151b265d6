"""GPU parity of the tensor-core prefill path (GEMM family: NVFP4 and FP8
per-channel, M >= 17) against the CPU oracle, through the C ABI: exact
single-weight decode, raw projections, the tiny shape at ragged token
counts, the 27B-class prefill shape at its token counts (sampled rows),
the dequantise-once GEMM (decoded fp16 weights staged before the GEMM),
determinism and the automatic path choice."""
import numpy as np
import pytest

import oracle
import weight_quantized_swiglu_gb300 as q
from weight_quantized_swiglu_gb300 import inputs as gen
from helpers import bits_from_dev, compare, to_dev

pytestmark = pytest.mark.gpu

# GEMM tiles need K % 64 == 0, I % 128 == 0 (gate/up rows in 128-row halves)
# and hidden K % 256 == 0 (down rows): the tiny shape qualifies.
TK, TI = gen.TINY_K, gen.TINY_I


@pytest.fixture(scope="module")
def torch_cuda(cuda_available):
    import torch
    from weight_quantized_swiglu_gb300 import build
    build.build()
    q.lib()
    return torch


def run_forward(torch, mlp, x_bits, path):
    M = x_bits.shape[0]
    out = torch.empty((M, mlp.K), dtype=torch.int16, device="cuda")
    act = torch.empty((M, mlp.I), dtype=torch.int16, device="cuda")
    mlp.forward_debug(to_dev(x_bits), act, out, path=path)
    torch.cuda.synchronize()
    mlp.check()
    return bits_from_dev(out), bits_from_dev(act)


FMTS = ["nvfp4", "fp8"]


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_one_hot_returns_decoded_weights_exactly(torch_cuda, fmt):
    """x = e_k rows: y[r, n] = the decoded W[n, k] exactly (E2M1 * E4M3, or
    e4m3fn), for gate, up and down, at k positions on scale-group, k-step
    and tile boundaries."""
    torch = torch_cuda
    case = gen.gen_dense_case(fmt, TK, TI, 1, seed=201)
    mlp = q.QuantMLP.from_case(case, max_M=64)
    for which, proj in ((0, case.gate), (1, case.up), (2, case.down)):
        Kp = proj.K
        ks = [0, 1, 15, 16, 31, 32, 63, 64, 127, 128, Kp - 64, Kp - 17, Kp - 16, Kp - 1, 100, 200,
              Kp // 2, Kp // 2 + 1, 65, 191]
        x = np.zeros((len(ks), Kp), dtype=np.uint16)
        for r, k in enumerate(ks):
            x[r, k] = 0x3F80  # 1.0
        y = torch.empty((len(ks), proj.N), dtype=torch.float32, device="cuda")
        mlp.debug_project(which, to_dev(x), y, path=q.PATH_GEMM)
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        ref = oracle.decode_proj(proj)
        for r, k in enumerate(ks):
            assert np.array_equal(got[r], ref[:, k]), (which, k)
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_pair_gemm_one_hot_is_bit_exact(torch_cuda, fmt):
    """The CTA-pair GEMM path (each CTA of a cluster holds half of the 256
    tokens of a tile and decodes half of its 256 weight rows): x =
    e_k rows in both halves of the token tile, one per k on scale-group,
    k-step and tile boundaries, return the decoded weights bit for bit, for
    gate (rows decoded by the first CTA of each pair), up (the second) and
    down."""
    torch = torch_cuda
    case = gen.gen_dense_case(fmt, TK, TI, 1, seed=205)
    mlp = q.QuantMLP.from_case(case, max_M=512)
    for which, proj in ((0, case.gate), (1, case.up), (2, case.down)):
        Kp = proj.K
        M = 300  # a full 256-token tile and a ragged second one
        ks = [(r * 37) % Kp for r in range(M)]
        ks[:8] = [0, 15, 16, 31, 63, 64, Kp - 1, Kp - 16]
        ks[128:132] = [1, 17, 65, Kp - 2]  # the second CTA's half of the first tile
        x = np.zeros((M, Kp), dtype=np.uint16)
        for r, k in enumerate(ks):
            x[r, k] = 0x3F80
        y = torch.empty((M, proj.N), dtype=torch.float32, device="cuda")
        mlp.debug_project(which, to_dev(x), y, path=q.PATH_GEMM_PAIR)
        torch.cuda.synchronize()
        mlp.check()
        got = y.cpu().numpy().astype(np.float64)
        ref = oracle.decode_proj(proj)
        for r, k in enumerate(ks):
            assert np.array_equal(got[r], ref[:, k]), (which, r, k)
    # fewer tokens than one pair tile: rejected before any launch
    y = torch.empty((255, case.gate.N), dtype=torch.float32, device="cuda")
    x = torch.zeros((255, case.gate.K), dtype=torch.int16, device="cuda")
    assert q.qmlp_debug_project(mlp.h, 0, q.PATH_GEMM_PAIR, x, 255, y) == 4  # QMLP_ERR_SHAPE
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [200, 300])
def test_dq_gemm_one_hot_is_bit_exact(torch_cuda, fmt, M):
    """The dequantise-once GEMM (each projection decoded into bf16 stage
    images before the GEMM, which then copies them into shared memory as
    they are): x = e_k rows return the decoded weights bit for bit, for gate,
    up and down, at k positions on scale-group, k-step, swizzle-row and tile
    boundaries -- a misplaced 16-byte chunk of an image moves a weight. M =
    200 runs on single CTAs, M = 300 on CTA pairs (a full 256-token tile, each
    CTA holding half of its tokens and half of every image, and a ragged
    one)."""
    torch = torch_cuda
    case = gen.gen_dense_case(fmt, TK, TI, 1, seed=207)
    mlp = q.QuantMLP.from_case(case, max_M=768)  # the decode buffer exists from max_M = 768
    for which, proj in ((0, case.gate), (1, case.up), (2, case.down)):
        Kp = proj.K
        ks = [(r * 29 + 3) % Kp for r in range(M)]
        ks[:12] = [0, 7, 8, 15, 16, 31, 32, 63, 64, Kp - 1, Kp - 16, Kp - 64]
        ks[128:132] = [1, 17, 65, Kp - 2]  # the second CTA's tokens of a pair tile
        x = np.zeros((M, Kp), dtype=np.uint16)
        for r, k in enumerate(ks):
            x[r, k] = 0x3F80
        y = torch.empty((M, proj.N), dtype=torch.float32, device="cuda")
        mlp.debug_project(which, to_dev(x), y, path=q.PATH_GEMM_DQ)
        torch.cuda.synchronize()
        mlp.check()
        got = y.cpu().numpy().astype(np.float64)
        ref = oracle.decode_proj(proj)
        for r, k in enumerate(ks):
            assert np.array_equal(got[r], ref[:, k]), (which, r, k)
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [17, 129, 300])
def test_dq_gemm_parity_and_same_bits_as_decoder_warps(torch_cuda, M, fmt):
    """The dequantise-once GEMM against the oracle, and bit for bit against
    the GEMM whose decoder warps decode in the main loop: both multiply the
    same exact weight values (bf16 images against the bf16 activations there,
    fp16 against the prescaled fp16 activations here) in the same k order
    (M = 17 also runs split-K; M = 300 runs on CTA pairs)."""
    case = gen.gen_dense_case(fmt, TK, TI, M, seed=270 + M)
    mlp = q.QuantMLP.from_case(case, max_M=768)
    out, act = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM_DQ)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    gout, gact = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM)
    assert np.array_equal(act, gact) and np.array_equal(out, gout)
    mlp.close()


def test_dq_forward_in_a_cuda_graph(torch_cuda):
    """The dequantise-once forward decodes the down projection on the
    handle's side stream (forked and joined with events, beside the gate/up
    GEMM); captured in a CUDA graph and replayed with new x it gives the
    bytes of an eager call, and a stage call (no fork) agrees too."""
    torch = torch_cuda
    M = 300
    case = gen.gen_dense_case("nvfp4", TK, TI, M, seed=291)
    mlp = q.QuantMLP.from_case(case, max_M=768)
    x = to_dev(case.x)
    out = torch.empty((M, TK), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mlp.forward(x, out, path=q.PATH_GEMM_DQ, stream=s)  # warm-up (kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mlp.forward(x, out, path=q.PATH_GEMM_DQ, stream=s)
    for seed in (292, 293):
        xb = gen.gen_x_only(seed, M, TK)
        x.copy_(to_dev(xb))
        g.replay()
        torch.cuda.synchronize()
        eager = torch.empty_like(out)
        mlp.forward(to_dev(xb), eager, path=q.PATH_GEMM_DQ)
        torch.cuda.synchronize()
        assert np.array_equal(bits_from_dev(out), bits_from_dev(eager)), seed
    staged = torch.empty_like(out)
    mlp.forward_stage(0, x, None, M, path=q.PATH_GEMM_DQ)
    mlp.forward_stage(1, None, staged, M, path=q.PATH_GEMM_DQ)
    torch.cuda.synchronize()
    mlp.check()
    assert np.array_equal(bits_from_dev(staged), bits_from_dev(out))
    mlp.close()


def test_dq_gemm_needs_the_decode_buffer(torch_cuda):
    """A handle created for fewer than 768 tokens holds no decode buffer:
    the dequantise-once path is refused (SHAPE) before any launch, and the
    automatic path keeps the decoder-warp GEMM."""
    torch = torch_cuda
    case = gen.gen_dense_case("nvfp4", TK, TI, 64, seed=280)
    mlp = q.QuantMLP.from_case(case, max_M=767)
    x = to_dev(case.x)
    out = torch.empty((64, TK), dtype=torch.int16, device="cuda")
    assert q.qmlp_forward_path(mlp.h, q.PATH_GEMM_DQ, x, 64, out, None) == 4  # QMLP_ERR_SHAPE
    auto, _ = run_forward(torch, mlp, case.x, q.PATH_AUTO)
    gemm, _ = run_forward(torch, mlp, case.x, q.PATH_GEMM)
    assert np.array_equal(auto, gemm)
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [17, 200])
def test_gemm_raw_projection_matches_oracle(torch_cuda, M, fmt):
    """Unscaled projections (fp32 out) on random bf16 x, every projection;
    M = 200 leaves a 72-row ragged second token tile."""
    torch = torch_cuda
    case = gen.gen_dense_case(fmt, TK, TI, 1, seed=202)
    mlp = q.QuantMLP.from_case(case, max_M=256)
    for which, proj in ((0, case.gate), (1, case.up), (2, case.down)):
        xb = gen.gen_x_only(210 + which + M, M, proj.K)
        y = torch.empty((M, proj.N), dtype=torch.float32, device="cuda")
        mlp.debug_project(which, to_dev(xb), y, path=q.PATH_GEMM)
        torch.cuda.synchronize()
        ref = oracle.project(proj, xb)
        got = y.cpu().numpy().astype(np.float64)
        err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert err < 1e-5, (which, err)
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [17, 128, 129, 300])
def test_gemm_parity_tiny(torch_cuda, M, fmt):
    case = gen.gen_dense_case(fmt, TK, TI, M, seed=220 + M)
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [9, 40, 128])
def test_gemm_split_k_parity(torch_cuda, M, fmt):
    """K=1024, I=2048: at M <= 128 the gate/up GEMM (16 column tiles) runs 2
    k-splits and the down GEMM (4 column tiles) 4, each writing fp32 partials
    that a reduce kernel adds in split order; same bytes on every call."""
    case = gen.gen_dense_case(fmt, 1024, 2048, M, seed=250 + M)
    mlp = q.QuantMLP.from_case(case, max_M=128)  # GEMM tiles exist when max_M > 16
    out, act = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    out2, _ = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM)
    assert np.array_equal(out, out2)
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_parity_mid_m_27b(torch_cuda, fmt):
    """K=5120, I=17408 at M = 40 (between the decode batch and the prefill
    tile): the automatic path is the GEMM with a 7-way split-K down
    projection; every row against the oracle."""
    case = gen.gen_dense_case(fmt, gen.DENSE_K, gen.DENSE_I, 40, seed=260)
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x, q.PATH_AUTO)
    ref = oracle.dense_forward(case)
    compare(act, ref["act"], what="act")
    compare(out, ref["out"], what="out")
    mlp.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_is_the_automatic_path_above_16_tokens(torch_cuda, fmt):
    """(The tiny shape has no I partition: its decode path takes 16 tokens
    per pass, and the GEMM starts at 17.)"""
    case = gen.gen_dense_case(fmt, TK, TI, 40, seed=230)
    mlp = q.QuantMLP.from_case(case)
    auto, _ = run_forward(torch_cuda, mlp, case.x, q.PATH_AUTO)
    gemm, _ = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM)
    assert np.array_equal(auto, gemm)
    mlp.close()


def test_gemm_activation_magnitudes_keep_precision(torch_cuda):
    """Rows scaled by 2^-40 and 2^30 and a zero row go through the per-token
    fp16 prescale without loss (the same staging as the decode path)."""
    case = gen.gen_dense_case("nvfp4", TK, TI, 48, seed=231)
    xf = oracle.bf16_bits_to_f64(case.x)
    xf[:16] *= 2.0 ** -40
    xf[16:32] *= 2.0 ** 30
    xf[47] = 0.0
    case.x = oracle.bf16_rne_array(xf)
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM)
    ref = oracle.dense_forward(case)
    for r in (0, 15, 16, 31, 40):
        compare(act[r:r + 1], ref["act"][r:r + 1], what=f"act row {r}")
    assert np.array_equal(oracle.bf16_bits_to_f64(act[47]), oracle.bf16_bits_to_f64(ref["act"][47]))
    mlp.close()


def prefill_rows(M, seed):
    """Rows the oracle checks at a prefill size: every row up to 512 tokens;
    above, the first and the last row of every 128-token tile (so every token
    tile of the persistent schedule is hit, at both ends) plus 128 seeded
    random rows from the rest."""
    if M <= 512:
        return np.arange(M, dtype=np.int32)
    ends = np.concatenate([np.arange(0, M, 128), np.minimum(np.arange(127, M + 127, 128), M - 1)])
    rest = np.setdiff1d(np.arange(M), ends)
    rnd = np.random.default_rng(seed).choice(rest, 128, replace=False)
    return np.unique(np.concatenate([ends, rnd])).astype(np.int32)


def test_prefill_rows_cover_every_tile():
    rows = prefill_rows(8192, 1)
    assert rows.size == 64 * 2 + 128
    assert set(range(0, 8192, 128)) <= set(rows.tolist()) and set(range(127, 8192, 128)) <= set(rows.tolist())
    assert np.array_equal(prefill_rows(512, 1), np.arange(512))


@pytest.mark.parametrize("name", ["nvfp4_prefill", "fp8_prefill"])
@pytest.mark.parametrize("variant", [0, 1])
def test_parity_prefill(torch_cuda, variant, name):
    """The 27B-class prefill shape (K=5120, I=17408) at M = 512 and 8192 in
    the launch configuration the bench times, NVFP4 and FP8 per-channel. At
    M = 512 the oracle checks every row; at M = 8192 it checks 256 rows (rows
    are independent, so each is an exact oracle for its row): both ends of
    every 128-token tile and 128 seeded random rows."""
    case = gen.workload_case(name, variant)
    M = case.M
    mlp = q.QuantMLP.from_case(case)
    out, act = run_forward(torch_cuda, mlp, case.x, q.PATH_AUTO)
    rows = prefill_rows(M, 240 + variant)
    ref = oracle.dense_forward(case, rows=rows)
    compare(act[rows], ref["act"], what="act")
    compare(out[rows], ref["out"], what="out")
    # every tile, row by row: one row that went wrong (a mis-assigned or
    # skipped tile) must not hide inside the whole-sample norm. The contract's
    # rel-L2 bound is for whole outputs (a single row of a correct result can
    # sit just above it: act values that round the other way in fp32 and fp64
    # move ~1 % of a row's outputs by one bf16 ulp); per row the check is the
    # contract's max|delta| bound against the row's own max, and rel-L2 within
    # 5e-3 -- a wrong tile is off by ~1.
    g_all, r_all = oracle.bf16_bits_to_f64(out[rows]), oracle.bf16_bits_to_f64(ref["out"])
    for i, r in enumerate(rows):
        if r % 128 in (0, 127) or r == M - 1:
            d = np.abs(g_all[i] - r_all[i])
            assert d.max() <= 2e-2 * np.abs(r_all[i]).max(), f"row {r}"
            assert np.linalg.norm(d) <= 5e-3 * np.linalg.norm(r_all[i]), f"row {r}"
    out2, _ = run_forward(torch_cuda, mlp, case.x, q.PATH_AUTO)
    assert np.array_equal(out, out2)
    if M >= 768:
        # the automatic path is the dequantise-once GEMM here; the GEMM with
        # decoder warps gives the same bits
        gout, gact = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM)
        assert np.array_equal(act, gact) and np.array_equal(out, gout)
    # the CTA-pair GEMM on the same inputs, against the same reference rows
    pout, pact = run_forward(torch_cuda, mlp, case.x, q.PATH_GEMM_PAIR)
    compare(pact[rows], ref["act"], what="pair act")
    compare(pout[rows], ref["out"], what="pair out")
    mlp.close()
