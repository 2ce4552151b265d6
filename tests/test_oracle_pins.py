"""Pins for the CPU oracle (CPU only).

Each test checks the oracle against something other than itself: published
format tables (tests/golden), library routines (torch's float8 and bf16 casts,
numpy's float16 cast, numpy float64 matmul), exact rational arithmetic
(fractions) and brute force on tiny inputs, plus invariants of the method.
A plausible slip in the oracle (a dropped term, a swapped nibble order, a
group index of k/32 instead of k/16, a transposed operand, a sign error)
fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from weight_quantized_swiglu_gb300 import inputs as gen


# ----------------------------------------------------------------------------
# independent helpers (not the oracle's code)
# ----------------------------------------------------------------------------
def golden_e2m1():
    return {int(c): float(v) for c, v in read_golden("e2m1_ocp_mx.txt")}


def torch_e4m3_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def nearest_bits(v: float, value_of, candidates):
    """Brute-force round-to-nearest-even over candidate encodings."""
    fv = Fraction(v)
    best = None
    for b in candidates:
        val = value_of(b)
        if not math.isfinite(val):
            continue
        d = abs(Fraction(val) - fv)
        key = (d, b & 1)  # ties -> even encoding
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def bf16_val(b):
    return float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])


def fp16_val(b):
    return float(np.array([b], dtype=np.uint16).view(np.float16)[0])


def np_decode_nvfp4(p):
    """Independent NVFP4 decode: numpy unpack + golden E2M1 + torch E4M3."""
    t2 = golden_e2m1()
    lut2 = np.array([t2[c] for c in range(16)])
    lut4 = torch_e4m3_table()
    codes = np.empty((p.N, p.K), dtype=np.uint8)
    codes[:, 0::2] = p.w & 0x0F
    codes[:, 1::2] = p.w >> 4
    sc = np.repeat(lut4[p.scale], 16, axis=1)
    return lut2[codes] * sc


def np_decode_fp8(p):
    return torch_e4m3_table()[p.w]


# ----------------------------------------------------------------------------
# element tables
# ----------------------------------------------------------------------------
def test_e2m1_all_16_codes_match_ocp_table():
    g = golden_e2m1()
    assert sorted(g) == list(range(16))
    for c in range(16):
        v = oracle.e2m1(c)
        assert v == g[c], (c, v, g[c])
        assert math.copysign(1.0, v) == math.copysign(1.0, g[c]), c  # -0 keeps its sign


def test_e4m3_all_256_codes_match_torch_float8():
    ref = torch_e4m3_table()
    for b in range(256):
        v = oracle.e4m3(b)
        if b in (0x7F, 0xFF):
            assert math.isnan(v) and math.isnan(ref[b])
        else:
            assert v == ref[b], (hex(b), v, ref[b])
            assert math.copysign(1.0, v) == math.copysign(1.0, ref[b])


def test_e4m3_spot_values_match_ofp8_table():
    for hx, val in read_golden("e4m3_spot_values.txt"):
        v = oracle.e4m3(int(hx, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val)), hx


def test_e2m1_times_e4m3_products_fit_bf16_and_fp16_exactly():
    # the decoded NVFP4 weight has at most 6 significant bits: exact in bf16/fp16
    for c in range(16):
        for s in range(256):
            if s in (0x7F, 0xFF):
                continue
            w = oracle.e2m1(c) * oracle.e4m3(s)
            assert oracle.bf16_value(oracle.bf16_rne(w)) == w
            assert oracle.fp16_value(oracle.fp16_rne(w)) == w


# ----------------------------------------------------------------------------
# rounding
# ----------------------------------------------------------------------------
def _special_doubles(rng, n):
    vals = list(rng.standard_normal(n) * 10.0 ** rng.integers(-45, 40, size=n))
    vals += [0.0, -0.0, 1.0, -1.0, 3.4e38, 3.39e38, 1e-40, -1e-40, 9.2e-41, 1e-45, 65504.0, 65520.0,
             65519.99, 6.0e-8, 5.9e-8, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]
    return vals


def test_bf16_rne_matches_torch_for_fp32_representable_values():
    rng = np.random.default_rng(1)
    with np.errstate(over='ignore'):
        f32 = np.array(_special_doubles(rng, 4000), dtype=np.float32)
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_rne_array(f32.astype(np.float64))
    fin = np.isfinite(f32)
    assert np.array_equal(got[fin], ref[fin])


def test_bf16_rne_rounds_once_from_double_brute_force():
    # values a hair off a bf16 midpoint: rounding through fp32 first would land
    # on the midpoint and tie-break, single rounding must go to the near side
    rng = np.random.default_rng(2)
    cases = []
    for _ in range(300):
        b = int(rng.integers(0x0080, 0x7F00))
        lo, hi = bf16_val(b), bf16_val(b + 1)
        mid = (lo + hi) / 2
        cases += [mid, mid + mid * 2.0 ** -40, mid - mid * 2.0 ** -40]
    for v in cases:
        b0 = oracle.bf16_rne(v)
        f32b = int(torch.tensor([v], dtype=torch.float64).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
        want = nearest_bits(v, bf16_val, [f32b - 1, f32b, f32b + 1])
        assert b0 == want, (v, hex(b0), hex(want))


def test_fp16_rne_matches_numpy_and_brute_force():
    rng = np.random.default_rng(3)
    vals = np.array(_special_doubles(rng, 4000) + list(rng.uniform(-1, 1, 2000) * 2.0 ** -20),
                    dtype=np.float64)
    with np.errstate(over='ignore'):
        ref = vals.astype(np.float16).view(np.uint16)
    got = oracle.fp16_rne_array(vals)
    assert np.array_equal(got, ref)
    for v in vals[:400]:
        if abs(v) >= 65520 or not math.isfinite(v):
            continue
        b = int(np.float16(v).view(np.uint16))
        want = nearest_bits(float(v), fp16_val, [(b - 1) & 0xFFFF, b, (b + 1) & 0xFFFF])
        assert oracle.fp16_rne(float(v)) == want


def test_bf16_and_fp16_value_decoders_match_library():
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint16)
    for b in bits[::50]:
        vb = oracle.bf16_value(int(b))
        rb = bf16_val(int(b))
        assert (math.isnan(vb) and math.isnan(rb)) or vb == rb
        vh = oracle.fp16_value(int(b))
        rh = fp16_val(int(b))
        assert (math.isnan(vh) and math.isnan(rh)) or vh == rh


# ----------------------------------------------------------------------------
# dense projections
# ----------------------------------------------------------------------------
def test_nvfp4_decode_matches_independent_decode():
    rng = np.random.default_rng(4)
    p = gen.gen_nvfp4_proj(rng, 24, 96)
    assert np.array_equal(oracle.decode_proj(p), np_decode_nvfp4(p))


def test_fp8_decode_matches_torch_float8():
    rng = np.random.default_rng(5)
    p = gen.gen_fp8_proj(rng, 16, 64)
    assert np.array_equal(oracle.decode_proj(p), np_decode_fp8(p))


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_one_hot_x_recovers_single_weights_at_k_boundaries(fmt):
    rng = np.random.default_rng(6)
    K, N = 96, 32
    p = gen.gen_nvfp4_proj(rng, N, K) if fmt == "nvfp4" else gen.gen_fp8_proj(rng, N, K)
    ref = np_decode_nvfp4(p) if fmt == "nvfp4" else np_decode_fp8(p)
    ks = [0, 15, 16, 31, K - 1]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for r, k in enumerate(ks):
        x[r, k] = 0x3F80  # bf16 1.0
    y = oracle.project(p, x)
    for r, k in enumerate(ks):
        assert np.array_equal(y[r], ref[:, k]), k


def test_project_matches_numpy_matmul():
    rng = np.random.default_rng(7)
    p = gen.gen_nvfp4_proj(rng, 40, 128)
    x = gen.gen_x_bf16(rng, 3, 128)
    xd = oracle.bf16_bits_to_f64(x)
    ref = xd @ np_decode_nvfp4(p).T
    y = oracle.project(p, x)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def _exact_dense_reference(case):
    """Dense SwiGLU by exact rationals for the dot products; SiLU in float64
    (math.exp); bf16 rounding by brute force over neighbours."""
    if case.fmt == "nvfp4":
        wg, wu, wd = (np_decode_nvfp4(p) for p in (case.gate, case.up, case.down))
        sg = [float(np.float32(1.0) / case.gate.global_scale)] * case.I
        su = [float(np.float32(1.0) / case.up.global_scale)] * case.I
        sd = [float(np.float32(1.0) / case.down.global_scale)] * case.K
    else:
        wg, wu, wd = (np_decode_fp8(p) for p in (case.gate, case.up, case.down))
        sg, su, sd = (list(map(float, p.scale)) for p in (case.gate, case.up, case.down))
    xd = oracle.bf16_bits_to_f64(case.x)
    M = xd.shape[0]
    g = np.empty((M, case.I))
    u = np.empty((M, case.I))
    act_bits = np.empty((M, case.I), dtype=np.uint16)
    for m in range(M):
        xf = [Fraction(float(v)) for v in xd[m]]
        for i in range(case.I):
            G = Fraction(sg[i]) * sum(a * Fraction(float(b)) for a, b in zip(xf, wg[i]))
            U = Fraction(su[i]) * sum(a * Fraction(float(b)) for a, b in zip(xf, wu[i]))
            g[m, i], u[m, i] = float(G), float(U)
            gv = float(G)
            a = gv / (1.0 + math.exp(-gv)) * float(U)
            bb = int(torch.tensor([a], dtype=torch.float64).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
            act_bits[m, i] = nearest_bits(a, bf16_val, [(bb + d) & 0xFFFF for d in (-1, 0, 1)])
    actd = oracle.bf16_bits_to_f64(act_bits)
    out_pre = np.empty((M, case.K))
    for m in range(M):
        af = [Fraction(float(v)) for v in actd[m]]
        for o in range(case.K):
            out_pre[m, o] = float(Fraction(sd[o]) * sum(a * Fraction(float(b)) for a, b in zip(af, wd[o])))
    return g, u, act_bits, out_pre


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_dense_forward_brute_force_tiny(fmt):
    case = gen.gen_dense_case(fmt, K=32, I=32, M=3, seed=11)
    g, u, act_bits, out_pre = _exact_dense_reference(case)
    res = oracle.dense_forward(case, want_pre=True)
    np.testing.assert_allclose(res["g"], g, rtol=1e-13, atol=1e-13 * np.abs(g).max())
    np.testing.assert_allclose(res["u"], u, rtol=1e-13, atol=1e-13 * np.abs(u).max())
    # act bits: identical unless the fp64 pre-activation sits on a bf16 midpoint
    assert np.mean(res["act"] == act_bits) > 0.99
    np.testing.assert_allclose(res["out_pre"], out_pre, rtol=1e-11, atol=1e-11 * np.abs(out_pre).max())
    out_ref = oracle.bf16_rne_array(out_pre)
    assert np.mean(res["out"] == out_ref) > 0.99


def test_dense_forward_matches_numpy_pipeline_medium():
    case = gen.gen_dense_case("nvfp4", K=128, I=96, M=4, seed=12)
    wg, wu, wd = (np_decode_nvfp4(p) for p in (case.gate, case.up, case.down))
    inv = lambda p: float(np.float32(1.0) / p.global_scale)
    xd = oracle.bf16_bits_to_f64(case.x)
    G = inv(case.gate) * (xd @ wg.T)
    U = inv(case.up) * (xd @ wu.T)
    A = G / (1.0 + np.exp(-G)) * U
    act = torch.from_numpy(A).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    O = inv(case.down) * (act @ wd.T)
    res = oracle.dense_forward(case, want_pre=True)
    np.testing.assert_allclose(res["g"], G, rtol=1e-12, atol=1e-12 * np.abs(G).max())
    assert np.mean(oracle.bf16_bits_to_f64(res["act"]) == act) > 0.98
    np.testing.assert_allclose(res["out_pre"], O, rtol=2e-2, atol=1e-2 * np.abs(O).max())


def test_dense_invariants_sign_of_x_and_codes():
    case = gen.gen_dense_case("nvfp4", K=64, I=32, M=2, seed=13)
    base = oracle.dense_forward(case, want_pre=True)
    # x -> -x negates both pre-activations
    neg = gen.DenseCase(**{**case.__dict__, "x": case.x ^ np.uint16(0x8000)})
    r = oracle.dense_forward(neg, want_pre=True)
    assert np.array_equal(r["g"], -base["g"]) and np.array_equal(r["u"], -base["u"])
    # flipping every gate code's sign bit (c ^ 8) negates the gate pre-activation only
    g2 = gen.Proj(**{**case.gate.__dict__, "w": case.gate.w ^ np.uint8(0x88)})
    r = oracle.dense_forward(gen.DenseCase(**{**case.__dict__, "gate": g2}), want_pre=True)
    assert np.array_equal(r["g"], -base["g"]) and np.array_equal(r["u"], base["u"])


def test_fp8_output_linear_in_channel_scale():
    case = gen.gen_dense_case("fp8", K=64, I=32, M=2, seed=14)
    base = oracle.dense_forward(case, want_pre=True)
    d2 = gen.Proj(**{**case.down.__dict__, "scale": (case.down.scale * np.float32(2.0)).astype(np.float32)})
    r = oracle.dense_forward(gen.DenseCase(**{**case.__dict__, "down": d2}), want_pre=True)
    assert np.array_equal(r["out_pre"], 2.0 * base["out_pre"])
    assert np.array_equal(r["act"], base["act"])


def test_nvfp4_global_scale_is_fp32_reciprocal():
    case = gen.gen_dense_case("nvfp4", K=32, I=16, M=1, seed=15)
    res = oracle.dense_forward(case, want_pre=True)
    dots = oracle.project(case.gate, case.x)
    inv = float(np.float32(1.0) / case.gate.global_scale)
    assert np.array_equal(res["g"], inv * dots)


# ----------------------------------------------------------------------------
# AWQ routed experts
# ----------------------------------------------------------------------------
def np_awq_decode(w, meta, meta_bytes, e):
    """Independent AWQ decode: numpy nibble unpack, records read as
    little-endian fp16, half_fma emulated by one float64 -> float16 cast."""
    _, N, half = w.shape
    Kr = half * 2
    codes = np.empty((N, Kr), dtype=np.uint8)
    codes[:, 0::2] = w[e] & 0x0F
    codes[:, 1::2] = w[e] >> 4
    rec = meta[e]
    s = (rec[..., 0].astype(np.uint16) | (rec[..., 1].astype(np.uint16) << 8)).view(np.float16).astype(np.float64)
    if meta_bytes == 4:
        b = (rec[..., 2].astype(np.uint16) | (rec[..., 3].astype(np.uint16) << 8)).view(np.float16).astype(np.float64)
    else:
        b = (-(rec[..., 2].astype(np.float64)) * s).astype(np.float16).astype(np.float64)
    s = np.repeat(s, 32, axis=1)
    b = np.repeat(b, 32, axis=1)
    return (codes.astype(np.float64) * s + b).astype(np.float16).astype(np.float64)


def test_awq_half_fma_exhaustive_codes_and_zeros():
    # every q in 0..15 and zero in 0..15 with 600 seeded scales, against
    # exact rationals rounded by brute force
    rng = np.random.default_rng(16)
    scales = rng.uniform(1e-3, 2e-2, 600).astype(np.float16)
    E, N, Kr = 1, 16 * 16, 32
    for sc in scales:
        q = np.repeat(np.arange(16, dtype=np.uint8), 16)  # row n = 16*q + z
        z = np.tile(np.arange(16, dtype=np.uint8), 16)
        codes = np.repeat(q[:, None], Kr, axis=1)
        w = gen.pack_nibbles(codes)[None]
        meta3 = np.empty((E, N, 1, 3), dtype=np.uint8)
        sb = np.array([sc], dtype=np.float16).view(np.uint16)[0]
        meta3[..., 0] = sb & 0xFF
        meta3[..., 1] = sb >> 8
        meta3[..., 2] = z[None, :, None]
        got = oracle.awq_decode(w, meta3, 3, 0)[:, 0]
        for n in range(N):
            s = Fraction(float(sc))
            b = float(np.float16(float(-int(z[n]) * s)))
            exact = int(q[n]) * s + Fraction(b)
            want = nearest_bits(float(exact), fp16_val,
                                [(int(np.float16(float(exact)).view(np.uint16)) + d) & 0xFFFF for d in (-1, 0, 1)])
            assert got[n] == fp16_val(want), (n, got[n], fp16_val(want))


@pytest.mark.parametrize("meta_bytes", [4, 3])
def test_awq_decode_matches_independent_decode(meta_bytes):
    c = gen.gen_moe_case(seed=17, E=3, K=64, I=32, topk=3, n_invalid=0, n_dup=0)
    m13 = c.w13_meta4 if meta_bytes == 4 else c.w13_meta3
    m2 = c.w2_meta4 if meta_bytes == 4 else c.w2_meta3
    for e in range(3):
        assert np.array_equal(oracle.awq_decode(c.w13, m13, meta_bytes, e), np_awq_decode(c.w13, m13, meta_bytes, e))
        assert np.array_equal(oracle.awq_decode(c.w2, m2, meta_bytes, e), np_awq_decode(c.w2, m2, meta_bytes, e))


def test_awq_one_hot_boundaries():
    c = gen.gen_moe_case(seed=18, E=2, K=128, I=32, topk=1, n_invalid=0, n_dup=0)
    ref = np_awq_decode(c.w13, c.w13_meta4, 4, 1)
    for k in (0, 31, 32, 127):
        x = np.zeros(128, dtype=np.float16)
        x[k] = 1.0
        c1 = gen.MoeCase(**{**c.__dict__, "x_fp16": x.view(np.uint16), "ids": np.array([1], np.int32),
                            "router_w": np.array([1.0], np.float32)})
        r = oracle.moe_m1_forward(c1, 4, "fp16", want_stages=True)
        assert np.array_equal(oracle.fp16_bits_to_f64(r["gu"][0]), ref[:, k].astype(np.float16).astype(np.float64))


def _np_moe(c, meta_bytes, x_dtype, ids, rw):
    x = oracle.fp16_bits_to_f64(c.x_fp16) if x_dtype == "fp16" else oracle.bf16_bits_to_f64(c.x_bf16)
    m13 = c.w13_meta4 if meta_bytes == 4 else c.w13_meta3
    m2 = c.w2_meta4 if meta_bytes == 4 else c.w2_meta3
    acc = np.zeros(c.K)
    for r, e in enumerate(ids):
        if not (0 <= e < c.E):
            continue
        h = (np_awq_decode(c.w13, m13, meta_bytes, e) @ x).astype(np.float16).astype(np.float64)
        g, u = h[:c.I], h[c.I:]
        a = (g / (1.0 + np.exp(-g)) * u).astype(np.float16).astype(np.float64)
        y = (np_awq_decode(c.w2, m2, meta_bytes, e) @ a).astype(np.float16).astype(np.float64)
        acc += float(rw[r]) * y
    return acc.astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("meta_bytes,x_dtype", [(4, "fp16"), (3, "bf16")])
def test_moe_forward_matches_numpy_pipeline(meta_bytes, x_dtype):
    c = gen.gen_moe_case(seed=19, E=6, K=64, I=32, topk=5, n_invalid=1, n_dup=1)
    got = oracle.moe_m1_forward(c, meta_bytes, x_dtype)["out"]
    ref = _np_moe(c, meta_bytes, x_dtype, c.ids, c.router_w)
    # matmul summation order differs from the oracle's sequential sum: allow a
    # 1-ulp flip on a few fp16 roundings
    d = np.abs(oracle.fp16_bits_to_f64(got) - oracle.fp16_bits_to_f64(ref))
    assert d.max() <= 2 * 2.0 ** -10 * np.abs(oracle.fp16_bits_to_f64(ref)).max()
    assert np.mean(got == ref) > 0.95


def test_moe_invalid_ids_contribute_zero_and_duplicates_keep_weights():
    c = gen.gen_moe_case(seed=20, E=8, K=64, I=32, topk=4, n_invalid=0, n_dup=0)
    ids = np.array([3, 5, 8, -1], np.int32)
    rw = np.array([0.25, 0.5, 0.125, 0.125], np.float32)
    full = oracle.moe_m1_forward(c, 4, "fp16", ids=ids, rw=rw, want_stages=True)
    only_valid = oracle.moe_m1_forward(c, 4, "fp16", ids=ids[:2], rw=rw[:2])
    assert np.array_equal(full["out"], only_valid["out"])
    assert list(full["valid"]) == [True, True, False, False]
    # duplicate id: both routes carry identical stage outputs and their own weights
    ids_d = np.array([3, 3], np.int32)
    rw_d = np.array([0.75, 0.25], np.float32)
    d = oracle.moe_m1_forward(c, 4, "fp16", ids=ids_d, rw=rw_d, want_stages=True)
    assert np.array_equal(d["y"][0], d["y"][1])
    y = oracle.fp16_bits_to_f64(d["y"][0])
    assert np.array_equal(d["out"], (0.75 * y + 0.25 * y).astype(np.float16).view(np.uint16))


def test_moe_4b_and_3b_metadata_identical():
    c = gen.gen_moe_case(seed=21, E=6, K=64, I=32, topk=4)
    a = oracle.moe_m1_forward(c, 4, "fp16", want_stages=True)
    b = oracle.moe_m1_forward(c, 3, "fp16", want_stages=True)
    for key in ("out", "gu", "act", "y"):
        assert np.array_equal(a[key], b[key]), key
