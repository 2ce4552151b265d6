"""The seeded input recipe: every generator draws what its docstring states
(value ranges, the code sets it may use, the route structure) and the same
seed gives the same bytes. CPU only; small shapes."""
import numpy as np
import pytest

from weight_quantized_swiglu_gb300 import inputs as gen


def test_seed_formula_and_determinism():
    assert gen.seed_for(0, 0) == 20261202
    assert gen.seed_for(3, 1) == 20261202 + 301
    a = gen.gen_dense_case("nvfp4", 64, 32, 2, 7)
    b = gen.gen_dense_case("nvfp4", 64, 32, 2, 7)
    for p, q in ((a.gate, b.gate), (a.up, b.up), (a.down, b.down)):
        assert np.array_equal(p.w, q.w) and np.array_equal(p.scale, q.scale)
        assert p.global_scale == q.global_scale
    assert np.array_equal(a.x, b.x)
    c = gen.gen_dense_case("nvfp4", 64, 32, 2, 8)
    assert not np.array_equal(a.gate.w, c.gate.w)


def test_nibble_packing_low_nibble_is_even_k():
    codes = np.array([[1, 2, 3, 4, 15, 0]], dtype=np.uint8)
    assert gen.pack_nibbles(codes).tolist() == [[0x21, 0x43, 0x0F]]


def test_nvfp4_projection_recipe():
    rng = np.random.default_rng(1)
    p = gen.gen_nvfp4_proj(rng, 256, 512)
    assert p.w.shape == (256, 256) and p.w.dtype == np.uint8
    assert p.scale.shape == (256, 32) and p.scale.dtype == np.uint8
    codes = np.concatenate([p.w & 0xF, p.w >> 4]).ravel()
    counts = np.bincount(codes, minlength=16)
    assert counts.min() > 0.8 * codes.size / 16   # every code drawn, roughly uniformly
    e, m = p.scale >> 3, p.scale & 7
    assert e.min() == 1 and e.max() == 9           # biased exponent field 1..9: normal numbers only
    assert m.min() == 0 and m.max() == 7
    assert not np.any(p.scale & 0x80)               # positive scales
    assert 100.0 <= float(p.global_scale) < 1000.0 and p.global_scale.dtype == np.float32


def test_fp8_projection_recipe():
    rng = np.random.default_rng(2)
    p = gen.gen_fp8_proj(rng, 128, 512)
    assert p.w.shape == (128, 512)
    assert not np.any((p.w & 0x7F) == 0x7F)         # never a NaN code
    assert np.unique(p.w).size == 254               # every finite code, both signs, subnormals, +-0
    assert p.scale.dtype == np.float32 and p.scale.shape == (128,)
    assert p.scale.min() >= 1e-3 and p.scale.max() < 1e-2


def test_activation_recipe_is_rounded_standard_normal():
    x = gen.gen_x_only(5, 64, 1024)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(float(xf.mean())) < 0.02 and abs(float(xf.std()) - 1.0) < 0.02
    # the bf16 bits are torch's RNE rounding of the fp32 draw
    rng = np.random.default_rng(5)
    raw = rng.standard_normal((64, 1024), dtype=np.float32)
    assert np.array_equal(x, gen.f32_to_bf16_bits(raw))


@pytest.mark.parametrize("shape", [(4, 8, 3)])
def test_awq_metadata_records(shape):
    rng = np.random.default_rng(3)
    m4, m3 = gen._awq_meta(rng, shape)
    s4 = (m4[..., 0].astype(np.uint16) | (m4[..., 1].astype(np.uint16) << 8)).view(np.float16)
    b4 = (m4[..., 2].astype(np.uint16) | (m4[..., 3].astype(np.uint16) << 8)).view(np.float16)
    s3 = (m3[..., 0].astype(np.uint16) | (m3[..., 1].astype(np.uint16) << 8)).view(np.float16)
    z = m3[..., 2]
    assert np.array_equal(s4.view(np.uint16), s3.view(np.uint16))   # one scale, two layouts
    assert float(s3.min()) >= np.float16(1e-3) and float(s3.max()) <= np.float16(2e-2)
    assert z.max() <= 15
    # the 4-byte bias is the fp16 nearest to the exact -z*s (checked by its two fp16 neighbours)
    exact = -(z.astype(np.float64)) * s3.astype(np.float64)
    err = np.abs(b4.astype(np.float64) - exact)
    up = np.nextafter(b4, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(b4, np.float16(-np.inf)).astype(np.float64)
    assert np.all(err <= np.abs(up - exact)) and np.all(err <= np.abs(dn - exact))


def test_route_recipe():
    rng = np.random.default_rng(4)
    E, topk = 512, 10
    for _ in range(50):
        ids, rw = gen.gen_routes(rng, E, topk)
        assert ids.dtype == np.int32 and rw.dtype == np.float32 and ids.shape == rw.shape == (topk,)
        valid = ids[(ids >= 0) & (ids < E)]
        assert np.count_nonzero(ids == E) == 1                  # one invalid id (E)
        assert valid.size == topk - 1 and np.unique(valid).size == topk - 2   # one duplicate
        assert np.all(rw > 0) and abs(float(rw.astype(np.float64).sum()) - 1.0) < 1e-6


def test_token_routes_are_per_token_recipes():
    tok = gen.gen_moe_tokens(9, 6, E=32, K=64, I=32)
    assert tok.ids.shape == (6, 10) and tok.rw.shape == (6, 10)
    assert tok.x16.shape == (6, 64) and tok.xb.shape == (6, 64)
    for t in range(6):
        ids = tok.ids[t]
        assert np.count_nonzero(ids == 32) == 1 and np.unique(ids[ids < 32]).size == 8
    assert np.array_equal(tok.case.ids, tok.ids[0]) and np.array_equal(tok.case.x_fp16, tok.x16[0])
