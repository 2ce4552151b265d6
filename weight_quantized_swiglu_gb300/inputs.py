"""Seeded synthetic inputs for the weight-quantized SwiGLU MLP.

This module only draws random numbers and packs them into the byte layouts the
library accepts. It holds none of the method's arithmetic (no decoding, no
dot products, no activation): both the CUDA path and the CPU oracle consume the
exact bytes produced here, so any disagreement between them is a disagreement
in the method, never in the inputs.

Value distributions follow the workloads the method is quoted on:

* NVFP4 projections (Qwen3.8-27B-NVFP4, "NVFP4 numerics as implemented"):
  E2M1 codes uniform over 0..15, two per byte with the low nibble holding the
  earlier k; one E4M3 scale per 16 input channels whose biased exponent field
  is uniform in 1..9 (unbiased -6..2) and whose mantissa field is uniform in
  0..7; one fp32 global scale per tensor uniform in [100, 1000).
* FP8 per-channel W8A16 (vllm.cpp issue "tp>1 fp8w tail-MLP shard ...",
  "Logic anchor" / "Correctness" item 1): e4m3fn bytes drawn uniformly over
  the 254 finite codes (both signs, subnormals, +-0), fp32 per-output-channel
  scale uniform in [1e-3, 1e-2].
* AWQ int4 group-32 routed experts (1Cat-vLLM PR "Add native-g32 AWQ QPN M1
  operator", "What it does"): u4 codes uniform 0..15, fp16 scale uniform in
  [1e-3, 2e-2], u8 zero uniform 0..15; the 4-byte record stores the fp16 bias
  half(-z*s) of the same zero, so both record layouts describe one weight set.
* Activations x ~ N(0, 1) drawn in fp32 and cast once (round to nearest even)
  to bf16 or fp16 by torch/numpy.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

BASE_SEED = 20261202

# Workload sizes (hidden K, intermediate I).
TINY_K, TINY_I = 256, 512
DENSE_K, DENSE_I = 5120, 17408
MOE_E, MOE_K, MOE_I, MOE_TOPK = 512, 2560, 160, 10


def seed_for(config: int, variant: int) -> int:
    """Seed of one workload: base + 100*config + variant (variant 0 = first M)."""
    return BASE_SEED + 100 * config + variant


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (torch's RNE cast) and return the raw bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def f32_to_fp16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16).copy()


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes [..., K] into bytes [..., K/2], low nibble = even k."""
    c = codes.astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


# ----------------------------------------------------------------------------
# NVFP4 / FP8 dense projections
# ----------------------------------------------------------------------------
@dataclass
class Proj:
    """One projection of shape [N, K] in the library's input layout.

    NVFP4: w = packed E2M1 bytes [N, K/2], scale = E4M3 bytes [N, K/16],
           global_scale = fp32 (the dequantization factor is 1/global_scale).
    FP8:   w = e4m3fn bytes [N, K], scale = fp32 [N], global_scale unused (1).
    """
    fmt: str
    N: int
    K: int
    w: np.ndarray
    scale: np.ndarray
    global_scale: np.float32 = np.float32(1.0)


def gen_nvfp4_proj(rng: np.random.Generator, N: int, K: int) -> Proj:
    assert K % 16 == 0
    codes = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    e = rng.integers(1, 10, size=(N, K // 16), dtype=np.uint8)
    m = rng.integers(0, 8, size=(N, K // 16), dtype=np.uint8)
    scale = ((e << 3) | m).astype(np.uint8)
    g = np.float32(rng.uniform(100.0, 1000.0))
    return Proj("nvfp4", N, K, pack_nibbles(codes), scale, g)


FP8_FINITE_CODES = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=np.uint8)


def gen_fp8_proj(rng: np.random.Generator, N: int, K: int) -> Proj:
    w = FP8_FINITE_CODES[rng.integers(0, FP8_FINITE_CODES.size, size=(N, K))]
    scale = rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)
    return Proj("fp8", N, K, np.ascontiguousarray(w), scale, np.float32(1.0))


@dataclass
class DenseCase:
    fmt: str
    K: int
    I: int
    M: int
    x: np.ndarray          # bf16 bits, [M, K]
    gate: Proj
    up: Proj
    down: Proj
    seed: int = 0
    name: str = ""


def gen_x_bf16(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def gen_dense_case(fmt: str, K: int, I: int, M: int, seed: int, name: str = "") -> DenseCase:
    """x first, then gate, up, down (codes, scales, global per projection)."""
    rng = np.random.default_rng(seed)
    x = gen_x_bf16(rng, M, K)
    gen = gen_nvfp4_proj if fmt == "nvfp4" else gen_fp8_proj
    gate = gen(rng, I, K)
    up = gen(rng, I, K)
    down = gen(rng, K, I)
    return DenseCase(fmt, K, I, M, x, gate, up, down, seed, name)


def gen_x_only(seed: int, M: int, K: int) -> np.ndarray:
    return gen_x_bf16(np.random.default_rng(seed), M, K)


# ----------------------------------------------------------------------------
# AWQ routed experts
# ----------------------------------------------------------------------------
@dataclass
class MoeCase:
    E: int
    K: int
    I: int
    topk: int
    w13: np.ndarray          # u8 [E, 2I, K/2]
    w13_meta4: np.ndarray    # u8 [E, 2I, K/32, 4]  {fp16 scale, fp16 bias}
    w13_meta3: np.ndarray    # u8 [E, 2I, K/32, 3]  {fp16 scale, u8 zero}
    w2: np.ndarray           # u8 [E, K, I/2]
    w2_meta4: np.ndarray     # u8 [E, K, I/32, 4]
    w2_meta3: np.ndarray     # u8 [E, K, I/32, 3]
    x_fp16: np.ndarray       # u16 bits [K]
    x_bf16: np.ndarray       # u16 bits [K]
    ids: np.ndarray          # int32 [topk]
    router_w: np.ndarray     # fp32 [topk]
    seed: int = 0


def _awq_meta(rng: np.random.Generator, shape) -> tuple[np.ndarray, np.ndarray]:
    s = rng.uniform(1e-3, 2e-2, size=shape).astype(np.float16)
    z = rng.integers(0, 16, size=shape, dtype=np.uint8)
    # bias stored by the 4-byte layout: fp16 of -z*s, rounded once from the
    # exact float64 product (numpy's float64 -> float16 cast is RNE).
    b = (-(z.astype(np.float64)) * s.astype(np.float64)).astype(np.float16)
    s_bytes = s.view(np.uint16)
    b_bytes = b.view(np.uint16)
    meta4 = np.empty(shape + (4,), dtype=np.uint8)
    meta4[..., 0] = s_bytes & 0xFF
    meta4[..., 1] = s_bytes >> 8
    meta4[..., 2] = b_bytes & 0xFF
    meta4[..., 3] = b_bytes >> 8
    meta3 = np.empty(shape + (3,), dtype=np.uint8)
    meta3[..., 0] = s_bytes & 0xFF
    meta3[..., 1] = s_bytes >> 8
    meta3[..., 2] = z
    return meta4, meta3


def gen_awq_weights(rng: np.random.Generator, E: int, K: int, I: int):
    c13 = rng.integers(0, 16, size=(E, 2 * I, K), dtype=np.uint8)
    w13 = pack_nibbles(c13)
    m13_4, m13_3 = _awq_meta(rng, (E, 2 * I, K // 32))
    c2 = rng.integers(0, 16, size=(E, K, I), dtype=np.uint8)
    w2 = pack_nibbles(c2)
    m2_4, m2_3 = _awq_meta(rng, (E, K, I // 32))
    return w13, m13_4, m13_3, w2, m2_4, m2_3


def gen_routes(rng: np.random.Generator, E: int, topk: int, n_invalid: int = 1, n_dup: int = 1):
    """topk route slots: distinct valid ids, plus duplicates and invalid ids at
    seeded positions; router weights are the softmax (fp64, stored fp32) of
    N(0,1) logits over the topk slots."""
    n_distinct = topk - n_invalid - n_dup
    distinct = rng.choice(E, size=n_distinct, replace=False).astype(np.int32)
    dups = distinct[rng.integers(0, n_distinct, size=n_dup)] if n_dup else np.empty(0, np.int32)
    invalid = np.full(n_invalid, E, dtype=np.int32)
    ids = np.concatenate([distinct, dups, invalid]).astype(np.int32)
    ids = ids[rng.permutation(topk)]
    logits = rng.standard_normal(topk)
    p = np.exp(logits - logits.max())
    rw = (p / p.sum()).astype(np.float32)
    return ids, rw


def gen_moe_case(seed: int, E: int = MOE_E, K: int = MOE_K, I: int = MOE_I, topk: int = MOE_TOPK,
                 n_invalid: int = 1, n_dup: int = 1) -> MoeCase:
    rng = np.random.default_rng(seed)
    xf = rng.standard_normal(K, dtype=np.float32)
    x16 = f32_to_fp16_bits(xf)
    xb = f32_to_bf16_bits(xf)
    w13, m13_4, m13_3, w2, m2_4, m2_3 = gen_awq_weights(rng, E, K, I)
    ids, rw = gen_routes(rng, E, topk, n_invalid, n_dup)
    return MoeCase(E, K, I, topk, w13, m13_4, m13_3, w2, m2_4, m2_3, x16, xb, ids, rw, seed)


@dataclass
class MoeTokens:
    """M tokens over one expert bank: `case` holds the weights (its one-token
    fields are token 0's); x16 / xb [M, K] bits, ids [M, topk] int32,
    rw [M, topk] fp32."""
    case: MoeCase
    x16: np.ndarray
    xb: np.ndarray
    ids: np.ndarray
    rw: np.ndarray

    @property
    def M(self) -> int:
        return self.ids.shape[0]


def gen_moe_tokens(seed: int, M: int, E: int = MOE_E, K: int = MOE_K, I: int = MOE_I, topk: int = MOE_TOPK,
                   n_invalid: int = 1, n_dup: int = 1) -> MoeTokens:
    """x [M, K] first, then the weights, then every token's routes in token
    order (each token: the one-token recipe -- distinct ids, duplicates and
    invalid ids at seeded positions, softmax router weights)."""
    rng = np.random.default_rng(seed)
    xf = rng.standard_normal((M, K), dtype=np.float32)
    x16 = f32_to_fp16_bits(xf)
    xb = f32_to_bf16_bits(xf)
    w13, m13_4, m13_3, w2, m2_4, m2_3 = gen_awq_weights(rng, E, K, I)
    ids = np.empty((M, topk), dtype=np.int32)
    rw = np.empty((M, topk), dtype=np.float32)
    for t in range(M):
        ids[t], rw[t] = gen_routes(rng, E, topk, n_invalid, n_dup)
    case = MoeCase(E, K, I, topk, w13, m13_4, m13_3, w2, m2_4, m2_3, x16[0].copy(), xb[0].copy(),
                   ids[0].copy(), rw[0].copy(), seed)
    return MoeTokens(case, x16, xb, ids, rw)


def rotating_ids(call: int, topk: int = MOE_TOPK, n_experts: int = 480) -> np.ndarray:
    """Ids of call `call` when cycling `n_experts` experts, topk distinct per call."""
    base = (call * topk) % n_experts
    return ((base + np.arange(topk)) % n_experts).astype(np.int32)


# ----------------------------------------------------------------------------
# The five workloads
# ----------------------------------------------------------------------------
WORKLOADS = {
    # name: (config index, fmt, K, I, (M values))
    "tiny_nvfp4": (0, "nvfp4", TINY_K, TINY_I, (1, 4)),
    "dense_nvfp4_decode": (1, "nvfp4", DENSE_K, DENSE_I, (1, 4)),
    "dense_fp8_decode": (2, "fp8", DENSE_K, DENSE_I, (1, 16)),
    "nvfp4_prefill": (3, "nvfp4", DENSE_K, DENSE_I, (512, 8192)),
    # config 4 is the routed-expert workload (gen_moe_case)
    "fp8_prefill": (5, "fp8", DENSE_K, DENSE_I, (512, 8192)),
}


def workload_case(name: str, variant: int) -> DenseCase:
    cfg, fmt, K, I, Ms = WORKLOADS[name]
    return gen_dense_case(fmt, K, I, Ms[variant], seed_for(cfg, variant), name)
