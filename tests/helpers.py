"""Shared helpers for the GPU parity tests (conversion and tolerance checks)."""
import numpy as np

import oracle

# Output tolerance (both must hold, against the oracle rounded to the same
# output dtype): relative L2 <= 1e-3 and max|delta| <= 2e-2 * max|ref|.
REL_L2 = 1e-3
MAX_ABS_FRAC = 2e-2


def to_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.cuda()


def bits_from_dev(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def compare(got_bits: np.ndarray, ref_bits: np.ndarray, dtype: str = "bf16", what: str = ""):
    conv = oracle.bf16_bits_to_f64 if dtype == "bf16" else oracle.fp16_bits_to_f64
    g = conv(got_bits)
    r = conv(ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / max(nr, 1e-300)
    mx = np.abs(g - r).max() / max(np.abs(r).max(), 1e-300)
    assert np.abs(r).max() > 0, f"{what}: degenerate all-zero reference"
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_FRAC, f"{what}: max|d|/max|ref| {mx:.3e} > {MAX_ABS_FRAC}"
    return rel, mx
