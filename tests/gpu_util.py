"""Helpers shared by the GPU parity tests (no test functions here)."""

import numpy as np
import pytest
import torch

from invariant_vd_step_gb300 import build, synth, vd
from oracle.bf16 import bits_to_f64

# Logit tolerance of the step against the oracle: |gpu - ref| <= ATOL + RTOL*|ref|.
ATOL, RTOL = 2e-2, 1e-2


def ready():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    vd.lib()


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16 / fp32 CUDA tensor -> float64 numpy (exact)."""
    if t.dtype == torch.bfloat16:
        return bits_to_f64(synth.bf16_to_u16(t))
    return t.detach().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


def bf16_ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 units-in-the-last-place between bf16-valued arrays."""
    def ordered(x):
        u = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.int64)
        return np.where(u & 0x8000, 0x8000 - u, u)  # monotone integer image
    return np.abs(ordered(a) - ordered(b))


def parity_stats(got: np.ndarray, ref: np.ndarray) -> dict:
    """The stated tolerance read literally (max-abs 2e-2 and max-rel 1e-2,
    each on its own) and combined the way allclose combines them."""
    d = np.abs(got - ref)
    a = np.abs(ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(a > 0, d / a, np.where(d > 0, np.inf, 0.0))
    return {"logits": int(d.size), "max_abs": float(d.max()), "max_rel": float(rel.max()),
            "beyond_abs": int((d > ATOL).sum()), "beyond_rel": int((d > RTOL * a).sum()),
            "beyond_literal": int(((d > ATOL) | (d > RTOL * a)).sum()),
            "beyond_combined": int((d > ATOL + RTOL * a).sum()),
            "beyond_twice_combined": int((d > 2 * (ATOL + RTOL * a)).sum())}


def report(name: str, stats: dict):
    """One machine-readable line per parity measurement (shown with pytest -s)."""
    import json
    print(f"PARITY {name} {json.dumps(stats, sort_keys=True)}", flush=True)


def assert_logits_close(got: np.ndarray, ref: np.ndarray):
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    assert np.all(excess <= 0), f"max excess over tolerance {excess.max():.3g} (max |d| {np.abs(got - ref).max():.3g})"


def cuda_bf16(t):
    return t.to("cuda")
