"""Pins for the oracle's bfloat16 rounding (definition of the format, RNE)."""

import numpy as np
import torch

from oracle.bf16 import bits_to_f64, f64_to_bits, round_bf16


def test_hand_worked_ties_and_overflow():
    cases = [
        (1.0, 1.0),
        (1 + 2.0 ** -8, 1.0),                      # tie, even neighbour 1.0
        (1 + 3 * 2.0 ** -8, 1 + 2.0 ** -6),        # tie, even neighbour 1+2^-6
        (1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -7),  # just above the tie
        (-(1 + 2.0 ** -8), -1.0),
        (2.0 ** -134, 0.0),                        # half a subnormal quantum -> 0
        (3 * 2.0 ** -134, 2.0 ** -132),            # 1.5 quanta -> 2 (even)
        (2.0 ** -133, 2.0 ** -133),                # smallest subnormal kept
        (2.0 ** 128 - 2.0 ** 120, 2.0 ** 128 - 2.0 ** 120),  # largest finite
        (2.0 ** 128 - 2.0 ** 119, np.inf),         # tie above max -> overflow
        (-(2.0 ** 130), -np.inf),
        (0.1, 0.10009765625),                      # 0x3DCD
    ]
    for x, want in cases:
        got = round_bf16(np.array([x]))[0]
        assert got == want, (x, got, want)
    z = round_bf16(np.array([-0.0]))[0]
    assert z == 0 and np.signbit(z)
    assert np.isnan(round_bf16(np.array([np.nan]))[0])


def test_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    parts = [
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(50000) * 1e30).astype(np.float32),
        (rng.standard_normal(50000) * 1e-39).astype(np.float32),  # subnormals
        rng.integers(0, 2 ** 32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]
    # exact ties: low 16 bits == 0x8000 with random upper bits
    up = rng.integers(0, 2 ** 16, 20000, dtype=np.uint32)
    parts.append(((up << 16) | 0x8000).astype(np.uint32).view(np.float32))
    x = np.concatenate(parts)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy().astype(np.float64)
    got = round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bits_roundtrip():
    u = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    f = bits_to_f64(u)
    fin = np.isfinite(f)
    back = f64_to_bits(f[fin])
    np.testing.assert_array_equal(back, u[fin])
    t = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(f[fin], t[fin])
