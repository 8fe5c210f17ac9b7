"""How far two exact evaluations of the 8B-shaped layer drift apart when they
disagree by one part in 1e5 at a single point before a bf16 rounding.

Every module output is rounded to bf16, so a tiny disagreement flips a few
roundings; the flips feed the next roundings and the logits of the
Llama-3.1-8B-shaped layer + LM head (random init, 4000 random cached keys)
move by up to ~2e-2.  That is the stated GPU-vs-oracle tolerance itself, so
the full-size GPU check cannot ask more than "within it almost everywhere,
within twice it everywhere".  This test measures the floor on the oracle
alone (no GPU) and pins that it is of that size.
"""

import math

import numpy as np
import pytest

from invariant_vd_step_gb300 import synth
from oracle import decoder as od
from oracle.bf16 import round_bf16


def _weights(spec, **kw):
    """The model's weights, except that the embedding table holds only the
    rows up to the probe token 1234 (its own seeded stream): the floor is a
    property of the layer and LM-head arithmetic, whatever the input row, and
    the full table is the largest tensor to generate."""
    W = synth.make_weights(spec, seed=0, exclude=("embed",), **kw)
    W["embed"] = synth.make_normal_bf16((1235, spec.d_model), seed=77, std=0.02)
    return synth.weights_to_numpy(W)


@pytest.fixture(scope="module")
def layer():
    spec = synth.LLAMA8B_1L
    return spec, od.OracleDecoder(spec, _weights(spec))


def test_bf16_flip_cascade_reaches_the_stated_tolerance(layer, monkeypatch):
    spec, dec = layer
    rng = np.random.default_rng(4)
    c = 4000
    K = round_bf16(rng.standard_normal((c, spec.n_kv_heads, spec.head_dim)))
    V = round_bf16(rng.standard_normal((c, spec.n_kv_heads, spec.head_dim)))
    ref, _ = dec.step(np.array([1234]), [(K, V)])
    exact_attention = od.attention

    def perturbed(q, Kf, Vf, positions, window):
        # the exact attention output, off by 1e-5 relative before its rounding
        n, Hq, hd = q.shape
        rep = Hq // Kf.shape[1]
        out = np.empty((n, Hq, hd))
        for t in range(n):
            p = int(positions[t])
            for h in range(Hq):
                s = (Kf[:p + 1, h // rep] @ q[t, h]) / math.sqrt(hd)
                e = np.exp(s - s.max())
                out[t, h] = (e / e.sum()) @ Vf[:p + 1, h // rep]
        out *= 1 + 1e-5 * np.random.default_rng(99).standard_normal(out.shape)
        return round_bf16(out)

    monkeypatch.setattr(od, "attention", perturbed)
    alt, _ = dec.step(np.array([1234]), [(K, V)])
    monkeypatch.setattr(od, "attention", exact_attention)
    d = np.abs(alt - ref)
    assert 5e-3 < d.max() < 5e-2, d.max()


def test_gemma_block_flip_cascade_is_wider(monkeypatch):
    """The same measurement on the Gemma-3-4B-shaped block (2 layers, one
    local window-1024 and one global; embedding scale, (1 + w) gains,
    sandwich norms, vocab 262144).  A single 1e-5 disagreement already puts
    logits beyond the stated tolerance (17 of 262144 here, against 3 of
    128256 for the 8B-shaped layer): the same order as all that a 99.99 %
    criterion allows (26), while the GPU differs from the oracle in many
    roundings, not one.  That is why the full-size Gemma check asks for
    99.9 % (and twice the tolerance everywhere)."""
    spec = synth.GEMMA3_4B.with_(name="gemma3-4b-shape-2layer", n_layers=2, local_global_period=2)
    dec = od.OracleDecoder(spec, _weights(spec, gain_std=0.1))
    rng = np.random.default_rng(4)
    c = 4000
    cache = [(round_bf16(rng.standard_normal((c, spec.n_kv_heads, spec.head_dim))),
              round_bf16(rng.standard_normal((c, spec.n_kv_heads, spec.head_dim)))) for _ in range(2)]
    ref, _ = dec.step(np.array([1234]), cache)
    exact_attention = od.attention

    def perturbed(q, Kf, Vf, positions, window):
        n, Hq, hd = q.shape
        rep = Hq // Kf.shape[1]
        out = np.empty((n, Hq, hd))
        for t in range(n):
            p = int(positions[t])
            lo = max(0, p - window + 1) if window > 0 else 0
            for h in range(Hq):
                s = (Kf[lo:p + 1, h // rep] @ q[t, h]) / math.sqrt(hd)
                e = np.exp(s - s.max())
                out[t, h] = (e / e.sum()) @ Vf[lo:p + 1, h // rep]
        out *= 1 + 1e-5 * np.random.default_rng(99).standard_normal(out.shape)
        return round_bf16(out)

    monkeypatch.setattr(od, "attention", perturbed)
    alt, _ = dec.step(np.array([1234]), cache)
    monkeypatch.setattr(od, "attention", exact_attention)
    d = np.abs(alt - ref)[0]
    tol = 2e-2 + 1e-2 * np.abs(ref[0])
    beyond = int((d > tol).sum())
    assert 1e-2 < d.max() < 5e-2, d.max()
    assert 0.5e-4 * d.size < beyond < 1e-3 * d.size, beyond
    assert np.all(d <= 2 * tol)
