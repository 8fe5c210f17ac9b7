"""Stored expected values from the pages' worked examples (tests/golden/).

Each fixture names the passage it comes from: the all-zero model's outputs
(all-zero logits, token id zero) and the prefix-comparability verdicts of
Definition 2.1's example (views of 50 and 30 tokens) with its variations.
The oracle and the library's Definition 2.1 checker are pinned to them.
"""

import os

import numpy as np

from invariant_vd_step_gb300 import invariance, synth
from oracle import decoder as od
from oracle import fp32 as oc
from oracle import sampler

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [line.split() for line in f if line.strip() and not line.startswith("#")]


def test_zero_model_outputs_match_the_golden_values():
    kv = dict(_rows("zero_model_outputs.txt"))
    want_bits, want_token = int(kv["logit_float32_bits"], 16), int(kv["greedy_token"])
    for spec, Oracle in ((s, o) for s in (synth.TINY, synth.TINY.with_(name="tiny-window", sliding_window=8,
                                                                           local_global_period=2))
                         for o in (od.OracleDecoder, oc.Fp32Decoder)):
        dec = Oracle(spec, synth.weights_to_numpy(synth.make_weights(spec, zero=True)))
        for seed, n in ((3, 1), (4, 17), (5, 40)):
            logits = dec.forward(synth.make_tokens(n, spec.vocab, seed=seed))
            bits = np.asarray(logits, dtype=np.float32).view(np.uint32)
            assert np.all(bits == want_bits), (spec.name, n)
            assert sampler.argmax_lowest(logits) == want_token
            assert sampler.sample(logits, 0.0, seed, 0) == want_token


def test_definition_2_1_checker_matches_the_golden_verdicts():
    rows = _rows("prefix_comparable_views.txt")
    header, cases = rows[0], rows[1:]
    assert header == ["case", "len_a", "len_b", "altered", "index", "comparable"]
    rng = np.random.default_rng(0)
    base = [(rng.standard_normal(16).astype(np.float32), int(rng.integers(0, 100))) for _ in range(64)]
    assert len(cases) >= 8
    for name, la, lb, altered, idx, verdict in cases:
        a = [(l.copy(), t) for l, t in base[:int(la)]]
        b = [(l.copy(), t) for l, t in base[:int(lb)]]
        i = int(idx)
        if altered == "A":
            a[i][0][3] = np.nextafter(a[i][0][3], np.float32(np.inf))  # one ulp on one logit
        elif altered == "B":
            b[i][0][3] = np.nextafter(b[i][0][3], np.float32(np.inf))
        elif altered == "B_token":
            b[i] = (b[i][0], b[i][1] + 1)
        want = verdict == "true"
        assert invariance.prefix_comparable(a, b) is want, name
        assert invariance.prefix_comparable(b, a) is want, name  # the relation is symmetric
