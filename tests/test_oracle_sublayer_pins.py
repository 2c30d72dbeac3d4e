"""Pins of the oracle's steps either side of the recurrence (oracle/sublayer.py).

Worked numbers of the illustrated DeltaNet page (tests/golden/
sublayer_norms.json) and closed forms; each check would fail for a plausible
slip (normalising across tokens or heads instead of per (token, head), the
wrong denominator, a sign in the gate parameterisation).
"""
import json
import math
from pathlib import Path

import numpy as np

import oracle
from oracle import sublayer

GOLD = json.loads((Path(__file__).resolve().parent / "golden" /
                   "sublayer_norms.json").read_text())


def test_l2_norm_worked_example():
    x = np.array(GOLD["x"])
    assert np.allclose(sublayer.l2_normalize(x), GOLD["l2"]["out"])
    assert math.isclose(np.linalg.norm(x), GOLD["l2"]["denominator"])


def test_rms_norm_worked_example():
    x = np.array(GOLD["x"])
    d = GOLD["rms"]["decimals"]
    assert np.allclose(np.round(sublayer.rms_norm(x), d), GOLD["rms"]["out"])
    assert round(math.sqrt(np.mean(x * x)), d) == GOLD["rms"]["denominator"]


def test_norms_are_per_token():
    toks = np.array(GOLD["per_token"]["tokens"])          # two tokens
    l2 = sublayer.l2_normalize(toks)
    assert np.allclose(l2[0], l2[1]) and np.allclose(l2[0], GOLD["l2"]["out"])
    assert np.allclose(np.linalg.norm(toks, axis=-1),
                       GOLD["per_token"]["l2_denominators"])
    rms = sublayer.rms_norm(toks)
    assert np.allclose(rms[0], rms[1])                    # same ratios, same output
    # different ratios stay distinguishable
    assert not np.allclose(sublayer.rms_norm(np.array([4.0, 3.0])), rms[0])


def test_rms_and_l2_differ_by_sqrt_d():
    x = np.random.default_rng(0).standard_normal((5, 3, 128))
    assert np.allclose(sublayer.rms_norm(x), sublayer.l2_normalize(x) * math.sqrt(128))
    assert np.allclose(np.mean(sublayer.rms_norm(x) ** 2, axis=-1), 1.0)
    w = np.linspace(0.5, 2.0, 128)
    assert np.allclose(sublayer.rms_norm(x, w), sublayer.rms_norm(x) * w)


def test_gate_activations_closed_forms():
    x = np.linspace(-30, 30, 121)
    assert sublayer.sigmoid(0.0) == 0.5
    assert np.allclose(sublayer.sigmoid(x) + sublayer.sigmoid(-x), 1.0)
    assert math.isclose(sublayer.softplus(0.0), math.log(2.0))
    assert np.allclose(sublayer.softplus(x) - sublayer.softplus(-x), x)
    # alpha = e^{-softplus(a)} = 1 / (1 + e^a) = sigmoid(-a): a gate in (0, 1)
    assert np.allclose(np.exp(-sublayer.softplus(x)), sublayer.sigmoid(-x))
    assert math.isclose(sublayer.softplus(800.0), 800.0)  # no overflow


def test_zero_vector_stays_zero():
    assert np.all(sublayer.l2_normalize(np.zeros(8)) == 0)


def _raw(B, H, T, d, seed):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s)
    return f(B, T, H, d), f(B, T, H, d), f(B, T, H, d), f(B, T, H), f(B, T, H)


def test_fused_forward_invariants():
    q, k, v, a, b = _raw(1, 2, 40, 16, 1)
    ones = np.ones(16)
    out, hT = sublayer.fused_forward(q, k, v, a, b, weight=ones, eps=0.0)
    # the recurrence sees unit q, k: scaling the raw vectors changes nothing
    out2, hT2 = sublayer.fused_forward(3.0 * q, 0.25 * k, v, a, b, weight=ones,
                                       eps=0.0)
    assert np.allclose(out, out2) and np.allclose(hT, hT2)
    # output RMS is 1 per (token, head) with a unit weight and no gate
    assert np.allclose(np.mean(out ** 2, axis=-1), 1.0)
    # the gate multiplies elementwise; an all-zero gate logit halves the output
    out3, _ = sublayer.fused_forward(q, k, v, a, b, weight=ones,
                                     gate=np.zeros_like(v), eps=0.0)
    assert np.allclose(out3, 0.5 * out)
    # without weight and gate the read-out is passed through unchanged
    o_plain, _ = sublayer.fused_forward(q, k, v, a, b)
    assert np.allclose(o_plain * np.sqrt(np.mean(o_plain ** 2, axis=-1,
                                                  keepdims=True)) ** -1, out)
    # the recurrence between the two is the oracle's, on the activated inputs
    o_ref, h_ref = oracle.forward(q / np.linalg.norm(q, axis=-1, keepdims=True),
                                  k / np.linalg.norm(k, axis=-1, keepdims=True),
                                  v, -np.log1p(np.exp(a)), 1 / (1 + np.exp(-b)))
    assert np.allclose(hT, h_ref)
