"""Pins of the KDA oracle (oracle/kda.py) to the pages and to other forms.

- The walk-through's worked example (tests/golden/kda_example.json): column
  forgetting of diag(10, 20) with alpha = (0.9, 0.2) against the scalar 0.9,
  three forgetting steps, a mixed-direction read, and the delta step that
  turns diag(9, 4) into diag(9, 6).
- Equal decays on every channel reduce KDA to the scalar-gate recurrence
  with the decay before the prediction (the C token loop of oracle/).
- The generalised Householder product form S_T = S_0 H_1 .. H_T + sum_t
  beta_t v_t k_t^T H_{t+1} .. H_T with H_t = diag(alpha_t)(I - beta_t k_t
  k_t^T), by dense products on tiny inputs.
"""
import json
from pathlib import Path

import numpy as np
import pytest

import oracle
from oracle import kda

GOLD = json.loads((Path(__file__).parent / "golden" / "kda_example.json").read_text())


def _step(S, q, k, v, alpha, beta):
    return kda.step(np.array(S, float), np.array(q, float), np.array(k, float),
                    np.array(v, float), np.log(np.array(alpha, float)), beta)


def test_column_forgetting_example():
    S0 = GOLD["state"]
    z = [0.0, 0.0]
    for name, q in (("q_a", GOLD["q_a"]), ("q_b", GOLD["q_b"])):
        o, _ = _step(S0, q, z, z, [GOLD["alpha_gdn"]] * 2, 0.0)
        np.testing.assert_allclose(o, GOLD["read_after_gdn_forget"][name], atol=1e-12)
        o, _ = _step(S0, q, z, z, GOLD["alpha_kda"], 0.0)
        np.testing.assert_allclose(o, GOLD["read_after_kda_forget"][name], atol=1e-12)


def test_three_forgetting_steps_and_mixed_read():
    S = np.array(GOLD["state"], float)
    qm = np.array([1.0, 1.0]) / np.sqrt(2.0)
    z = [0.0, 0.0]
    o, _ = _step(S, qm, z, z, [1.0, 1.0], 0.0)
    np.testing.assert_allclose(o * np.sqrt(2), GOLD["mixed_q_read_before_times_sqrt2"], atol=1e-12)
    o, _ = _step(S, qm, z, z, GOLD["alpha_kda"], 0.0)
    np.testing.assert_allclose(o * np.sqrt(2), GOLD["mixed_q_read_after_times_sqrt2"], atol=1e-12)
    for _ in range(3):
        _, S = _step(S, z, z, z, GOLD["alpha_kda"], 0.0)
    np.testing.assert_allclose(S, GOLD["three_forget_steps_state"], atol=1e-12)


def test_delta_step_after_forgetting():
    w = GOLD["write_step"]
    # the forgetting of the example, then the write, in one step
    o, S = _step(GOLD["state"], w["k"], w["k"], w["v"], GOLD["alpha_kda"], w["beta"])
    np.testing.assert_allclose(S, w["state_after"], atol=1e-12)
    np.testing.assert_allclose(o, np.array(w["state_after"]) @ np.array(w["k"]), atol=1e-12)
    # the prediction the step corrects is the forgotten state's read of k
    Sb = np.array(GOLD["state"]) * np.array(GOLD["alpha_kda"])[None, :]
    np.testing.assert_allclose(Sb @ np.array(w["k"]), w["prediction"], atol=1e-12)


def _rand(seed, B, T, H, dk, dv):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, H))))
    h0 = 0.1 * rng.standard_normal((B, H, dk, dv))
    return q, k, v, beta, h0


@pytest.mark.parametrize("packed", [False, True])
def test_equal_channels_reduce_to_scalar_gate(packed):
    B, T, H, dk, dv = 2, 37, 2, 8, 5
    q, k, v, beta, h0 = _rand(3, B, T, H, dk, dv)
    rng = np.random.default_rng(4)
    g1 = -np.log1p(np.exp(rng.standard_normal((B, T, H))))
    g = np.repeat(g1[..., None], dk, axis=-1)
    cu = None
    if packed:
        q, k, v, g, g1, beta = (x.reshape(1, B * T, *x.shape[2:]) for x in (q, k, v, g, g1, beta))
        cu = np.array([0, 20, B * T])
    o_ref, h_ref = oracle.forward(q, k, v, g1, beta, h0, cu_seqlens=cu, variant=oracle.G1)
    o, h = kda.forward(q, k, v, g, beta, h0, cu_seqlens=cu)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(h, h_ref, rtol=1e-10, atol=1e-12)


def test_householder_product_form():
    T, dk, dv = 6, 4, 3
    q, k, v, beta, h0 = _rand(5, 1, T, 1, dk, dv)
    rng = np.random.default_rng(6)
    g = -np.abs(rng.standard_normal((1, T, 1, dk)))
    _, hT = kda.forward(q, k, v, g, beta, h0)
    S0 = h0[0, 0].T
    Hs = [np.diag(np.exp(g[0, t, 0])) @ (np.eye(dk) - beta[0, t, 0] * np.outer(k[0, t, 0], k[0, t, 0]))
          for t in range(T)]
    def prod(a, b):
        P = np.eye(dk)
        for t in range(a, b):
            P = P @ Hs[t]
        return P
    S = S0 @ prod(0, T)
    for t in range(T):
        S = S + beta[0, t, 0] * np.outer(v[0, t, 0], k[0, t, 0]) @ prod(t + 1, T)
    np.testing.assert_allclose(hT[0, 0].T, S, rtol=1e-10, atol=1e-12)
