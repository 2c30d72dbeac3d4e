"""Pins of the fp64 oracle against what the pages and the mathematics fix.

CPU only. Each test names the passage it follows. A plausible mistake in the
oracle (a dropped term, a wrong sign or index, a transposed state, the gate
on the wrong side of the prediction) fails at least one of them.
"""
import json
from pathlib import Path

import numpy as np
import pytest

import oracle
from oracle import chunked
from gated_deltanet_chunkwise_gb300 import inputs

GOLD = Path(__file__).resolve().parent / "golden"


def gold(name):
    return json.loads((GOLD / name).read_text())


def one_head(q, k, v, g, beta, h0=None, variant=oracle.G1):
    """Run the oracle on a single sequence/head given [T, d] arrays."""
    q = np.asarray(q, float)[None, :, None, :]
    k = np.asarray(k, float)[None, :, None, :]
    v = np.asarray(v, float)[None, :, None, :]
    g = np.asarray(g, float)[None, :, None]
    beta = np.asarray(beta, float)[None, :, None]
    if h0 is not None:
        h0 = np.asarray(h0, float)[None, None]
    out, hT = oracle.forward(q, k, v, g, beta, h0=h0, variant=variant)
    return out[0, :, 0, :], hT[0, 0]


# --------------------------------------------------------------------------
# Worked numbers printed on the pages
# --------------------------------------------------------------------------

def test_delta_rule_1d_half_and_full_step():
    d = gold("delta_rule_1d.json")
    for case in ("beta_half", "beta_one"):
        b = d[case]["beta"]
        o, _ = one_head([[d["q"]]] * 3, [[d["k"]]] * 3, [[d["v"]]] * 3,
                        [0.0] * 3, [b] * 3)
        np.testing.assert_allclose(o[:, 0], d[case]["reads"], rtol=0, atol=1e-15)
    # beta -> 0 limit must not be the additive 3, 6, 9 of plain accumulation
    assert not np.allclose(o[:, 0], d["additive_contrast"]["reads"])


def test_deltanet_2d_example():
    d = gold("deltanet_2d.json")
    T = len(d["outputs"])
    for variant in (oracle.G1, oracle.G0):  # alpha = 1: both forms coincide
        o, _ = one_head([d["q"]] * T, [d["k"]] * T, [d["v"]] * T, [0.0] * T,
                        [d["beta"]] * T, variant=variant)
        np.testing.assert_allclose(o, d["outputs"], rtol=0, atol=1e-15)


def test_prediction_error_and_state_orientation():
    """The state rows are value features; storage holds the transpose.

    With beta = 1 and q = k the read equals the target; with q = (0, 1) the
    read is the untouched second key column of S; the final state differs from
    S only by error * k^T."""
    d = gold("prediction_error.json")
    S = np.array(d["S_value_by_key"])
    k = np.array(d["k"])
    err = np.array(d["v"]) - S @ k
    np.testing.assert_allclose(S @ k, d["prediction"])
    np.testing.assert_allclose(err, d["error"])
    for beta in (1.0, 0.5, 0.25):
        o, ZT = one_head([[0.0, 1.0]], [d["k"]], [d["v"]], [0.0], [beta],
                         h0=S.T)
        expect = S + beta * np.outer(np.array(d["error"]), k)
        np.testing.assert_allclose(ZT, expect.T, rtol=0, atol=1e-15)
        np.testing.assert_allclose(o[0], expect @ np.array([0.0, 1.0]),
                                   rtol=0, atol=1e-15)
        o2, _ = one_head([d["k"]], [d["k"]], [d["v"]], [0.0], [beta], h0=S.T)
        np.testing.assert_allclose(
            o2[0], (1 - beta) * np.array(d["prediction"]) + beta * np.array(d["v"]),
            rtol=0, atol=1e-15)


def test_gdn_gate_placement_3_7():
    d = gold("gdn_gate_placement.json")
    g = [np.log(d["alpha"])]
    o, hT = one_head([[1.0]], [[1.0]], [[d["target"]]], g, [d["beta"]],
                     h0=[[d["old_prediction"]]], variant=oracle.G1)
    assert o[0, 0] == pytest.approx(d["updated_prediction"], abs=1e-14)
    assert hT[0, 0] == pytest.approx(d["updated_prediction"], abs=1e-14)
    # the intermediate numbers of the same paragraph
    decayed = d["alpha"] * d["old_prediction"]
    assert decayed == pytest.approx(d["decayed_prediction"])
    assert d["target"] - decayed == pytest.approx(d["error"])
    # the other reading gives a different number, so the pin separates them
    o0, _ = one_head([[1.0]], [[1.0]], [[d["target"]]], g, [d["beta"]],
                     h0=[[d["old_prediction"]]], variant=oracle.G0)
    assert o0[0, 0] == pytest.approx(d["variant0_updated_prediction_derived"],
                                     abs=1e-14)


def test_wy_split_1d():
    d = gold("wy_split_1d.json")
    k = np.array([[d["k"]]])
    v = np.array([[d["v"]]])
    W, U0, Kbar, gamma, _ = chunked.wy_factors(k, v, np.zeros(1),
                                               np.array([d["beta"]]))
    assert W[0, 0] == pytest.approx(d["w"])
    assert U0[0, 0] == pytest.approx(d["u"])
    P1 = gamma - (W.T @ Kbar)[0, 0]
    assert P1 == pytest.approx(d["P1"])
    assert (U0.T @ Kbar)[0, 0] == pytest.approx(d["S1_from_zero"])
    # entry state 2: both the representation and the token loop give 2.5
    assert d["entry_state"] * P1 + d["S1_from_zero"] == pytest.approx(d["exit_state"])
    _, hT = one_head([[1.0]], k, v, [0.0], [d["beta"]], h0=[[d["entry_state"]]])
    assert hT[0, 0] == pytest.approx(d["exit_state"], abs=1e-15)


def test_gate_prefix_ratio_and_score():
    d = gold("gate_prefix.json")
    g = np.log(np.array(d["alpha"]))
    np.testing.assert_allclose(np.exp(chunked.local_cumsum(g)), d["b"])
    D = chunked.decay_matrix(g)
    assert D[2, 0] == pytest.approx(d["ratio_b3_over_b1"])
    # two-step cancellation: only alpha_2 survives at (2, 1); diagonal is 1
    assert D[1, 0] == pytest.approx(d["alpha"][1])
    np.testing.assert_allclose(np.diag(D), 1.0)
    assert D[0, 1] == 0.0 and D[0, 2] == 0.0 and D[1, 2] == 0.0
    q = np.zeros((3, 1)); k = np.zeros((3, 1))
    q[2, 0] = d["q3"]; k[0, 0] = d["k1"]
    assert chunked.gated_scores(q, k, g)[2, 0] == pytest.approx(d["score_3_1"])


# --------------------------------------------------------------------------
# Closed forms and invariants
# --------------------------------------------------------------------------

def _rand_head(rng, T, dk, dv, unit=True):
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    if unit:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    g = -np.logaddexp(0, rng.standard_normal(T))
    beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    return q, k, v, g, beta


@pytest.mark.parametrize("variant", [oracle.G1, oracle.G0])
def test_beta_zero_is_pure_decay(variant):
    rng = np.random.default_rng(1)
    q, k, v, g, _ = _rand_head(rng, 37, 5, 3)
    S0 = rng.standard_normal((5, 3))  # storage orientation
    o, hT = one_head(q, k, v, g, np.zeros(37), h0=S0, variant=variant)
    G = np.cumsum(g)
    np.testing.assert_allclose(hT, np.exp(G[-1]) * S0, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o, np.exp(G)[:, None] * (q @ S0), rtol=1e-12,
                               atol=1e-14)


def test_orthonormal_keys_full_step_overwrite():
    """alpha = 1, beta = 1, k_t = e_t: each write replaces the column of S
    along e_t by v_t exactly; S_T = S_0 (I - sum e e^T) + sum v_t e_t^T."""
    rng = np.random.default_rng(2)
    dk, dv, T = 6, 4, 4
    E = np.eye(dk)[:T]
    v = rng.standard_normal((T, dv))
    q = rng.standard_normal((T, dk))
    S0 = rng.standard_normal((dv, dk))  # math orientation
    _, hT = one_head(q, E, v, np.zeros(T), np.ones(T), h0=S0.T)
    expect = S0 @ (np.eye(dk) - E.T @ E) + v.T @ E
    np.testing.assert_allclose(hT.T, expect, rtol=0, atol=1e-14)


def test_single_token_rank1_update_alpha_one():
    """S_1 = S_0 + beta (v - S_0 k) k^T, o = S_1 q (math orientation)."""
    rng = np.random.default_rng(3)
    for dk, dv in [(1, 1), (3, 5), (8, 2)]:
        q, k, v, _, beta = _rand_head(rng, 1, dk, dv, unit=False)
        S0 = rng.standard_normal((dv, dk))
        S1 = S0 + beta[0] * np.outer(v[0] - S0 @ k[0], k[0])
        for variant in (oracle.G1, oracle.G0):
            o, hT = one_head(q, k, v, [0.0], beta, h0=S0.T, variant=variant)
            np.testing.assert_allclose(hT.T, S1, rtol=1e-14, atol=1e-14)
            np.testing.assert_allclose(o[0], S1 @ q[0], rtol=1e-13, atol=1e-14)


def test_unit_key_interpolation_invariant():
    """For |k| = 1: S_t k_t = (1 - beta) alpha S_{t-1} k_t + beta v_t (G1)."""
    rng = np.random.default_rng(4)
    dk, dv = 7, 3
    Z = rng.standard_normal((dk, dv))
    for _ in range(20):
        q, k, v, g, beta = _rand_head(rng, 1, dk, dv)
        _, Z1 = one_head(k, k, v, g, beta, h0=Z)
        lhs = Z1.T @ k[0]
        rhs = (1 - beta[0]) * np.exp(g[0]) * (Z.T @ k[0]) + beta[0] * v[0]
        np.testing.assert_allclose(lhs, rhs, rtol=1e-13, atol=1e-14)
        Z = Z1


@pytest.mark.parametrize("variant", [oracle.G1, oracle.G0])
def test_householder_bruteforce_small_T(variant):
    rng = np.random.default_rng(5)
    for T in range(1, 9):
        q, k, v, g, beta = _rand_head(rng, T, 4, 3, unit=(T % 2 == 0))
        S0 = rng.standard_normal((3, 4))
        o_ref, S_ref = chunked.householder_bruteforce(q, k, v, g, beta, S0,
                                                      variant)
        o, hT = one_head(q, k, v, g, beta, h0=S0.T, variant=variant)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(hT.T, S_ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Cross-derivations: affine composition, WY/UT chunks, sequence parallelism
# --------------------------------------------------------------------------

def _batch(seed, B=2, T=45, H=2, dk=8, dv=6, h0=True, lengths=None,
           gated=True):
    d = inputs.chunk_inputs(B, H, T, dk, dv, dtype="f32", seed=seed, h0=h0,
                            lengths=lengths, gated=gated)
    return d


def test_compose_is_associative():
    rng = np.random.default_rng(6)
    mk = lambda: (rng.standard_normal((5, 5)), rng.standard_normal((5, 3)))
    a, b, c = mk(), mk(), mk()
    l = chunked.compose(c, chunked.compose(b, a))
    r = chunked.compose(chunked.compose(c, b), a)
    np.testing.assert_allclose(l[0], r[0], rtol=1e-12)
    np.testing.assert_allclose(l[1], r[1], rtol=1e-12)
    # and it means "apply a, then b": check on a state
    Z = rng.standard_normal((5, 3))
    np.testing.assert_allclose(l[0] @ Z + l[1],
                               c[0] @ (b[0] @ (a[0] @ Z + a[1]) + b[1]) + c[1],
                               rtol=1e-12)


@pytest.mark.parametrize("variant", [oracle.G1, oracle.G0])
@pytest.mark.parametrize("chunk", [1, 4, 16, 45])
def test_affine_scan_equals_token_loop(variant, chunk):
    d = _batch(10)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o_ref, h_ref = oracle.forward(*args, variant=variant)
    o, h = chunked.affine_forward(*args, chunk=chunk, variant=variant)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h, h_ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("variant", [oracle.G1, oracle.G0])
@pytest.mark.parametrize("chunk", [1, 2, 8, 64, 100])
def test_wy_chunk_form_is_chunk_size_invariant(variant, chunk):
    d = _batch(11, T=100)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o_ref, h_ref = oracle.forward(*args, variant=variant)
    o, h = chunked.wy_forward(*args, chunk=chunk, variant=variant)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(h, h_ref, rtol=1e-10, atol=1e-11)


def test_wy_representation_of_chunk_transform():
    """P = prod alpha_t (I - beta_t k_t k_t^T) equals gamma I - W^T Kbar, and
    the zero-entry state equals U0^T Kbar (right-multiplied, math
    orientation)."""
    rng = np.random.default_rng(7)
    L, dk, dv = 9, 5, 4
    _, k, v, g, beta = _rand_head(rng, L, dk, dv)
    P = np.eye(dk)
    Sz = np.zeros((dv, dk))
    for t in range(L):
        Ht = np.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(k[t], k[t]))
        P = P @ Ht
        Sz = Sz @ Ht + beta[t] * np.outer(v[t], k[t])
    W, U0, Kbar, gamma, IA = chunked.wy_factors(k, v, g, beta)
    np.testing.assert_allclose(gamma * np.eye(dk) - W.T @ Kbar, P, rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose(U0.T @ Kbar, Sz, rtol=1e-12, atol=1e-13)
    # T = (I + A)^{-1} is unit lower triangular and inverts I + A
    Tm = np.linalg.inv(IA)
    np.testing.assert_allclose(np.triu(Tm, 1), 0, atol=1e-14)
    np.testing.assert_allclose(np.diag(Tm), 1, atol=1e-14)


@pytest.mark.parametrize("combine", ["chain", "scan"])
@pytest.mark.parametrize("parts", [2, 4, 8, 9])
@pytest.mark.parametrize("gated", [True, False])
def test_sequence_parallel_correction_equals_serial(parts, gated, combine):
    d = _batch(12, B=1, T=8 * 16 + 5, H=2, gated=gated)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o_ref, h_ref = oracle.forward(*args)
    o, h = chunked.sp_forward(*args, chunk=16, parts=parts, combine=combine)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(h, h_ref, rtol=1e-10, atol=1e-11)


def test_sp_difference_recursion():
    """S_[i+k] - dS_[i+k] = (S_[i] - dS_[i]) prod Phi (the CP derivation)."""
    rng = np.random.default_rng(8)
    dk, dv, L = 4, 3, 5
    Phis, Psis = [], []
    for _ in range(3):
        _, k, v, g, beta = _rand_head(rng, L, dk, dv)
        Phi, Psi = chunked.chunk_transform_phi_psi(k, v, g, beta)
        Phis.append(Phi); Psis.append(Psi)
    S = rng.standard_normal((dv, dk)); dS = np.zeros((dv, dk))
    diff0 = S - dS
    prod = np.eye(dk)
    for Phi, Psi in zip(Phis, Psis):
        S = S @ Phi + Psi; dS = dS @ Phi + Psi; prod = prod @ Phi
    np.testing.assert_allclose(S - dS, diff0 @ prod, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Resume, packing, ragged lengths
# --------------------------------------------------------------------------

def test_resume_through_final_state():
    d = _batch(13, B=2, T=70)
    q, k, v, g, beta, h0 = (d[x].double().numpy() for x in
                            ("q", "k", "v", "g", "beta", "h0"))
    o_all, h_all = oracle.forward(q, k, v, g, beta, h0)
    t = 29
    o1, h1 = oracle.forward(q[:, :t], k[:, :t], v[:, :t], g[:, :t],
                            beta[:, :t], h0)
    o2, h2 = oracle.forward(q[:, t:], k[:, t:], v[:, t:], g[:, t:],
                            beta[:, t:], h1)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), o_all, rtol=1e-13,
                               atol=1e-14)
    np.testing.assert_allclose(h2, h_all, rtol=1e-13, atol=1e-14)


def test_packed_sequences_equal_separate_calls():
    lengths = [5, 0, 33, 1, 64]
    d = _batch(14, B=len(lengths), H=3, lengths=lengths)
    q, k, v, g, beta, h0 = (d[x].double().numpy() for x in
                            ("q", "k", "v", "g", "beta", "h0"))
    cu = d["cu_seqlens"].numpy()
    o, h = oracle.forward(q, k, v, g, beta, h0, cu_seqlens=cu)
    for n, L in enumerate(lengths):
        s = slice(int(cu[n]), int(cu[n + 1]))
        on, hn = oracle.forward(q[:, s], k[:, s], v[:, s], g[:, s], beta[:, s],
                                h0[n:n + 1])
        np.testing.assert_allclose(o[:, s], on, rtol=0, atol=0)
        np.testing.assert_allclose(h[n:n + 1], hn, rtol=0, atol=0)
    # empty sequence: its final state is its initial state
    np.testing.assert_array_equal(h[1], h0[1])
    # and the chunk-form cross-check agrees on the packed layout
    o_w, h_w = chunked.wy_forward(q, k, v, g, beta, h0, cu_seqlens=cu, chunk=8)
    np.testing.assert_allclose(o_w, o, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(h_w, h, rtol=1e-10, atol=1e-11)


def test_recurrent_step_is_one_token():
    d = inputs.decode_inputs(3, 2, 8, 4, dtype="f32", seed=15)
    o, s = oracle.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                 d["state"])
    Z = d["state"].double().numpy()
    q, k, v = (d[x].double().numpy() for x in ("q", "k", "v"))
    a = np.exp(d["g"].double().numpy())
    b = d["beta"].double().numpy()
    for n in range(3):
        for h in range(2):
            S = Z[n, h].T * a[n, h]  # decay first (G1), math orientation
            u = b[n, h] * (v[n, h] - S @ k[n, h])
            S1 = S + np.outer(u, k[n, h])
            np.testing.assert_allclose(s[n, h], S1.T, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(o[n, h], S1 @ q[n, h], rtol=1e-13,
                                       atol=1e-14)


def test_oracle_rejects_bad_packing():
    d = _batch(16, B=2, lengths=[3, 4])
    cu = d["cu_seqlens"].numpy().copy()
    cu[1] = 9  # non-monotone / past the end
    with pytest.raises(ValueError):
        oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                       cu_seqlens=cu)


def test_map_scan_matches_left_fold():
    """The Hillis-Steele prefixes equal the left fold of the composition, and
    composing a map with the identity map (I, 0) changes nothing."""
    rng = np.random.default_rng(21)
    dk, dv = 5, 3
    maps = [(rng.standard_normal((dk, dk)), rng.standard_normal((dv, dk)))
            for _ in range(11)]
    pref = chunked.scan_maps(maps)
    S = rng.standard_normal((dv, dk))
    x = S
    for (M, dS), (Mp, dSp) in zip(maps, pref):
        x = x @ M + dS          # apply the maps one after another
        np.testing.assert_allclose(S @ Mp + dSp, x, rtol=1e-10, atol=1e-10)
    ident = (np.eye(dk), np.zeros((dv, dk)))
    for M, dS in chunked.scan_maps([ident, maps[0]])[-1:]:
        np.testing.assert_allclose(M, maps[0][0], atol=0)
        np.testing.assert_allclose(dS, maps[0][1], atol=0)
