"""Pins of the gradient oracle (oracle/backward.py) against things other than
itself: central finite differences of the loss through the forward oracles
(oracle.kda.forward and the C token loop oracle.forward), closed forms, and
automatic differentiation of an independent PyTorch statement of the forward
map. The loss is L = sum(dout * out) + sum(dhT * hT).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward, kda

NAMES = ("q", "k", "v", "g", "beta", "h0")


def rand_case(B, T, H, dk, dv, seed, *, packed=None, scalar=False):
    rng = np.random.default_rng(seed)
    rows = B * T if packed is None else sum(packed)
    shape = lambda d: (1, rows, H, d) if packed is not None else (B, T, H, d)
    N = B if packed is None else len(packed)
    c = {
        "q": rng.normal(size=shape(dk)), "k": rng.normal(size=shape(dk)) / np.sqrt(dk),
        "v": rng.normal(size=shape(dv)),
        "g": (-rng.uniform(0.05, 1.0, size=shape(1)[:-1]) if scalar
              else -rng.uniform(0.05, 1.0, size=shape(dk))),
        "beta": rng.uniform(0.1, 0.9, size=shape(1)[:-1]),
        "h0": rng.normal(size=(N, H, dk, dv)),
        "dout": rng.normal(size=shape(dv)), "dhT": rng.normal(size=(N, H, dk, dv)),
        "cu": None if packed is None else np.concatenate([[0], np.cumsum(packed)]).astype(np.int32),
    }
    return c


def loss(c, fwd, **over):
    x = {n: over.get(n, c[n]) for n in NAMES}
    out, hT = fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], cu_seqlens=c["cu"])
    return float((c["dout"] * out).sum() + (c["dhT"] * hT).sum())


def finite_difference(c, fwd, name, eps=1e-6):
    base = c[name]
    grad = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = base.copy(), base.copy()
        xp[i] += eps
        xm[i] -= eps
        grad[i] = (loss(c, fwd, **{name: xp}) - loss(c, fwd, **{name: xm})) / (2 * eps)
    return grad


def check_fd(c, grads, fwd):
    for name in NAMES:
        fd = finite_difference(c, fwd, name)
        an = grads["d" + name]
        scale = max(np.abs(fd).max(), 1e-12)
        assert np.abs(an - fd).max() / scale < 1e-6, name


def test_kda_gradients_match_finite_differences():
    c = rand_case(2, 5, 2, 3, 2, seed=1)
    grads = backward.kda_backward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                                  c["h0"], c["dout"], c["dhT"])
    check_fd(c, grads, kda.forward)


def test_kda_gradients_packed_match_finite_differences():
    c = rand_case(0, 0, 1, 3, 2, seed=2, packed=[3, 0, 4, 1])
    grads = backward.kda_backward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                                  c["h0"], c["dout"], c["dhT"],
                                  cu_seqlens=c["cu"])
    check_fd(c, grads, kda.forward)
    # the empty sequence: its state passes straight through
    assert np.array_equal(grads["dh0"][1], c["dhT"][1])


def test_scalar_gate_gradients_match_finite_differences_of_the_c_oracle():
    """The scalar-gate wrapper against the independent C token loop (decay
    before the prediction)."""
    c = rand_case(2, 6, 1, 3, 2, seed=3, scalar=True)
    grads = backward.backward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                              c["h0"], c["dout"], c["dhT"])
    fwd = lambda *a, cu_seqlens=None: oracle.forward(*a, cu_seqlens=cu_seqlens,
                                                     variant=oracle.G1)
    check_fd(c, grads, fwd)


def test_g0_placement_gradients_match_finite_differences_of_the_c_oracle():
    """The other gate placement (predict with the undecayed state, then
    decay) against the C token loop with variant G0."""
    c = rand_case(2, 6, 1, 3, 2, seed=7, scalar=True)
    grads = backward.backward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                              c["h0"], c["dout"], c["dhT"], variant=oracle.G0)
    fwd = lambda *a, cu_seqlens=None: oracle.forward(*a, cu_seqlens=cu_seqlens,
                                                     variant=oracle.G0)
    check_fd(c, grads, fwd)


def test_g0_and_g1_gradients_agree_without_decay():
    """g = 0: the two placements are the same map (plain DeltaNet), so all
    gradients but dg agree (dg does not: the maps differ for g != 0)."""
    c = rand_case(1, 6, 2, 4, 3, seed=8, scalar=True)
    c["g"][:] = 0.0
    g1 = backward.backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                           c["dout"], c["dhT"], variant=oracle.G1)
    g0 = backward.backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"],
                           c["dout"], c["dhT"], variant=oracle.G0)
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        assert np.allclose(g0[n], g1[n], atol=1e-12), n
    assert not np.allclose(g0["dg"], g1["dg"])


def test_closed_form_without_writes_or_decay():
    """beta = 0, g = 0: S_t = S_0 for every t, so dq_t = S_0^T dout_t,
    dh0 = dhT + sum_t q_t dout_t^T (as d_k x d_v), dk = dv = 0, and with
    dS_t = dhT^T + sum_{s >= t} dout_s q_s^T: dbeta_t = (dS_t k_t) . (v_t -
    S_0 k_t) and dg_t = column sums of dS_t (.) S_0."""
    c = rand_case(1, 7, 1, 4, 3, seed=4)
    c["beta"][:] = 0.0
    c["g"][:] = 0.0
    gr = backward.kda_backward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                               c["h0"], c["dout"], c["dhT"])
    S0 = c["h0"][0, 0].T
    q, k, v, do = (c[n][0, :, 0] for n in ("q", "k", "v", "dout"))
    assert np.allclose(gr["dq"][0, :, 0], do @ S0, atol=1e-12)
    assert np.allclose(gr["dh0"][0, 0], c["dhT"][0, 0] + q.T @ do, atol=1e-12)
    for n in ("dk", "dv"):
        assert np.abs(gr[n]).max() == 0.0
    dS = c["dhT"][0, 0].T.copy()
    expect, expect_g = np.zeros(7), np.zeros((7, 4))
    for t in range(6, -1, -1):
        dS = dS + np.outer(do[t], q[t])
        expect[t] = (dS @ k[t]) @ (v[t] - S0 @ k[t])
        expect_g[t] = (dS * S0).sum(axis=0)
    assert np.allclose(gr["dbeta"][0, :, 0], expect, atol=1e-12)
    assert np.allclose(gr["dg"][0, :, 0], expect_g, atol=1e-12)


def torch_forward(q, k, v, g, beta, h0):
    """Independent statement of the forward map in PyTorch (fp64), state
    d_k x d_v as on the lqnn.cn page: S <- diag(a) S, e = v - S^T k,
    S <- S + beta k e^T, o = S^T q."""
    B, T, H, dk = q.shape
    outs, hTs = [], []
    for n in range(B):
        for h in range(H):
            S = h0[n, h]
            o = []
            for t in range(T):
                S = torch.exp(g[n, t, h])[:, None] * S
                e = v[n, t, h] - S.T @ k[n, t, h]
                S = S + beta[n, t, h] * torch.outer(k[n, t, h], e)
                o.append(S.T @ q[n, t, h])
            outs.append(torch.stack(o))
            hTs.append(S)
    out = torch.stack(outs).reshape(B, H, T, -1).permute(0, 2, 1, 3)
    return out, torch.stack(hTs).reshape(B, H, dk, -1)


def test_gradients_match_autograd_of_an_independent_forward():
    c = rand_case(2, 12, 2, 6, 5, seed=5)
    ts = {n: torch.tensor(c[n], requires_grad=True) for n in NAMES}
    out, hT = torch_forward(*(ts[n] for n in NAMES))
    L = (torch.tensor(c["dout"]) * out).sum() + (torch.tensor(c["dhT"]) * hT).sum()
    L.backward()
    gr = backward.kda_backward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                               c["h0"], c["dout"], c["dhT"])
    for n in NAMES:
        ref = ts[n].grad.numpy()
        assert np.abs(gr["d" + n] - ref).max() <= 1e-9 * max(np.abs(ref).max(), 1.0), n


@pytest.mark.parametrize("plant", ["drop_decay_in_dS", "sign_dk", "no_beta_in_dv"])
def test_a_planted_mistake_is_caught(plant):
    """A copy of the sweep with one plausible mistake fails the finite-
    difference pin (so the pin can see such mistakes)."""
    c = rand_case(1, 4, 1, 3, 2, seed=6)
    g0 = backward.kda_backward(c["q"], c["k"], c["v"], c["g"], c["beta"],
                               c["h0"], c["dout"], c["dhT"])
    bad = {k_: v_.copy() for k_, v_ in g0.items()}
    if plant == "drop_decay_in_dS":
        bad["dh0"] = bad["dh0"] / np.exp(c["g"][0, 0, 0])[:, None]
    elif plant == "sign_dk":
        bad["dk"] = -bad["dk"]
    else:
        bad["dv"] = bad["dv"] / c["beta"][..., None]
    with pytest.raises(AssertionError):
        check_fd(c, bad, kda.forward)


@pytest.mark.parametrize("weight,gate", [(True, True), (True, False),
                                         (False, True), (False, False)])
def test_fused_gradients_match_finite_differences(weight, gate):
    """The steps either side of the recurrence (L2 norms, softplus and
    sigmoid activations, RMSNorm with a weight, sigmoid output gate) against
    central differences through the fused forward oracle."""
    from oracle import sublayer
    rng = np.random.default_rng(9)
    B, T, H, dk, dv = 2, 5, 1, 3, 4
    c = {"q": rng.normal(size=(B, T, H, dk)) * 2.0,
         "k": rng.normal(size=(B, T, H, dk)),
         "v": rng.normal(size=(B, T, H, dv)),
         "a": rng.normal(size=(B, T, H)), "b": rng.normal(size=(B, T, H)),
         "h0": rng.normal(size=(B, H, dk, dv)),
         "w": 1.0 + 0.3 * rng.normal(size=dv) if weight else None,
         "z": rng.normal(size=(B, T, H, dv)) if gate else None}
    dout = rng.normal(size=(B, T, H, dv))
    dhT = rng.normal(size=(B, H, dk, dv))
    names = ["q", "k", "v", "a", "b", "h0"] + (["w"] if weight else []) + (["z"] if gate else [])

    def L(**over):
        x = {n: over.get(n, c[n]) for n in c}
        out, hT = sublayer.fused_forward(x["q"], x["k"], x["v"], x["a"], x["b"],
                                         x["h0"], weight=x["w"], gate=x["z"],
                                         eps=1e-6)
        return float((dout * out).sum() + (dhT * hT).sum())

    got = backward.fused_backward(c["q"], c["k"], c["v"], c["a"], c["b"], c["h0"],
                                  dout, dhT, weight=c["w"], gate=c["z"], eps=1e-6)
    key = {"q": "dq", "k": "dk", "v": "dv", "a": "da", "b": "db", "h0": "dh0",
           "w": "dweight", "z": "dgate"}
    for n in names:
        base = c[n]
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp, xm = base.copy(), base.copy()
            xp[i] += 1e-6
            xm[i] -= 1e-6
            fd[i] = (L(**{n: xp}) - L(**{n: xm})) / 2e-6
        an = got[key[n]]
        assert np.abs(an - fd).max() / max(np.abs(fd).max(), 1e-12) < 1e-6, n
