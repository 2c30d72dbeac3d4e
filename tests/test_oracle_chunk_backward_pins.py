"""Pins of the chunk-form adjoint (oracle/chunked_backward.py): chunk by
chunk it must give the gradients of the token-by-token reverse sweep
(oracle.backward, pinned to finite differences in
tests/test_oracle_backward_pins.py) at every chunk size, for dense and packed
inputs, and stay finite under decays far stronger than one chunk can span in
floating point. The loss is L = sum(dout * out) + sum(dhT * hT)."""
import numpy as np
import pytest

from oracle import backward, chunked_backward

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def case(B, T, H, dk, dv, seed, *, packed=None, g_scale=1.0):
    rng = np.random.default_rng(seed)
    rows = B * T if packed is None else sum(packed)
    shape = (lambda d: (1, rows, H, d)) if packed is not None else (lambda d: (B, T, H, d))
    N = B if packed is None else len(packed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    return {
        "q": unit(rng.normal(size=shape(dk))), "k": unit(rng.normal(size=shape(dk))),
        "v": rng.normal(size=shape(dv)),
        "g": -g_scale * np.log1p(np.exp(rng.normal(size=shape(1)[:-1]))),
        "beta": 1 / (1 + np.exp(-rng.normal(size=shape(1)[:-1]))),
        "h0": 0.1 * rng.normal(size=(N, H, dk, dv)),
        "dout": rng.normal(size=shape(dv)), "dhT": 0.1 * rng.normal(size=(N, H, dk, dv)),
        "cu": None if packed is None else np.concatenate([[0], np.cumsum(packed)]).astype(np.int32),
    }


def both(c, C):
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], c["h0"], c["dout"], c["dhT"])
    ref = backward.backward(*args, cu_seqlens=c["cu"], variant=1)
    got = chunked_backward.chunk_backward(*args, cu_seqlens=c["cu"], C=C)
    return got, ref


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("C", [1, 5, 16, 64, 150])
def test_chunk_adjoint_equals_the_token_sweep(C):
    got, ref = both(case(2, 150, 2, 16, 12, seed=1), C)
    for n in GRADS:
        assert rel(got[n], ref[n]) < 1e-11, (n, C)


def test_chunk_adjoint_packed():
    got, ref = both(case(0, 0, 2, 16, 8, seed=2, packed=[37, 0, 1, 64, 90]), 16)
    for n in GRADS:
        assert rel(got[n], ref[n]) < 1e-11, n


def test_chunk_adjoint_under_strong_decay():
    # g around -30 per token: e^{G} underflows within a chunk, yet every factor
    # the adjoint forms is a ratio of decays at most 1
    got, ref = both(case(1, 100, 1, 8, 8, seed=3, g_scale=30.0), 64)
    for n in GRADS:
        assert np.isfinite(got[n]).all(), n
        assert rel(got[n], ref[n]) < 1e-10, n


def test_chunk_adjoint_first_and_last_chunk_terms():
    # without h0 and dhT the entry-state and exit-gradient terms vanish; with
    # them every term of the chunk boundary is exercised (a dropped one shows)
    c = case(1, 130, 1, 8, 8, seed=4)
    for h0, dhT in ((None, None), (c["h0"], None), (None, c["dhT"])):
        cc = dict(c, h0=h0, dhT=dhT)
        got, ref = both(cc, 64)
        for n in GRADS:
            assert rel(got[n], ref[n]) < 1e-11, n
