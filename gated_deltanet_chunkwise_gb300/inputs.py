"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: it only draws random numbers
and shapes them into the distributions of the workloads (q, k ~ N(0, 1) then
L2-normalised per token and head; v ~ N(0, 1); beta = sigmoid(N(0, 1));
g = log alpha = -softplus(N(0, 1)); h0 ~ 0.1 N(0, 1)). Draws come from one
numpy PCG64 stream per call (platform independent) in the fixed order
lengths (packed batches only), q, k, v, g, beta, h0, all drawn in fp32.
q, k and v are then rounded to the compute dtype (round-to-nearest-even);
g, beta and the states stay fp32.
"""
from __future__ import annotations

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def _unit_rows(x):
    # fp32 L2 normalisation over the last axis, no epsilon (N(0,1) rows are
    # never zero).
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return (x / n).astype(np.float32)


def _softplus(x):
    return np.logaddexp(np.float32(0), x).astype(np.float32)


def _sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def chunk_inputs(B, H, T, dk, dv, *, dtype="bf16", seed=0, gated=True,
                 h0=False, lengths=None, length_range=None):
    """Inputs for the chunked forward pass, as CPU torch tensors.

    Dense batch: q, k [B, T, H, dk], v [B, T, H, dv], g, beta [B, T, H].
    Packed batch (``lengths`` given as a list, or ``length_range=(lo, hi)``
    with B sequences drawn uniform inclusive): tensors are [1, sum(len), H, ...]
    with ``cu_seqlens`` int32 [B + 1]. ``gated=False`` sets g = 0 (alpha = 1,
    plain DeltaNet) after drawing it, so both runs share q, k, v and beta.
    ``h0=True`` draws initial states [N, H, dk, dv] ~ 0.1 N(0, 1).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    cu = None
    if length_range is not None:
        lo, hi = length_range
        lengths = rng.integers(lo, hi + 1, size=B).tolist()
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        N = len(lengths)
        cu = np.zeros(N + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        Bt, Tt = 1, int(cu[-1])
    else:
        N, Bt, Tt = B, B, T
    q = _unit_rows(_normal(rng, (Bt, Tt, H, dk)))
    k = _unit_rows(_normal(rng, (Bt, Tt, H, dk)))
    v = _normal(rng, (Bt, Tt, H, dv))
    g = -_softplus(_normal(rng, (Bt, Tt, H)))
    beta = _sigmoid(_normal(rng, (Bt, Tt, H)))
    if not gated:
        g = np.zeros_like(g)
    s0 = (np.float32(0.1) * _normal(rng, (N, H, dk, dv))) if h0 else None
    tdt = DTYPES[dtype]
    out = {
        "q": torch.from_numpy(q).to(tdt),
        "k": torch.from_numpy(k).to(tdt),
        "v": torch.from_numpy(v).to(tdt),
        "g": torch.from_numpy(g),
        "beta": torch.from_numpy(beta),
        "h0": None if s0 is None else torch.from_numpy(s0),
        "cu_seqlens": None if cu is None else torch.from_numpy(cu),
    }
    return out


def decode_inputs(N, H, dk, dv, *, dtype="bf16", seed=0):
    """One token per (sequence, head) plus an fp32 state ~ 0.1 N(0, 1).

    q, k [N, H, dk] (unit rows), v [N, H, dv], g, beta [N, H], state
    [N, H, dk, dv]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _unit_rows(_normal(rng, (N, H, dk)))
    k = _unit_rows(_normal(rng, (N, H, dk)))
    v = _normal(rng, (N, H, dv))
    g = -_softplus(_normal(rng, (N, H)))
    beta = _sigmoid(_normal(rng, (N, H)))
    state = np.float32(0.1) * _normal(rng, (N, H, dk, dv))
    tdt = DTYPES[dtype]
    return {
        "q": torch.from_numpy(q).to(tdt),
        "k": torch.from_numpy(k).to(tdt),
        "v": torch.from_numpy(v).to(tdt),
        "g": torch.from_numpy(g),
        "beta": torch.from_numpy(beta),
        "state": torch.from_numpy(state),
    }


def fused_inputs(B, H, T, dk, dv, *, seed=0, h0=False, lengths=None,
                 weight=True, gate=True):
    """Raw inputs of gdn_chunk_fwd_fused: q and k NOT normalised (each row
    an N(0, 1) vector times a length drawn from U[0.25, 4)), v ~ N(0, 1),
    gate logits a and step logits b ~ N(0, 1) (fp32), h0 ~ 0.1 N(0, 1), the
    output norm weight 1 + 0.1 N(0, 1) (fp32 [dv]) and the output gate
    logits ~ N(0, 1) (bf16, like v). Draw order: lengths, q, q lengths, k,
    k lengths, v, a, b, h0, weight, gate."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        N = len(lengths)
        cu = np.zeros(N + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        Bt, Tt = 1, int(cu[-1])
    else:
        N, Bt, Tt, cu = B, B, T, None
    q = _normal(rng, (Bt, Tt, H, dk))
    q *= rng.uniform(0.25, 4.0, (Bt, Tt, H, 1)).astype(np.float32)
    k = _normal(rng, (Bt, Tt, H, dk))
    k *= rng.uniform(0.25, 4.0, (Bt, Tt, H, 1)).astype(np.float32)
    v = _normal(rng, (Bt, Tt, H, dv))
    a = _normal(rng, (Bt, Tt, H))
    b = _normal(rng, (Bt, Tt, H))
    h = (0.1 * _normal(rng, (N, H, dk, dv))).astype(np.float32) if h0 else None
    w = (1.0 + 0.1 * _normal(rng, (dv,))).astype(np.float32) if weight else None
    z = _normal(rng, (Bt, Tt, H, dv)) if gate else None
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
    bf = lambda x: t(x).to(torch.bfloat16)
    return {
        "q": bf(q), "k": bf(k), "v": bf(v), "a": t(a), "b": t(b),
        "h0": None if h is None else t(h),
        "cu_seqlens": None if cu is None else t(cu),
        "norm_weight": None if w is None else t(w),
        "gate": None if z is None else bf(z),
    }


def kda_inputs(B, H, T, dk, dv, *, seed=0, h0=False, lengths=None,
               length_range=None):
    """Inputs for the per-channel-decay recurrence (gdn_kda_fwd): as
    ``chunk_inputs`` (bf16 q, k unit rows, v; fp32 beta; optional h0 and
    packing) but with log-decays per key channel, g [.., H, dk] =
    max(-softplus(N(0, 1)), -5): each step's log-decay in (-5, 0), the range
    the walk-through quotes for a KDA model's gates."""
    d = chunk_inputs(B, H, T, dk, dv, dtype="bf16", seed=seed, h0=h0,
                     lengths=lengths, length_range=length_range)
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    shape = tuple(d["q"].shape)
    g = np.maximum(-_softplus(_normal(rng, shape)), np.float32(-5.0))
    d["g"] = torch.from_numpy(g.astype(np.float32))
    return d


def grad_inputs(d, *, seed=0, dhT=True):
    """Upstream gradients for a backward call on the forward inputs ``d``:
    dout bf16 shaped like v ~ N(0, 1), and dhT fp32 [N, H, dk, dv] ~ 0.1 N(0,
    1) (None with ``dhT=False``)."""
    rng = np.random.Generator(np.random.PCG64(seed + 104729))
    v = d["v"]
    dout = torch.from_numpy(_normal(rng, tuple(v.shape))).to(torch.bfloat16)
    N = (d["cu_seqlens"].numel() - 1) if d.get("cu_seqlens") is not None else v.shape[0]
    H, dk, dv = v.shape[2], d["q"].shape[-1], v.shape[-1]
    g = None
    if dhT:
        g = torch.from_numpy((0.1 * _normal(rng, (N, H, dk, dv))).astype(np.float32))
    return dout, g
