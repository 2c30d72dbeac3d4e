"""The steps either side of the recurrence, in fp64 (oracle; TEST
INFRASTRUCTURE ONLY, see ``oracle/__init__.py``).

Illustrated DeltaNet page, architecture table and the L2 Norm / RMSNorm
paragraphs: q and k are L2-normalised per (token, head) over their features;
beta comes from a sigmoid; the read-out o_t = S_t q_t is RMS-normalised per
(token, head) over its d_v features and scaled by a learned per-feature
vector w; its GDN section (the Qwen GDN module) follows the normalisation
with a sigmoid output gate. The log-gate g = -softplus(a) is the gate
parameterisation of the workloads (alpha = exp(-softplus(x))).

Readings (the pages leave these open): a zero q or k vector stays zero (its
length is 0, nothing to divide); the RMSNorm epsilon is added to the mean of
squares; the output gate multiplies after the weight, out = RMSNorm(o) * w *
sigmoid(z), z an input of the same shape as o; the normalisation is applied
when a weight is given (a unit weight is passed as ones) and the gate when
gate logits are given, so either step can be left out.
"""
from __future__ import annotations

import numpy as np

from . import G1, forward


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def l2_normalize(x):
    """x / ||x|| along the last axis (each token and head on its own)."""
    x = _f64(x)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return np.divide(x, n, out=np.zeros_like(x), where=n > 0)


def sigmoid(x):
    x = _f64(x)
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def softplus(x):
    """log(1 + e^x), written so that it neither overflows nor cancels."""
    x = _f64(x)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def rms_norm(x, weight=None, eps=0.0):
    """x / sqrt(mean(x^2) + eps) along the last axis, times weight."""
    x = _f64(x)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    y = x / r
    return y if weight is None else y * _f64(weight)


def prologue(q_raw, k_raw, a, b):
    """(q, k, g, beta) of the recurrence from the raw per-head inputs."""
    return l2_normalize(q_raw), l2_normalize(k_raw), -softplus(a), sigmoid(b)


def epilogue(o, weight=None, gate=None, eps=1e-6):
    """RMSNorm(o) * weight when a weight is given, then * sigmoid(gate) when
    gate logits are given."""
    y = _f64(o) if weight is None else rms_norm(o, weight, eps)
    return y if gate is None else y * sigmoid(gate)


def fused_forward(q_raw, k_raw, v, a, b, h0=None, cu_seqlens=None,
                  weight=None, gate=None, eps=1e-6, variant=G1):
    """The recurrence with the steps either side: returns (out, hT)."""
    q, k, g, beta = prologue(q_raw, k_raw, a, b)
    o, hT = forward(q, k, v, g, beta, h0, cu_seqlens=cu_seqlens,
                    variant=variant)
    return epilogue(o, weight, gate, eps), hT
