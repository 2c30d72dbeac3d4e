"""Gradients of the forward pass in fp64 (oracle; TEST INFRASTRUCTURE ONLY,
see ``oracle/__init__.py``).

The backward pass of the pages (illustrated DeltaNet walk-through, the cost
table and memory paragraphs: a chunkwise model keeps only the state at each
chunk boundary and recomputes the rest for the gradient; the lqnn.cn page,
section on the chunk form, block recompute) has a plain definition: the
derivative of the forward map. Here that derivative is written out as the
reverse sweep of the token recurrence, with every intermediate kept (no
recomputation: the oracle holds all states). For a per-channel decay (KDA,
the walk-through's hybrid-architecture section; the scalar gate is every
channel equal) one token is
    S_bar = S diag(a),  a = e^{g_t}     e = v_t - S_bar k_t,  u = beta_t e
    S_t = S_bar + u k_t^T               o_t = S_t q_t
and, given dS (the gradient arriving at S_t) and do_t, its adjoint is
    dq_t = S_t^T do_t                   dS += do_t q_t^T
    du = dS k_t,  dk_t = dS^T u - beta_t S_bar^T du
    dbeta_t = du . e,  dv_t = beta_t du
    dS_bar = dS - beta_t du k_t^T
    dg_t = colsum(dS_bar (.) S_bar)     dS_{t-1} = dS_bar diag(a).
With the other gate placement of the scalar gate (the lqnn.cn page, section
1.2: correct against the undecayed state, then decay), one token is
    e = v_t - S k_t,  u = beta_t e,  S_t = S diag(a) + u k_t^T,  o_t = S_t q_t
and its adjoint differs in the last three steps:
    dk_t = dS^T u - beta_t S^T du;  dg_t = colsum(dS (.) S diag(a));
    dS_{t-1} = dS diag(a) - beta_t du k_t^T.
The loss these gradients belong to is L = sum(dout (.) out) + sum(dhT (.)
hT); tests/test_oracle_backward_pins.py pins the sweep against central
finite differences of that loss computed with the forward oracles, against
closed forms, and against automatic differentiation of an independent
PyTorch statement of the forward map.

State layout as in ``oracle.kda``: S is d_v x d_k, h0 / hT hold S^T.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _sequences(B, T, cu_seqlens):
    if cu_seqlens is not None:
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        return [slice(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]
    return [slice(n * T, (n + 1) * T) for n in range(B)]


def kda_backward(q, k, v, g, beta, h0, dout, dhT=None, cu_seqlens=None,
                 decay_first=True):
    """Gradients of L = sum(dout * out) + sum(dhT * hT) for the per-channel
    forward (``oracle.kda.forward``; ``decay_first=False``: the placement
    that predicts with the undecayed state). q, k, g [B, T, H, dk]; v, dout
    [B, T, H, dv]; beta [B, T, H]; h0, dhT [N, H, dk, dv] or None. Returns a
    dict dq, dk, dv, dg, dbeta (shapes of the inputs) and dh0 [N, H, dk,
    dv]."""
    q, k, v, g, beta, h0, dout, dhT = map(
        _f64, (q, k, v, g, beta, h0, dout, dhT))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    flat = lambda x: x.reshape(B * T, H, -1)
    qf, kf, vf, gf, of = map(flat, (q, k, v, g, dout))
    bf = beta.reshape(B * T, H)
    seqs = _sequences(B, T, cu_seqlens)
    grads = {n: np.zeros_like(x) for n, x in
             (("dq", qf), ("dk", kf), ("dv", vf), ("dg", gf))}
    grads["dbeta"] = np.zeros_like(bf)
    dh0 = np.zeros((len(seqs), H, dk, dv))
    for n, sl in enumerate(seqs):
        for h in range(H):
            S = np.zeros((dv, dk)) if h0 is None else h0[n, h].T.copy()
            keep = []  # (state the prediction reads, e, S_t) per token
            for t in range(sl.start, sl.stop):
                a = np.exp(gf[t, h])[None, :]
                Sp = S * a if decay_first else S
                e = vf[t, h] - Sp @ kf[t, h]
                S = (Sp if decay_first else S * a) + np.outer(bf[t, h] * e, kf[t, h])
                keep.append((Sp, e, S))
            dS = np.zeros((dv, dk)) if dhT is None else dhT[n, h].T.copy()
            for i in range(len(keep) - 1, -1, -1):
                t = sl.start + i
                Sb, e, St = keep[i]
                qt, kt, b = qf[t, h], kf[t, h], bf[t, h]
                grads["dq"][t, h] = St.T @ of[t, h]
                dS = dS + np.outer(of[t, h], qt)
                u = b * e
                du = dS @ kt
                grads["dk"][t, h] = dS.T @ u - b * (Sb.T @ du)
                grads["dbeta"][t, h] = du @ e
                grads["dv"][t, h] = b * du
                a = np.exp(gf[t, h])[None, :]
                if decay_first:
                    dSb = dS - b * np.outer(du, kt)
                    grads["dg"][t, h] = (dSb * Sb).sum(axis=0)
                    dS = dSb * a
                else:
                    grads["dg"][t, h] = (dS * Sb * a).sum(axis=0)
                    dS = dS * a - b * np.outer(du, kt)
            dh0[n, h] = dS.T
    out = {n: x.reshape(B, T, H, -1) for n, x in grads.items()}
    out["dbeta"] = grads["dbeta"].reshape(B, T, H)
    out["dh0"] = dh0
    return out


def backward(q, k, v, g, beta, h0, dout, dhT=None, cu_seqlens=None,
             variant=1):
    """The same for the scalar gate (``oracle.forward``; variant 1 = G1,
    decay before the prediction, 0 = G0): g [B, T, H] is every channel's
    log-decay, so dg is the sum over channels of the per-channel one."""
    g = _f64(g)
    dk = np.asarray(_f64(q)).shape[-1]
    gk = np.repeat(g[..., None], dk, axis=-1)
    out = kda_backward(q, k, v, gk, beta, h0, dout, dhT, cu_seqlens,
                       decay_first=(variant == 1))
    out["dg"] = out["dg"].sum(axis=-1)
    return out


def fused_backward(q_raw, k_raw, v, a, b, h0, dout, dhT=None, cu_seqlens=None,
                   weight=None, gate=None, eps=1e-6):
    """Gradients of ``oracle.sublayer.fused_forward`` (the recurrence with the
    steps either side, decay before the prediction) for L = sum(dout * out)
    + sum(dhT * hT). The steps' adjoints, written out:
      out = y * sigmoid(z), y = n * w, n = o r, r = (mean(o^2) + eps)^(-1/2):
        dz = dout * y * s (1 - s);  dy = dout * s;  dw = sum over rows of dy * n;
        do = r (dn - n mean(dn * n)),  dn = dy * w
      q = q_raw / |q_raw|:  dq_raw = (dq - q (q . dq)) / |q_raw|  (k alike)
      g = -softplus(a):  da = -dg sigmoid(a);  beta = sigmoid(b):  db = dbeta beta (1 - beta).
    Returns dq, dk, dv, da, db, dh0, and dweight / dgate (None when that step
    is absent)."""
    from . import forward
    from . import sublayer as sl
    q, k, g, beta = sl.prologue(q_raw, k_raw, a, b)
    o, _ = forward(q, k, v, g, beta, h0, cu_seqlens=cu_seqlens, variant=1)
    dy = _f64(dout)
    res = {"dweight": None, "dgate": None}
    pre = o if weight is None else sl.rms_norm(o, weight, eps)
    if gate is not None:
        s = sl.sigmoid(gate)
        res["dgate"] = dy * pre * s * (1.0 - s)
        dy = dy * s
    if weight is not None:
        r = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
        n = o * r
        res["dweight"] = (dy * n).reshape(-1, o.shape[-1]).sum(axis=0)
        dn = dy * _f64(weight)
        do = r * (dn - n * np.mean(dn * n, axis=-1, keepdims=True))
    else:
        do = dy
    core = backward(q, k, v, g, beta, h0, do, dhT, cu_seqlens, variant=1)

    def unnorm(x_raw, x_hat, dx_hat):
        x_raw = _f64(x_raw)
        ln = np.sqrt(np.sum(x_raw * x_raw, axis=-1, keepdims=True))
        proj = dx_hat - x_hat * np.sum(x_hat * dx_hat, axis=-1, keepdims=True)
        return np.divide(proj, ln, out=np.zeros_like(proj), where=ln > 0)

    res["dq"] = unnorm(q_raw, q, core["dq"])
    res["dk"] = unnorm(k_raw, k, core["dk"])
    res["dv"] = core["dv"]
    res["da"] = -core["dg"] * sl.sigmoid(a)
    res["db"] = core["dbeta"] * beta * (1.0 - beta)
    res["dh0"] = core["dh0"]
    return res
