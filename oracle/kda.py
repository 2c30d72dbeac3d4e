"""KDA: the delta rule with a per-channel decay, in fp64 (oracle; TEST
INFRASTRUCTURE ONLY, see ``oracle/__init__.py``).

Illustrated DeltaNet walk-through, KDA paragraphs of its hybrid-architecture
section: one attention head produces d_k decay factors alpha_t = (alpha_{t,1},
.., alpha_{t,d_k}), one per key channel (a column of the d_v x d_k state);
the forgetting step scales column c by alpha_{t,c}, S_bar = S_{t-1}
diag(alpha_t); then the delta rule runs on the forgotten state ("decay first,
then correct"): u_t = beta_t (v_t - S_bar k_t), S_t = S_bar + u_t k_t^T; the
read is o_t = S_t q_t after the write, as for the scalar gate. With every
alpha_{t,c} equal to one alpha_t this is the scalar-gate recurrence with the
decay before the prediction.

Inputs are the log-decays g_{t,c} = log alpha_{t,c} (<= 0), per token, head
and key channel. The walk-through notes a model that keeps each step's
log-decay in (-5, 0) so that a chunked algorithm's rescalings over 16-token
sub-chunks stay in range; the definition below needs no such bound.
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


def step(S, q_t, k_t, v_t, g_t, beta_t):
    """One token on the d_v x d_k state S: returns (o_t, S_t)."""
    Sb = S * np.exp(g_t)[None, :]          # column c times alpha_{t,c}
    u = beta_t * (v_t - Sb @ k_t)          # prediction error, scaled
    S_new = Sb + np.outer(u, k_t)
    return S_new @ q_t, S_new


def forward(q, k, v, g, beta, h0=None, cu_seqlens=None):
    """q, k [B, T, H, dk]; v [B, T, H, dv]; g [B, T, H, dk] (log-decays);
    beta [B, T, H]; h0 [N, H, dk, dv] (element (i, j) = S[j][i]) or None;
    cu_seqlens (packed: B = 1, N sequences) or None. Returns (out [B, T, H,
    dv], hT [N, H, dk, dv])."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    qf, kf, vf = (x.reshape(B * T, H, -1) for x in (q, k, v))
    gf = g.reshape(B * T, H, dk)
    bf = beta.reshape(B * T, H)
    if cu_seqlens is not None:
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        seqs = [slice(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]
    else:
        seqs = [slice(n * T, (n + 1) * T) for n in range(B)]
    out = np.zeros((B * T, H, dv))
    hT = np.zeros((len(seqs), H, dk, dv))
    for n, sl in enumerate(seqs):
        for h in range(H):
            S = np.zeros((dv, dk)) if h0 is None else h0[n, h].T.copy()
            for t in range(sl.start, sl.stop):
                out[t, h], S = step(S, qf[t, h], kf[t, h], vf[t, h], gf[t, h],
                                    bf[t, h])
            hT[n, h] = S.T
    return out.reshape(B, T, H, dv), hT
