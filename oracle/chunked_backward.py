"""The gradients of the chunk form, chunk by chunk, in fp64 (oracle; TEST
INFRASTRUCTURE ONLY, see ``oracle/__init__.py``).

The pages keep the state only at chunk boundaries and recompute inside a
chunk for the gradient (illustrated DeltaNet walk-through: cost table and
memory paragraphs; "GPU parallelisation of Gated DeltaNet", m.lqnn.cn: chunk
form and block recompute). They print no gradient formulas, so this module
writes out the adjoint of each step of the chunk form (decay before the
prediction, scalar gate) as derived here; tests/test_oracle_chunk_backward_pins.py
pins it to ``oracle.backward`` (itself pinned to finite differences) at
several chunk sizes. It is the algebra a chunked backward evaluates; the GPU
is never compared with it.

One chunk of L tokens with entry state S (d_v x d_k), local cumulative gate
G_r = g_1 + ... + g_r, E = e^G, gamma = e^{G_L}, D_rs = e^{G_r - G_s}:
    A = strict_lower(diag(beta) (K K^T) (.) D),   T = (I + A)^{-1}
    K_b = diag(beta E) K,  V_b = diag(beta) V,  W = T K_b,  U0 = T V_b
    U = U0 - W S^T,  P = (Q K^T) (.) D (.) M_incl,  K_bar = diag(e^{G_L - G}) K
    O = diag(E) Q S^T + P U,   S' = gamma S + U^T K_bar.
Given dO and dS' (the gradient arriving at the chunk's exit state):
    dU = P^T dO + K_bar dS'^T,    dP = (dO U^T) (.) M_incl
    dS = gamma dS' + dO^T diag(E) Q - dU^T W          (to the previous chunk)
    dQ = diag(E) dO S + (dP (.) D) K
    dK = (dP (.) D)^T Q + diag(e^{G_L - G}) U dS' + diag(beta E) T^T dW
         + B K + B^T K,   dW = -dU S,  B = diag(beta) (dA (.) D)
    dT = dW K_b^T + dU V_b^T,   dA = strict_lower(-T^T dT T^T)
    dV = diag(beta) T^T dU
    dbeta_r = E_r k_r . (T^T dW)_r + v_r . (T^T dU)_r + sum_s dA_rs D_rs k_r . k_s
    dG_r = beta_r E_r k_r . (T^T dW)_r + E_r q_r . (dO S)_r
           + sum_s (dA (.) A)_rs - sum_s (dA (.) A)_sr
           + sum_s (dP (.) P)_rs - sum_s (dP (.) P)_sr
           - e^{G_L - G_r} k_r . (U dS')_r
    dG_L += sum_r e^{G_L - G_r} k_r . (U dS')_r + gamma sum(dS' (.) S)
    dg_t = sum over r >= t of dG_r (the chunk-local prefix sum's adjoint).
Every exponent is a difference G_r - G_s with r >= s (or G_L - G_r), so
nothing overflows however strong the decay.
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


def _chunk_forward(Q, K, V, g, b, S):
    """The chunk form's intermediates for entry state S (d_v x d_k)."""
    L = Q.shape[0]
    G = np.cumsum(g)
    D = np.exp(np.tril(G[:, None] - G[None, :]))  # upper part unused (masked)
    E = np.exp(G)
    ebar = np.exp(G[-1] - G)
    A = np.tril(b[:, None] * (K @ K.T) * D, -1)
    T = np.linalg.inv(np.eye(L) + A)
    Kb = (b * E)[:, None] * K
    Vb = b[:, None] * V
    W = T @ Kb
    U = T @ Vb - W @ S.T
    P = np.tril((Q @ K.T) * D)
    S_next = E[-1] * S + U.T @ (ebar[:, None] * K)
    return dict(G=G, D=D, E=E, ebar=ebar, A=A, T=T, Kb=Kb, Vb=Vb, W=W, U=U,
                P=P), S_next


def _chunk_adjoint(Q, K, V, b, S, c, dO, dSx):
    """The chunk's input gradients and the gradient of its entry state."""
    G, D, E, ebar, A, T = c["G"], c["D"], c["E"], c["ebar"], c["A"], c["T"]
    Kb, Vb, W, U, P = c["Kb"], c["Vb"], c["W"], c["U"], c["P"]
    gam = E[-1]
    Kbar = ebar[:, None] * K
    dU = P.T @ dO + Kbar @ dSx.T
    dP = np.tril(dO @ U.T)
    dS = gam * dSx + dO.T @ (E[:, None] * Q) - dU.T @ W
    dOS = dO @ S
    dKbar = U @ dSx
    dW = -dU @ S
    dKb = T.T @ dW
    dVb = T.T @ dU
    dT = dW @ Kb.T + dU @ Vb.T
    dA = np.tril(-T.T @ dT @ T.T, -1)
    Bm = b[:, None] * dA * D
    dQ = E[:, None] * dOS + (dP * D) @ K
    dK = ((dP * D).T @ Q + ebar[:, None] * dKbar + (b * E)[:, None] * dKb
          + Bm @ K + Bm.T @ K)
    dV = b[:, None] * dVb
    kdkb = np.sum(K * dKb, axis=1)
    db = E * kdkb + np.sum(V * dVb, axis=1) + np.sum(dA * (K @ K.T) * D, axis=1)
    kbar_term = ebar * np.sum(K * dKbar, axis=1)
    dG = (b * E * kdkb + E * np.sum(Q * dOS, axis=1)
          + np.sum(dA * A, axis=1) - np.sum(dA * A, axis=0)
          + np.sum(dP * P, axis=1) - np.sum(dP * P, axis=0) - kbar_term)
    dG[-1] += kbar_term.sum() + gam * np.sum(dSx * S)
    dg = np.cumsum(dG[::-1])[::-1]
    return dQ, dK, dV, dg, db, dS


def chunk_backward(q, k, v, g, beta, h0, dout, dhT=None, cu_seqlens=None,
                   C=64):
    """Gradients of L = sum(dout * out) + sum(dhT * hT) for the scalar-gate
    forward (decay before the prediction), by chunks of C tokens: a forward
    pass keeping each chunk's entry state, then the chunks in reverse through
    the adjoint above. Shapes and result as ``oracle.backward.backward``."""
    q, k, v, g, beta, h0, dout, dhT = map(
        _f64, (q, k, v, g, beta, h0, dout, dhT))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    fl = lambda x: x.reshape((B * T,) + x.shape[2:])
    qf, kf, vf, gf, bf, of = map(fl, (q, k, v, g, beta, dout))
    if cu_seqlens is not None:
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        seqs = [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]
    else:
        seqs = [(n * T, (n + 1) * T) for n in range(B)]
    out = {"dq": np.zeros_like(qf), "dk": np.zeros_like(kf),
           "dv": np.zeros_like(vf), "dg": np.zeros_like(gf),
           "dbeta": np.zeros_like(bf)}
    dh0 = np.zeros((len(seqs), H, dk, dv))
    for n, (bos, eos) in enumerate(seqs):
        chunks = [(t, min(t + C, eos)) for t in range(bos, eos, C)]
        for h in range(H):
            S = np.zeros((dv, dk)) if h0 is None else h0[n, h].T.copy()
            kept = []
            for t0, t1 in chunks:
                c, S_next = _chunk_forward(qf[t0:t1, h], kf[t0:t1, h],
                                           vf[t0:t1, h], gf[t0:t1, h],
                                           bf[t0:t1, h], S)
                kept.append((S, c))
                S = S_next
            dS = np.zeros((dv, dk)) if dhT is None else dhT[n, h].T.copy()
            for (t0, t1), (S_in, c) in zip(reversed(chunks), reversed(kept)):
                dQ, dK, dV, dg, db, dS = _chunk_adjoint(
                    qf[t0:t1, h], kf[t0:t1, h], vf[t0:t1, h], bf[t0:t1, h],
                    S_in, c, of[t0:t1, h], dS)
                out["dq"][t0:t1, h] = dQ
                out["dk"][t0:t1, h] = dK
                out["dv"][t0:t1, h] = dV
                out["dg"][t0:t1, h] = dg
                out["dbeta"][t0:t1, h] = db
            dh0[n, h] = dS.T
    res = {name: x.reshape((B, T) + x.shape[1:]) for name, x in out.items()}
    res["dh0"] = dh0
    return res
