"""Numpy fp64 restatements of the Gated DeltaNet map in the pages' other forms.

TEST INFRASTRUCTURE ONLY (see the package docstring). These functions pin the
token-loop oracle from independent derivations; the GPU is never compared
with them. Nothing here is blocked, fused or reordered beyond what each cited
derivation states.

Orientation: the C oracle and the public state layout store Z = S^T
(d_k x d_v). Functions below say which orientation they use; all public
inputs/outputs use the storage layout of ``oracle.forward``:
q, k [B, T, H, dk], v [B, T, H, dv], g/beta [B, T, H], h0/hT [N, H, dk, dv].
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

G1, G0 = 1, 0


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _sequences(q, cu_seqlens):
    """Yield (n, token slice into the flattened [B*T] axis)."""
    B, T = q.shape[:2]
    if cu_seqlens is None:
        for n in range(B):
            yield n, slice(n * T, (n + 1) * T)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        for n in range(len(cu) - 1):
            yield n, slice(int(cu[n]), int(cu[n + 1]))


def _flat(x):
    B, T = x.shape[:2]
    return x.reshape((B * T,) + x.shape[2:])


# ---------------------------------------------------------------------------
# 1. Per-token affine maps and their composition
#    ("GPU parallelisation of Gated DeltaNet", m.lqnn.cn, sections 2.2-2.3 and
#    3.3-3.4). Storage orientation: Z_t = A_t Z_{t-1} + B_t, Z is d_k x d_v.
# ---------------------------------------------------------------------------

def token_affine(k_t, v_t, g_t, beta_t, variant=G1):
    """(A_t, B_t) of one token.

    variant 0 is the page's form, A_t = alpha I - beta k k^T. variant 1 decays
    before the prediction, so A_t = alpha (I - beta k k^T). B_t = beta k v^T in
    both (u_t k_t^T written in the storage orientation).
    """
    dk = k_t.shape[0]
    alpha = np.exp(g_t)
    kk = np.outer(k_t, k_t)
    if variant == G1:
        A = alpha * (np.eye(dk) - beta_t * kk)
    else:
        A = alpha * np.eye(dk) - beta_t * kk
    Bm = beta_t * np.outer(k_t, v_t)
    return A, Bm


def compose(later, earlier):
    """compose((A2, B2), (A1, B1)) = (A2 A1, A2 B1 + B2): apply earlier first."""
    A2, B2 = later
    A1, B1 = earlier
    return A2 @ A1, A2 @ B1 + B2


def affine_forward(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk=64,
                   variant=G1):
    """Chunk transforms by composition, a sequential scan over chunks for the
    chunk-start states (S_start = A_prefix S_0 + B_prefix), then each chunk's
    outputs recomputed from its start state with the per-token maps; the read
    o_t = Z_t^T q_t happens after the token's write."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    qf, kf, vf, gf, bf = map(_flat, (q, k, v, g, beta))
    out = np.zeros((B * T, H, dv))
    seqs = list(_sequences(q, cu_seqlens))
    hT = np.zeros((len(seqs), H, dk, dv))
    for n, sl in seqs:
        for h in range(H):
            Z0 = np.zeros((dk, dv)) if h0 is None else h0[n, h].copy()
            idx = np.arange(sl.start, sl.stop)
            chunks = [idx[i:i + chunk] for i in range(0, len(idx), chunk)]
            # per-chunk transform (A_chunk, B_chunk)
            transforms = []
            for c in chunks:
                acc = (np.eye(dk), np.zeros((dk, dv)))
                for t in c:
                    acc = compose(token_affine(kf[t, h], vf[t, h], gf[t, h],
                                               bf[t, h], variant), acc)
                transforms.append(acc)
            # sequential inclusive scan over chunks
            prefix = []
            acc = None
            for tr in transforms:
                acc = tr if acc is None else compose(tr, acc)
                prefix.append(acc)
            starts = [Z0] + [Ap @ Z0 + Bp for Ap, Bp in prefix[:-1]]
            for c, Zs in zip(chunks, starts):
                Z = Zs
                for t in c:
                    A, Bm = token_affine(kf[t, h], vf[t, h], gf[t, h],
                                         bf[t, h], variant)
                    Z = A @ Z + Bm
                    out[t, h] = Z.T @ qf[t, h]
            if prefix:
                Ap, Bp = prefix[-1]
                hT[n, h] = Ap @ Z0 + Bp
            else:
                hT[n, h] = Z0
    return out.reshape(B, T, H, dv), hT


# ---------------------------------------------------------------------------
# 2. Gate prefixes and the decay matrix (illustrated DeltaNet page, GLA gate
#    prefix products and the Lambda / Gamma / gamma table), scalar gate.
# ---------------------------------------------------------------------------

def local_cumsum(g_chunk):
    """G_r = sum_{l <= r} g_l inside one chunk (log of the prefix product b_r)."""
    return np.cumsum(g_chunk)


def decay_matrix(g_chunk, variant=G1):
    """D_rj = b_r / b_j = exp(G_r - G_j) for j <= r, 0 above the diagonal.

    For variant 0 the prediction of token r uses the state before alpha_r, so
    the matrix used inside the UT system is exp(G_{r-1} - G_j); this helper
    returns the read (output) matrix, which is the same in both variants."""
    G = local_cumsum(g_chunk)
    L = len(G)
    D = np.exp(G[:, None] - G[None, :])
    return np.where(np.tril(np.ones((L, L), dtype=bool)), D, 0.0)


def gated_scores(q_chunk, k_chunk, g_chunk):
    """(Q K^T) (.) D (.) lower-including-diagonal: weight of write j in read r."""
    return (q_chunk @ k_chunk.T) * decay_matrix(g_chunk)


# ---------------------------------------------------------------------------
# 3. WY / UT chunk form (illustrated DeltaNet page: pseudo-values U, WY
#    representation P_n = I - W^T K, UT transform T = (I - A)^{-1} with
#    A_tj = -beta_t k_t^T k_j, chunkwise state passing and output), gated with
#    the scalar Lambda/Gamma/gamma prefixes. Math orientation S = Z^T
#    (d_v x d_k).
# ---------------------------------------------------------------------------

def wy_factors(k_c, v_c, g_c, beta_c, variant=G1):
    """W (L x dk), U0 (L x dv), Kbar (L x dk), gamma for one chunk.

    A = strict_lower(diag(beta) (K K^T) (.) D'), T = (I + A)^{-1},
    W = T diag(beta (.) e^{G'}) K, U0 = T diag(beta) V, Kbar = diag(e^{G_L - G}) K,
    where D'/G' use G_r (variant 1) or G_{r-1} (variant 0)."""
    L = k_c.shape[0]
    G = local_cumsum(g_c)
    Gp = G if variant == G1 else G - g_c  # exponent base of the prediction
    Dp = np.exp(Gp[:, None] - G[None, :])
    A = np.tril(beta_c[:, None] * (k_c @ k_c.T) * Dp, k=-1)
    IA = np.eye(L) + A
    W = solve_triangular(IA, (beta_c * np.exp(Gp))[:, None] * k_c, lower=True,
                         unit_diagonal=True)
    U0 = solve_triangular(IA, beta_c[:, None] * v_c, lower=True,
                          unit_diagonal=True)
    Kbar = np.exp(G[-1] - G)[:, None] * k_c
    return W, U0, Kbar, float(np.exp(G[-1])), IA


def wy_chunk_step(S, q_c, k_c, v_c, g_c, beta_c, variant=G1):
    """One chunk from entry state S (d_v x d_k): returns (O_chunk, S_exit).

    U = U0 - W S^T;  O = diag(e^G) Q S^T + ((Q K^T) (.) D (.) M) U;
    S' = gamma S + U^T Kbar."""
    W, U0, Kbar, gamma, _ = wy_factors(k_c, v_c, g_c, beta_c, variant)
    G = local_cumsum(g_c)
    U = U0 - W @ S.T
    O = np.exp(G)[:, None] * (q_c @ S.T) + gated_scores(q_c, k_c, g_c) @ U
    S_next = gamma * S + U.T @ Kbar
    return O, S_next


def chunk_transform_phi_psi(k_c, v_c, g_c, beta_c, variant=G1):
    """S' = S Phi + Psi with Phi = gamma I - W^T Kbar (d_k x d_k) and
    Psi = U0^T Kbar (d_v x d_k): the chunk as an affine map of its entry."""
    W, U0, Kbar, gamma, _ = wy_factors(k_c, v_c, g_c, beta_c, variant)
    dk = k_c.shape[1]
    return gamma * np.eye(dk) - W.T @ Kbar, U0.T @ Kbar


def wy_forward(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk=64,
               variant=G1):
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    qf, kf, vf, gf, bf = map(_flat, (q, k, v, g, beta))
    out = np.zeros((B * T, H, dv))
    seqs = list(_sequences(q, cu_seqlens))
    hT = np.zeros((len(seqs), H, dk, dv))
    for n, sl in seqs:
        for h in range(H):
            S = np.zeros((dv, dk)) if h0 is None else h0[n, h].T.copy()
            for c0 in range(sl.start, sl.stop, chunk):
                c = slice(c0, min(c0 + chunk, sl.stop))
                O, S = wy_chunk_step(S, qf[c, h], kf[c, h], vf[c, h], gf[c, h],
                                     bf[c, h], variant)
                out[c, h] = O
            hT[n, h] = S.T
    return out.reshape(B, T, H, dv), hT


# ---------------------------------------------------------------------------
# 4. Sequence parallelism by incremental state and correction ("How to
#    Implement Sequence Parallelism in DeltaNet", papercache.org, sections
#    A2 CP=2 / CP=4): each sub-sequence p > 0 runs from Delta S = 0 and
#    M = I with Delta S <- Delta S Phi_i + Psi_i, M <- M Phi_i; the true
#    state is Delta S_[i] + S_start M_[i]; the starts form a serial chain.
#    The gated Phi_i = gamma_i I - W_i^T Kbar_i reduces to I - W^T K at
#    alpha = 1, the page's form.
#    combine="scan": the starts by an inclusive prefix scan instead of the
#    chain ("GPU parallelisation of Gated DeltaNet", section 3.4: the
#    chunk-level scan of affine maps, Hillis-Steele order). Sub-sequence p
#    maps its start to its end, S -> S M_p + dS_p; applying map a, then map
#    b, is S -> S (M_a M_b) + (dS_a M_b + dS_b), an associative product, so
#    after the rounds with offsets 1, 2, 4, ... entry p holds the map of
#    sub-sequences 0 .. p.
# ---------------------------------------------------------------------------

def scan_maps(maps):
    """Inclusive Hillis-Steele scan of [(M, dS), ...] under 'apply the
    earlier map, then the later one'."""
    pref = list(maps)
    d = 1
    while d < len(pref):
        nxt = list(pref)
        for p in range(d, len(pref)):
            Ma, dSa = pref[p - d]
            Mb, dSb = pref[p]
            nxt[p] = (Ma @ Mb, dSa @ Mb + dSb)
        pref = nxt
        d *= 2
    return pref


def sp_forward(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk=64, parts=2,
               variant=G1, combine="chain"):
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    qf, kf, vf, gf, bf = map(_flat, (q, k, v, g, beta))
    out = np.zeros((B * T, H, dv))
    seqs = list(_sequences(q, cu_seqlens))
    hT = np.zeros((len(seqs), H, dk, dv))
    for n, sl in seqs:
        starts = list(range(sl.start, sl.stop, chunk))
        nchunks = len(starts)
        per = -(-nchunks // parts) if nchunks else 0
        groups = [starts[p * per:(p + 1) * per] for p in range(parts)]
        groups = [gr for gr in groups if gr]
        for h in range(H):
            S0 = np.zeros((dv, dk)) if h0 is None else h0[n, h].T.copy()
            # phase 1 (independent per sub-sequence): Delta S and M per chunk
            records = []
            for gi, gr in enumerate(groups):
                dS = np.zeros((dv, dk))
                M = np.eye(dk)
                rec = []
                for c0 in gr:
                    c = slice(c0, min(c0 + chunk, sl.stop))
                    rec.append((c, dS.copy(), M.copy()))
                    Phi, Psi = chunk_transform_phi_psi(kf[c, h], vf[c, h],
                                                       gf[c, h], bf[c, h],
                                                       variant)
                    dS = dS @ Phi + Psi
                    M = M @ Phi
                records.append((rec, dS, M))
            # phase 2: true start states, by the serial chain over
            # sub-sequences or by the prefix scan of their maps
            if combine == "scan":
                pref = scan_maps([(M_end, dS_end) for _, dS_end, M_end in records])
                starts = [S0] + [S0 @ M + dS for M, dS in pref]
            else:
                starts = [S0]
                for _, dS_end, M_end in records:
                    starts.append(dS_end + starts[-1] @ M_end)
            # phase 3 (independent per chunk): correct, then output
            for (rec, _, _), S_start in zip(records, starts):
                for c, dS_i, M_i in rec:
                    S_i = dS_i + S_start @ M_i
                    O, _ = wy_chunk_step(S_i, qf[c, h], kf[c, h], vf[c, h],
                                         gf[c, h], bf[c, h], variant)
                    out[c, h] = O
            hT[n, h] = starts[-1].T
    return out.reshape(B, T, H, dv), hT


# ---------------------------------------------------------------------------
# 5. Householder-product sum (illustrated DeltaNet page, "generalized
#    Householder" paragraphs), gated: S_t = S_0 H_1...H_t
#    + sum_i beta_i v_i k_i^T H_{i+1}...H_t with H_t = alpha_t (I - beta_t
#    k_t k_t^T) (variant 1) or alpha_t I - beta_t k_t k_t^T (variant 0).
#    Dense products; tiny T only.
# ---------------------------------------------------------------------------

def householder_bruteforce(q, k, v, g, beta, S0, variant=G1):
    """One (sequence, head): q, k [T, dk], v [T, dv], g/beta [T], S0 (d_v x d_k).
    Returns (O [T, dv], S_T (d_v x d_k)) with every state formed from scratch."""
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    T, dk = k.shape
    Hs = []
    for t in range(T):
        a = np.exp(g[t])
        kk = np.outer(k[t], k[t])
        Hs.append(a * (np.eye(dk) - beta[t] * kk) if variant == G1
                  else a * np.eye(dk) - beta[t] * kk)

    def prod(i, t):  # H_i ... H_t (1-based inclusive), empty -> I
        P = np.eye(dk)
        for j in range(i, t + 1):
            P = P @ Hs[j - 1]
        return P

    O = np.zeros((T, v.shape[1]))
    S = S0
    for t in range(1, T + 1):
        S = S0 @ prod(1, t)
        for i in range(1, t + 1):
            S = S + beta[i - 1] * np.outer(v[i - 1], k[i - 1]) @ prod(i + 1, t)
        O[t - 1] = S @ q[t - 1]
    return O, S
