"""Independent formulations used to pin the oracle (test helpers, numpy fp64).

* ``closed_form_states`` -- the unrolled product form of the KDA recurrence
  ("Kimi K3: architecture and SGLang Day-0 Support", KDA math box: S_t is the sum
  over s <= t of [prod_{u=s+1..t} (I - beta_u k_u k_u^T) Diag(alpha_u)] beta_s k_s v_s^T),
  plus the initial-state term (prod_{u<=t} M_u) S_0 that the same unrolling gives
  for a nonzero S_0.  Every M_u is an explicit dk x dk matrix.
* ``chunked`` -- a second, chunk-parallel formulation (UT/WY form with a unit
  lower-triangular solve and decay-rescaled keys), derived from the recurrence
  by induction over the tokens of a chunk.  It is the algebra the CUDA kernels
  use, checked here in fp64 against the sequential oracle.
* ``chunked_backward`` -- the reverse-mode derivative of that chunk algebra (the
  backward kernels' algebra), checked in fp64 against the oracle's sequential
  backward.
"""
from __future__ import annotations

import numpy as np


def token_transition(k, g, beta):
    """M = (I - beta k k^T) Diag(exp(g)) for one token (k, g: [dk])."""
    k = np.asarray(k, np.float64)
    dk = k.shape[0]
    return (np.eye(dk) - beta * np.outer(k, k)) @ np.diag(np.exp(np.asarray(g, np.float64)))


def closed_form_states(k, v, g, beta, S0):
    """States S_1..S_T of one head by the unrolled product form.  k, g: [T, dk]; v: [T, dv]; beta: [T]."""
    T, dk = k.shape
    Ms = [token_transition(k[t], g[t], beta[t]) for t in range(T)]
    out = []
    for t in range(T):
        P = np.eye(dk)
        for u in range(t + 1):
            P = Ms[u] @ P
        S = P @ S0
        for s in range(t + 1):
            Q = np.eye(dk)
            for u in range(s + 1, t + 1):
                Q = Ms[u] @ Q
            S = S + Q @ (beta[s] * np.outer(k[s], v[s]))
        out.append(S)
    return np.stack(out)


def chunked(q, k, v, g, beta, S0, C=64, L=16, dtype=np.float64):
    """Chunk-parallel KDA for one head.  q, k, g: [T, dk]; v: [T, dv]; beta: [T]; S0: [dk, dv].

    Per chunk of up to C tokens with entry state S0 and in-chunk cumulative log-decay
    G_t = sum_{u<=t} g_u:
      A_ts = beta_t sum_j k_t[j] k_s[j] exp(G_t[j] - G_s[j])   (s < t)
      P_ts = sum_j q_t[j] k_s[j] exp(G_t[j] - G_s[j])          (s <= t)
      (I + A) U = diag(beta) (V - (K o exp(G)) S0)               (unit lower-triangular solve)
      O  = (Q o exp(G)) S0 + P U
      S' = Diag(exp(G_C)) S0 + (K o exp(G_C - G))^T U
    The pair decays exp(G_t - G_s) are split at a per-column-block reference
    r = last token of s's L-token block: exp(G_t - G_r) * exp(G_r - G_s), so no
    factor exceeds exp(L * |g|max) (finite in fp32 for |g| <= 5, L = 16).
    Returns (O [T, dv], S_T [dk, dv]) computed in `dtype`.
    """
    f = lambda x: np.asarray(x, dtype)
    q, k, v, g, beta, S = f(q), f(k), f(v), f(g), f(beta), f(S0).copy()
    T = q.shape[0]
    O = np.zeros((T, v.shape[1]), dtype)
    for c0 in range(0, T, C):
        c1 = min(c0 + C, T)
        n = c1 - c0
        qc, kc, vc, gc, bc = q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1]
        G = np.cumsum(gc, axis=0, dtype=dtype)
        A = np.zeros((n, n), dtype)
        P = np.zeros((n, n), dtype)
        for b0 in range(0, n, L):
            b1 = min(b0 + L, n)
            Gr = G[b1 - 1]                                  # reference: last token of the column block
            kminus = kc[b0:b1] * np.exp(Gr - G[b0:b1])      # <= 1
            kplus = kc[b0:] * np.exp(G[b0:] - Gr)           # rows t >= b0 (up to exp(L*5) inside the block)
            qplus = qc[b0:] * np.exp(G[b0:] - Gr)
            A[b0:, b0:b1] = kplus @ kminus.T
            P[b0:, b0:b1] = qplus @ kminus.T
        A = np.tril(A, -1) * bc[:, None]
        P = np.tril(P, 0)
        gam = np.exp(G)
        rhs = bc[:, None] * (vc - (kc * gam) @ S)
        U = np.zeros_like(rhs)
        for t in range(n):                                  # forward substitution, unit diagonal
            U[t] = rhs[t] - A[t, :t] @ U[:t]
        O[c0:c1] = (qc * gam) @ S + P @ U
        khat = kc * np.exp(G[-1] - G)
        S = np.exp(G[-1])[:, None] * S + khat.T @ U
    return O, S


def chunked_backward(q, k, v, g, beta, S0, dO, dST, C=64):
    """Chunk-parallel gradients of L = sum_t <dO_t, o_t> + <dST, S_T> for one head (fp64).

    The reverse-mode derivative of ``chunked``'s algebra, with the pair decays taken pairwise,
    E_ts = exp(G_t - G_s) <= 1 for s <= t.  Per chunk with entry state S and
    K+ = K o e^G, Q+ = Q o e^G, K^ = K o e^(G_C - G), a_ts = sum_j k_t k_s E_ts (s < t), A = diag(beta) a,
    P_ts = sum_j q_t k_s E_ts (s <= t), T = (I + A)^-1, W = T diag(beta) K+, U = T diag(beta) V - W S:
      dU = P^T dO + K^ dS'                      dS  = Q+^T dO + Diag(e^G_C) dS' - W^T dU
      dP = tril(dO U^T)   dQ+ = dO S^T   dK^ = U dS'^T   dW = -dU S^T   d(e^G_C) = rowsum(dS' o S)
      dT = dW (diag(beta) K+)^T + dU (diag(beta) V)^T      dA = -T^T dT T^T (strictly lower part)
    then the chain rule through beta, the e^G factors and the pair decays, and dg = the in-chunk reverse
    cumulative sum of dG.  The entry states run forward over the chunks and dS backward.
    Returns dict dq, dk, dv, dg [T, .], dbeta [T], ds0 [dk, dv].
    """
    f = lambda x: np.asarray(x, np.float64)
    q, k, v, g, beta, dO = f(q), f(k), f(v), f(g), f(beta), f(dO)
    T, dk = q.shape
    dv = v.shape[1]
    starts = list(range(0, T, C))
    # forward: entry state of every chunk
    S = f(S0).copy()
    entry, parts = [], []
    for c0 in starts:
        c1 = min(c0 + C, T)
        n = c1 - c0
        kc, vc, qc, bc = k[c0:c1], v[c0:c1], q[c0:c1], beta[c0:c1]
        G = np.cumsum(g[c0:c1], axis=0)
        E = np.exp(G[:, None, :] - G[None, :, :])        # [t, s, j]; used only where s <= t
        low = np.tril(np.ones((n, n)), -1)
        a = np.einsum("tj,sj,tsj->ts", kc, kc, E) * low
        P = np.einsum("tj,sj,tsj->ts", qc, kc, E) * np.tril(np.ones((n, n)))
        A = bc[:, None] * a
        Tm = np.linalg.inv(np.eye(n) + A)
        kp, qp, kh = kc * np.exp(G), qc * np.exp(G), kc * np.exp(G[-1] - G)
        BK, BV = bc[:, None] * kp, bc[:, None] * vc
        W = Tm @ BK
        U = Tm @ BV - W @ S
        entry.append(S)
        parts.append(dict(G=G, E=E, a=a, P=P, Tm=Tm, kp=kp, qp=qp, kh=kh, BK=BK, BV=BV, W=W, U=U))
        S = np.exp(G[-1])[:, None] * S + kh.T @ U
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), dg=np.zeros_like(g),
               dbeta=np.zeros_like(beta))
    dS = f(dST).copy()
    for ci in range(len(starts) - 1, -1, -1):
        c0 = starts[ci]
        c1 = min(c0 + C, T)
        n = c1 - c0
        z = parts[ci]
        S = entry[ci]
        kc, vc, qc, bc, dOc = k[c0:c1], v[c0:c1], q[c0:c1], beta[c0:c1], dO[c0:c1]
        dU = z["P"].T @ dOc + z["kh"] @ dS
        dP = np.tril(dOc @ z["U"].T)
        dqp = dOc @ S.T
        dkh = z["U"] @ dS.T
        dgamC = (dS * S).sum(axis=1)
        dW = -dU @ S.T
        dT = dW @ z["BK"].T + dU @ z["BV"].T
        dBK = z["Tm"].T @ dW
        dBV = z["Tm"].T @ dU
        dA = np.tril(-z["Tm"].T @ dT @ z["Tm"].T, -1)
        dS_entry = z["qp"].T @ dOc + np.exp(z["G"][-1])[:, None] * dS - z["W"].T @ dU
        dbeta = (dA * z["a"]).sum(axis=1) + (dBK * z["kp"]).sum(axis=1) + (dBV * vc).sum(axis=1)
        da = bc[:, None] * dA
        dkp = bc[:, None] * dBK
        dvc = bc[:, None] * dBV
        eG = np.exp(z["G"])
        dqc = dqp * eG
        dkc = dkp * eG + dkh * np.exp(z["G"][-1] - z["G"])
        dG = dqp * z["qp"] + dkp * z["kp"] - dkh * z["kh"]
        dGC = (dkh * z["kh"]).sum(axis=0) + dgamC * np.exp(z["G"][-1])
        E = z["E"]
        # a_ts = sum_j k_t k_s E_ts (s < t)
        X = da[:, :, None] * kc[:, None, :] * kc[None, :, :] * E
        dkc += np.einsum("ts,sj,tsj->tj", da, kc, E) + np.einsum("ts,tj,tsj->sj", da, kc, E)
        dG += X.sum(axis=1) - X.sum(axis=0)
        # P_ts = sum_j q_t k_s E_ts (s <= t)
        Y = dP[:, :, None] * qc[:, None, :] * kc[None, :, :] * E
        dqc += np.einsum("ts,sj,tsj->tj", dP, kc, E)
        dkc += np.einsum("ts,tj,tsj->sj", dP, qc, E)
        dG += Y.sum(axis=1) - Y.sum(axis=0)
        dG[-1] += dGC
        out["dq"][c0:c1] = dqc
        out["dk"][c0:c1] = dkc
        out["dv"][c0:c1] = dvc
        out["dbeta"][c0:c1] = dbeta
        out["dg"][c0:c1] = np.cumsum(dG[::-1], axis=0)[::-1]
        dS = dS_entry
    out["ds0"] = dS
    return out


def segment_reverse_fragments(q, k, v, g, beta, dO, C=64, seg_chunks=2):
    """The backward's state-gradient carry in segment form, for one head (fp64).

    Per chunk, dS_in = M_c^T dS_out + b_c with M_c^T = Diag(e^{G_C}) - W^T K^ (the transpose of the
    forward chunk transition S' = (Diag(e^{G_C}) - K^^T W) S + K^^T U~) and b_c = (Q+ - P W)^T dO, which
    depends on the chunk's inputs and dO only, not on the forward state.  A segment of `seg_chunks`
    chunks composes to dS_in = N dS_out + b~, found by running [b | X] backwards through its chunks from
    [0 | I].  Returns the list of (N, b~) per segment, in token order.
    """
    f = lambda x: np.asarray(x, np.float64)
    q, k, v, g, beta, dO = f(q), f(k), f(v), f(g), f(beta), f(dO)
    T, dk = q.shape
    chunk_terms = []
    for c0 in range(0, T, C):
        c1 = min(c0 + C, T)
        n = c1 - c0
        kc, qc, bc = k[c0:c1], q[c0:c1], beta[c0:c1]
        G = np.cumsum(g[c0:c1], axis=0)
        E = np.exp(G[:, None, :] - G[None, :, :])
        A = bc[:, None] * np.einsum("tj,sj,tsj->ts", kc, kc, E) * np.tril(np.ones((n, n)), -1)
        P = np.einsum("tj,sj,tsj->ts", qc, kc, E) * np.tril(np.ones((n, n)))
        W = np.linalg.inv(np.eye(n) + A) @ (bc[:, None] * kc * np.exp(G))
        kh = kc * np.exp(G[-1] - G)
        Mt = np.diag(np.exp(G[-1])) - W.T @ kh
        b = (qc * np.exp(G) - P @ W).T @ dO[c0:c1]
        chunk_terms.append((Mt, b))
    frags = []
    for s0 in range(0, len(chunk_terms), seg_chunks):
        X, y = np.eye(dk), np.zeros_like(chunk_terms[0][1])
        for Mt, b in reversed(chunk_terms[s0:s0 + seg_chunks]):
            X, y = Mt @ X, Mt @ y + b
        frags.append((X, y))
    return frags


def reverse_scan(frags, dST):
    """Exit gradients of every segment from the last one's (dST): exit_{p-1} = N_p exit_p + b~_p.
    Returns [exit_0, ..., exit_{P-1}, entry_0] (entry_0 = dL/dS_0)."""
    exits = [None] * len(frags)
    d = np.asarray(dST, np.float64)
    for p in range(len(frags) - 1, -1, -1):
        exits[p] = d
        N, b = frags[p]
        d = N @ d + b
    return exits + [d]
