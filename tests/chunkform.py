"""Chunk form of the gated delta rule, float64 numpy (design check, not the oracle).

The CUDA GDN kernels evaluate the recurrence chunk by chunk.  With the chunk's
start state S0 (d_v x d_k), inclusive cumulative log-decay G_t = sum_{s<=t}
log alpha_s and Gamma_ts = exp(G_t - G_s):
    u_t = eta_t (v_t - alpha_t S_{t-1} k_t)            (so S_t = alpha_t S_{t-1} + u_t k_t^T)
    (I + A) U = diag(eta) V - diag(eta e^G) K S0^T,   A_ts = eta_t Gamma_ts k_t.k_s  (s < t)
    O   = diag(e^G) Q S0^T + (tril_incl(Gamma) * Q K^T) U
    S_r = e^{G_{r-1}} S0 + U[:r]^T diag(Gamma_{r-1, :r}) K[:r]   (state after r tokens)
This is the algebra of the gated delta rule of the rainbus summary ("前置知识"),
rearranged as the chunked / masked-triangular-solve form that the DFlash-TfM
summary describes for GDN ("GDN을 위한 롤백 없는 트리 검증").  The test checks it
against the oracle's token loop.
"""
import numpy as np


def gdn_chunked(qh, kh, vh, alpha, eta, C, S0=None, state_at=()):
    L, H, dk = kh.shape
    dv = vh.shape[2]
    S = np.zeros((H, dv, dk)) if S0 is None else S0.copy()
    o = np.zeros((L, H, dv))
    states = {}
    want = set(state_at)
    if 0 in want:
        states[0] = S.copy()
    for c0 in range(0, L, C):
        n = min(C, L - c0)
        Snext = np.zeros_like(S)
        for h in range(H):
            Q, K, V = qh[c0:c0 + n, h], kh[c0:c0 + n, h], vh[c0:c0 + n, h]
            a, e = alpha[c0:c0 + n, h], eta[c0:c0 + n, h]
            G = np.cumsum(np.log(a))
            Gam = np.exp(G[:, None] - G[None, :])
            low = np.tril(np.ones((n, n)), -1)
            incl = np.tril(np.ones((n, n)))
            A = low * (e[:, None] * Gam * (K @ K.T))
            Tinv = np.linalg.inv(np.eye(n) + A)
            W = Tinv @ ((e * np.exp(G))[:, None] * K)
            Ut = Tinv @ (e[:, None] * V)
            U = Ut - W @ S[h].T
            o[c0:c0 + n, h] = np.exp(G)[:, None] * (Q @ S[h].T) + (incl * Gam * (Q @ K.T)) @ U
            for r in range(1, n + 1):
                if c0 + r in want:
                    st = np.exp(G[r - 1]) * S[h] + (U[:r] * np.exp(G[r - 1] - G[:r])[:, None]).T @ K[:r]
                    states.setdefault(c0 + r, np.zeros_like(S))[h] = st
            Snext[h] = np.exp(G[-1]) * S[h] + (U * Gam[-1][:, None]).T @ K
        S = Snext
    return o, S, states
