"""Pins of the oracle's Gated DeltaNet: literal matrix form, closed forms,
library conv, resume == scratch (Proposition 3.1), chunk form."""
import numpy as np
import pytest

from oracle import forkattn as orc
from tests.chunkform import gdn_chunked
from tree_forked_hybrid_gb300 import workloads as wl


def _inputs(rng, L, H, d, K=4):
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, H, d))
    v = rng.standard_normal((L, H, d))
    a = 1.0 / (1.0 + np.exp(-rng.normal(2.0, 0.5, size=(L, H))))
    e = 1.0 / (1.0 + np.exp(-rng.normal(0.0, 1.0, size=(L, H))))
    w = rng.uniform(-0.5, 0.5, size=(3, H, d, K))
    return q, k, v, a, e, w


def test_causal_conv_matches_numpy_convolve():
    rng = np.random.default_rng(0)
    L, C, K = 23, 5, 4
    x = rng.standard_normal((L, C))
    w = rng.standard_normal((C, K))
    got = orc.causal_conv(x, w, dtype=np.float64)
    for c in range(C):
        # y_t = sum_i w[i] x[t-K+1+i]  ==  full convolution with the reversed kernel
        want = np.convolve(x[:, c], w[c, ::-1])[:L]
        np.testing.assert_allclose(got[:, c], want, rtol=1e-12, atol=1e-12)
    hist = rng.standard_normal((K - 1, C))
    got_h = orc.causal_conv(x, w, hist, dtype=np.float64)
    full = orc.causal_conv(np.concatenate([hist, x]), w, dtype=np.float64)[K - 1:]
    np.testing.assert_allclose(got_h, full, rtol=1e-12, atol=1e-12)


def test_literal_matrix_form():
    """S_t = a S_{t-1} (I - e k k^T) + e v k^T with explicit d x d matrices."""
    rng = np.random.default_rng(1)
    L, H, d = 19, 2, 6
    q, k, v, a, e, w = _inputs(rng, L, H, d)
    o, S, _, _ = orc.gdn_sequence(q, k, v, a, e, w, dtype=np.float64)
    # independent inputs: numpy convolve, SiLU, L2 norm written out here
    def prep(x, s):
        y = np.zeros_like(x)
        for h in range(H):
            for c in range(d):
                y[:, h, c] = np.convolve(x[:, h, c], w[s, h, c, ::-1])[:L]
        return y / (1.0 + np.exp(-y))
    qh, kh, vh = prep(q, 0), prep(k, 1), prep(v, 2)
    qh = qh / np.sqrt((qh ** 2).sum(-1, keepdims=True) + 1e-6)
    kh = kh / np.sqrt((kh ** 2).sum(-1, keepdims=True) + 1e-6)
    for h in range(H):
        Sm = np.zeros((d, d))
        for t in range(L):
            kt = kh[t, h][:, None]
            Sm = a[t, h] * Sm @ (np.eye(d) - e[t, h] * kt @ kt.T) + e[t, h] * vh[t, h][:, None] @ kt.T
            np.testing.assert_allclose(o[t, h], Sm @ qh[t, h], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(S[h], Sm, rtol=1e-10, atol=1e-12)


def test_eta_zero_gives_zero():
    rng = np.random.default_rng(2)
    q, k, v, a, e, w = _inputs(rng, 11, 2, 8)
    o, S, _, _ = orc.gdn_sequence(q, k, v, a, np.zeros_like(e), w, dtype=np.float64)
    assert np.abs(o).max() == 0.0 and np.abs(S).max() == 0.0


def test_delta_rule_recall():
    """alpha = eta = 1: S_t k_t = v_t exactly, so querying with q_t = k_t returns v_t."""
    rng = np.random.default_rng(3)
    L, H, d = 13, 2, 8
    q, k, v, a, e, w = _inputs(rng, L, H, d)
    w[0] = w[1]  # q and k share conv weights and raw inputs -> identical normalised vectors
    o, _, _, _ = orc.gdn_sequence(k, k, v, np.ones_like(a), np.ones_like(e), w, dtype=np.float64)
    vh = orc.gdn_inputs(k, k, v, w, dtype=np.float64)[2]
    kh = orc.gdn_inputs(k, k, v, w, dtype=np.float64)[1]
    nrm = (kh ** 2).sum(-1)  # = |k|^2 = 1 - eps/(|x|^2+eps): exactly 1 up to the 1e-6 guard
    np.testing.assert_allclose(o, vh * 1.0, rtol=0, atol=1e-5 * np.abs(vh).max())
    assert np.all(np.abs(nrm - 1.0) < 1e-4)


def test_orthonormal_keys_sum_of_outer_products():
    """alpha = eta = 1 and orthonormal keys e_t: S = sum_t v_t e_t^T (the erase term vanishes)."""
    L, H, d = 5, 1, 8
    rng = np.random.default_rng(4)
    w = np.zeros((3, H, d, 4))
    w[..., 3] = 1.0  # identity tap: conv output = current raw input
    k = np.zeros((L, H, d))
    for t in range(L):
        k[t, 0, t] = 30.0  # silu(30 e_t) = silu(30) e_t, normalised -> e_t
    v = rng.standard_normal((L, H, d))
    q = rng.standard_normal((L, H, d))
    _, S, _, _ = orc.gdn_sequence(q, k, v, np.ones((L, H)), np.ones((L, H)), w, dtype=np.float64)
    vh = v / (1.0 + np.exp(-v))
    want = np.zeros((d, d))
    for t in range(L):
        want[:, t] = vh[t, 0]
    np.testing.assert_allclose(S[0], want, atol=1e-6)


def test_single_token_closed_form():
    rng = np.random.default_rng(5)
    q, k, v, a, e, w = _inputs(rng, 1, 3, 8)
    o, S, _, _ = orc.gdn_sequence(q, k, v, a, e, w, dtype=np.float64)
    qh, kh, vh = orc.gdn_inputs(q, k, v, w, dtype=np.float64)
    for h in range(3):
        np.testing.assert_allclose(S[h], e[0, h] * np.outer(vh[0, h], kh[0, h]), rtol=1e-12)
        np.testing.assert_allclose(o[0, h], e[0, h] * vh[0, h] * (kh[0, h] @ qh[0, h]), rtol=1e-12)


def test_resume_from_saved_state_equals_scratch():
    """Proposition 3.1 for the recurrence: trunk once, then each branch resumes
    from (S_P, conv window) == running s ⊕ q_i from scratch."""
    rng = np.random.default_rng(6)
    P, H, d = 29, 2, 8
    q, k, v, a, e, w = _inputs(rng, P + 9, H, d)
    o_t, S_P, _, win = orc.gdn_sequence(q[:P], k[:P], v[:P], a[:P], e[:P], w, dtype=np.float64)
    o_full, S_full, states, _ = orc.gdn_sequence(q, k, v, a, e, w, dtype=np.float64, state_at=[P])
    np.testing.assert_allclose(states[P], S_P, rtol=1e-12, atol=1e-14)
    o_b, S_b, _, _ = orc.gdn_sequence(q[P:], k[P:], v[P:], a[P:], e[P:], w, dtype=np.float64,
                                      S0=S_P, hist=win)
    np.testing.assert_allclose(o_b, o_full[P:], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_b, S_full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o_t, o_full[:P], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L,C,S0", [(64, 64, False), (100, 16, False), (37, 8, True), (5, 8, True)])
def test_chunk_form_equals_token_loop(L, C, S0):
    rng = np.random.default_rng(7)
    H, d = 2, 8
    q, k, v, a, e, w = _inputs(rng, L, H, d)
    S_init = rng.standard_normal((H, d, d)) * 0.3 if S0 else None
    at = [0, 1, L // 3, L - 1, L]
    o, S, st, _ = orc.gdn_sequence(q, k, v, a, e, w, dtype=np.float64, S0=S_init, state_at=at)
    qh, kh, vh = orc.gdn_inputs(q, k, v, w, dtype=np.float64)
    oc, Sc, stc = gdn_chunked(qh, kh, vh, a, e, C, S0=S_init, state_at=at)
    np.testing.assert_allclose(oc, o, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(Sc, S, rtol=1e-10, atol=1e-10)
    for t in at:
        np.testing.assert_allclose(stc[t], st[t], rtol=1e-10, atol=1e-10)


def test_round_level_resume_matches_scratch():
    """A round whose trunk starts from a checkpoint prefix: the oracle runs
    the full trunk from scratch; its state at the prefix equals a separate
    run over the prefix rows only."""
    a = wl.AttnShape("attn", 2, 1, 8, 0, 0.0)
    g = wl.GdnShape("gdn", 2, 8, 8, 4, 8)
    rnd = wl.custom_round([12], [2], [3, 4], attn_shapes=(a,), gdn_shape=g, T_cap=16, seed=3,
                          prefix_len=[7])
    lay = {"gdn": {k: rnd.f32("gdn", k).astype(np.float64) for k in ("q", "k", "v", "alpha", "eta")}}
    lay["gdn"]["conv_w"] = rnd.layers["gdn"]["conv_w"].astype(np.float64)
    pre = {"gdn": {k: rnd.prefix_f32("gdn", k).astype(np.float64) for k in ("q", "k", "v", "alpha", "eta")}}
    view = orc.RoundView(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, lay, pre)
    out = orc.run_gdn(view, "gdn", dtype=np.float64)
    # literal: trunk = prefix rows + 5 stream rows
    full = [np.concatenate([pre["gdn"][f][:7], lay["gdn"][f][:5]]) for f in ("q", "k", "v", "alpha", "eta")]
    o, S, _, _ = orc.gdn_sequence(*full, lay["gdn"]["conv_w"], dtype=np.float64)
    np.testing.assert_allclose(out["o"][:5], o[7:], rtol=1e-12)
    np.testing.assert_allclose(out["S_P"][0], S, rtol=1e-12)
    # and from the state after the 7 prefix rows + their conv window
    o7, S7, _, w7 = orc.gdn_sequence(*[x[:7] for x in full], lay["gdn"]["conv_w"], dtype=np.float64)
    o_r, S_r, _, _ = orc.gdn_sequence(*[x[7:] for x in full], lay["gdn"]["conv_w"], dtype=np.float64,
                                      S0=S7, hist=w7)
    np.testing.assert_allclose(S_r, S, rtol=1e-12, atol=1e-13)


def test_fp32_tracks_fp64():
    rng = np.random.default_rng(8)
    q, k, v, a, e, w = _inputs(rng, 200, 2, 32)
    o64, S64, _, _ = orc.gdn_sequence(q, k, v, a, e, w, dtype=np.float64)
    o32, S32, _, _ = orc.gdn_sequence(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32),
                                      a.astype(np.float32), e.astype(np.float32), w.astype(np.float32))
    assert np.abs(o32 - o64).max() < 1e-5
    assert np.linalg.norm(S32 - S64) / np.linalg.norm(S64) < 1e-5
