"""Pins of the oracle's options readout and of question independence."""
import numpy as np
import pytest
from scipy.special import softmax

from oracle import forkattn as orc
from tree_forked_hybrid_gb300 import workloads as wl


def test_readout_matches_scipy_softmax():
    rng = np.random.default_rng(0)
    nopt = np.array([2, 5, 1, 3])
    off = np.concatenate([[0], np.cumsum(nopt)])
    h = rng.standard_normal((4, 16))
    w = rng.standard_normal((int(nopt.sum()), 16))
    p = orc.readout(h, w, off, np.float64)
    for i in range(4):
        np.testing.assert_allclose(p[off[i]:off[i + 1]], softmax(w[off[i]:off[i + 1]] @ h[i]), rtol=1e-13)
    assert p[off[2]] == 1.0  # |O| = 1  =>  p = 1
    for i in range(4):
        assert abs(p[off[i]:off[i + 1]].sum() - 1.0) < 1e-14


def test_equal_logits_uniform_and_shift_invariance():
    w = np.ones((4, 8))
    p = orc.readout(np.ones((1, 8)), w, np.array([0, 4]), np.float64)
    np.testing.assert_allclose(p, 0.25, rtol=1e-15)
    rng = np.random.default_rng(1)
    h = rng.standard_normal((1, 8))
    w = rng.standard_normal((3, 8))
    c = rng.standard_normal(8)
    p1 = orc.readout(h, w, np.array([0, 3]), np.float64)
    # adding the same vector to every option row shifts every logit equally
    p2 = orc.readout(h, w + c[None, :], np.array([0, 3]), np.float64)
    np.testing.assert_allclose(p1, p2, rtol=1e-12)


def test_total_variation_definition():
    p = np.array([0.5, 0.5, 1.0])
    r = np.array([0.25, 0.75, 1.0])
    np.testing.assert_allclose(orc.total_variation(p, r, np.array([0, 2, 3])), [0.25, 0.0])


def _view(rnd, dtype=np.float64):
    lay = {}
    for name in rnd.layers:
        lay[name] = {k: (rnd.f32(name, k) if k != "conv_w" else rnd.layers[name][k]).astype(dtype)
                     for k in rnd.layers[name]}
    return orc.RoundView(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, lay)


def test_sibling_and_request_independence():
    """A question's oracle output does not depend on its siblings or on other requests."""
    a = wl.AttnShape("attn", 2, 1, 8, 0, 10000.0)
    g = wl.GdnShape("gdn", 2, 8, 8, 4, 8)
    r1 = wl.custom_round([10, 6], [3, 1], [4, 5, 3, 2], attn_shapes=(a,), gdn_shape=g, T_cap=40, seed=9)
    r2 = wl.custom_round([10, 6], [3, 1], [4, 5, 3, 2], attn_shapes=(a,), gdn_shape=g, T_cap=40, seed=9)
    m = orc.meta_ref(r1.desc(), 2, 4, 40, 8)
    # perturb question 1 (sibling of question 0) and all of request 1
    for name in r2.layers:
        for f in r2.layers[name]:
            if f == "conv_w":
                continue
            arr = r2.layers[name][f]
            for s in (2 + 1, 1, 2 + 3):
                st, L = m["seg_start"][s], m["seg_len"][s]
                arr[st:st + L] = arr[st:st + L][::-1].copy() if arr.dtype == np.uint16 else arr[st:st + L] * 0.5
    v1, v2 = _view(r1), _view(r2)
    o1 = orc.run_attention(v1, "attn", window=0, rope_theta=10000.0, dtype=np.float64)
    o2 = orc.run_attention(v2, "attn", window=0, rope_theta=10000.0, dtype=np.float64)
    g1 = orc.run_gdn(v1, "gdn", dtype=np.float64)
    g2 = orc.run_gdn(v2, "gdn", dtype=np.float64)
    for s in (0, 2 + 0, 2 + 2):  # trunk 0, question 0, question 2 of request 0
        st, L = m["seg_start"][s], m["seg_len"][s]
        assert np.array_equal(o1[st:st + L], o2[st:st + L])
        assert np.array_equal(g1["o"][st:st + L], g2["o"][st:st + L])
    assert np.array_equal(g1["S_P"][0], g2["S_P"][0])


def test_round_fp32_close_to_fp64():
    rnd = wl.make_round(0)
    v32, v64 = _view(rnd, np.float32), _view(rnd, np.float64)
    a32 = orc.run_attention(v32, "attn", window=0, rope_theta=0.0)
    a64 = orc.run_attention(v64, "attn", window=0, rope_theta=0.0, dtype=np.float64)
    assert np.abs(a32 - a64).max() < 1e-5
    g32 = orc.run_gdn(v32, "gdn")
    g64 = orc.run_gdn(v64, "gdn", dtype=np.float64)
    assert np.abs(g32["o"] - g64["o"]).max() < 1e-5
    p32 = orc.run_readout(v32, g32["o"], rnd.w_opt_f32(), rnd.opt_off)
    p64 = orc.run_readout(v64, g64["o"], rnd.w_opt_f32().astype(np.float64), rnd.opt_off, np.float64)
    assert np.abs(p32 - p64).max() < 1e-6
