"""Pins of the oracle's attention: library routine, brute-force fork mask, closed forms."""
import math

import numpy as np
import pytest
import torch

from oracle import forkattn as orc
from tree_forked_hybrid_gb300 import workloads as wl


def _sdpa(q, k, v, mask):
    """torch's CPU scaled_dot_product_attention in float64 (library routine)."""
    G = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)
    vt = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask))
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("window", [0, 7])
def test_isolated_sequence_matches_torch_sdpa(window):
    rng = np.random.default_rng(1)
    L, Hq, Hkv, d = 37, 4, 2, 16
    q = rng.standard_normal((L, Hq, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    x = np.arange(L)
    mask = x[None, :] <= x[:, None]
    if window:
        mask &= (x[:, None] - x[None, :]) < window
    got = orc.attention_sequence(q, k, v, window=window, dtype=np.float64)
    want = _sdpa(q, k, v, mask)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_rope_is_complex_rotation():
    rng = np.random.default_rng(2)
    L, H, d = 9, 3, 8
    x = rng.standard_normal((L, H, d))
    pos = rng.integers(0, 5000, size=L)
    got = orc.rope(x, pos, 10000.0, np.float64)
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = 10000.0 ** (-np.arange(half) * 2.0 / d)
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    np.testing.assert_allclose(got[..., :half], zr.real, atol=1e-12)
    np.testing.assert_allclose(got[..., half:], zr.imag, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(got, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)


def test_rope_depends_on_relative_position_only():
    rng = np.random.default_rng(3)
    d = 64
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    dots = []
    for shift in (0, 17, 4000):
        qr = orc.rope(q, np.array([100 + shift]), 10000.0, np.float64)
        kr = orc.rope(k, np.array([40 + shift]), 10000.0, np.float64)
        dots.append(float((qr * kr).sum()))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


def test_single_key_and_uniform_scores():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((6, 1, 8))
    q = np.zeros((6, 2, 8))
    k = rng.standard_normal((6, 1, 8))
    o = orc.attention_sequence(q, k, v, dtype=np.float64)
    # row 0 sees one key: o = v_0; with q = 0 every score ties: o_x = mean of v_0..v_x
    for x in range(6):
        np.testing.assert_allclose(o[x, 0], v[:x + 1, 0].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(o[x, 1], v[:x + 1, 0].mean(axis=0), atol=1e-14)
    ow = orc.attention_sequence(q, k, v, window=2, dtype=np.float64)
    for x in range(1, 6):
        np.testing.assert_allclose(ow[x, 0], v[x - 1:x + 1, 0].mean(axis=0), atol=1e-14)


def _small_round(seed, window, rope_theta, prefix=False):
    a = wl.AttnShape("attn", 4, 2, 16, window, rope_theta)
    g = wl.GdnShape("gdn", 2, 8, 8, 4, 8)
    if prefix:
        return wl.custom_round([9, 7], [2, 1], [3, 5, 4], attn_shapes=(a,), gdn_shape=g, T_cap=40,
                               seed=seed, prefix_len=[5, 0])
    return wl.custom_round([9, 7, 0], [2, 1, 2], [3, 5, 4, 1, 2], attn_shapes=(a,), gdn_shape=g,
                           T_cap=40, seed=seed)


@pytest.mark.parametrize("window,rope_theta,prefix", [(0, 0.0, False), (0, 10000.0, False),
                                                      (4, 10000.0, False), (0, 10000.0, True),
                                                      (3, 10000.0, True)])
def test_fork_structure_equals_isolated_runs(window, rope_theta, prefix):
    """Proposition 3.1 for attention: one flat stream with the (j, c, t) mask
    (brute force, every pair) equals running every trunk and s ⊕ q_i alone."""
    rnd = _small_round(5, window, rope_theta, prefix)
    view = orc.RoundView(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap,
                         {"attn": {k: rnd.f32("attn", k).astype(np.float64) for k in "qkv"}},
                         None if rnd.prefix is None else
                         {"attn": {k: rnd.prefix_f32("attn", k).astype(np.float64) for k in "qkv"}})
    iso = orc.run_attention(view, "attn", window=window, rope_theta=rope_theta, dtype=np.float64)
    m = view.meta
    T = int(m["T"])
    # keys: the prefix rows (outside the stream) followed by the stream rows
    kj, kc, kt, kk, kv = [], [], [], [], []
    for j in range(rnd.R):
        pl = int(rnd.prefix_len[j])
        off = int(m["req_prefix_off"][j])
        for u in range(pl):
            kj.append(j), kc.append(0), kt.append(u)
            kk.append(view.prefix["attn"]["k"][off + u]), kv.append(view.prefix["attn"]["v"][off + u])
    for y in range(T):
        kj.append(m["tok_req"][y]), kc.append(m["tok_branch"][y]), kt.append(m["tok_pos"][y])
        kk.append(view.layers["attn"]["k"][y]), kv.append(view.layers["attn"]["v"][y])
    kj, kc, kt = map(np.array, (kj, kc, kt))
    kk, kv = np.array(kk), np.array(kv)
    q = view.layers["attn"]["q"][:T]
    if rope_theta:
        q = orc.rope(q, m["tok_pos"][:T], rope_theta, np.float64)
        kk = orc.rope(kk, kt, rope_theta, np.float64)
    mask = np.zeros((T, kj.shape[0]), dtype=bool)
    for x in range(T):
        for y in range(kj.shape[0]):
            mask[x, y] = orc.visible(m["tok_req"][x], m["tok_branch"][x], m["tok_pos"][x],
                                     kj[y], kc[y], kt[y], window)
    flat = _sdpa(q, kk, kv, mask)
    np.testing.assert_allclose(flat, iso[:T], rtol=1e-11, atol=1e-11)
