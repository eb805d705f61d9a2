"""Pins of the oracle's small helpers: the L2 normalisation of q and k and the
conv window a checkpoint or trunk end keeps (rainbus summary "前置知识", "方法步骤详情")."""
import numpy as np

from oracle import forkattn as orc


def test_l2norm_closed_forms():
    x = np.array([[3.0, 4.0]], dtype=np.float64)
    assert np.allclose(orc.l2norm(x, eps=0.0), [[0.6, 0.8]], atol=1e-15)
    # the 1e-6 guard: |y| = |x| / sqrt(|x|^2 + 1e-6)
    y = orc.l2norm(np.array([[1e-3, 0.0]]), eps=1e-6)
    assert np.allclose(y, [[1e-3 / np.sqrt(1e-6 + 1e-6), 0.0]], atol=1e-15)
    assert np.array_equal(orc.l2norm(np.zeros((2, 5))), np.zeros((2, 5)))
    r = np.random.default_rng(0).standard_normal((7, 3, 16))
    n = orc.l2norm(r, eps=0.0)
    assert np.allclose(np.linalg.norm(n, axis=-1), 1.0, atol=1e-13)
    assert np.allclose(orc.l2norm(5.0 * r, eps=0.0), n, atol=1e-13)


def test_conv_window_holds_the_raw_rows_before_m():
    rng = np.random.default_rng(1)
    L, H, d, K = 9, 2, 8, 4
    q, k, v = (rng.standard_normal((L, H, d)).astype(np.float32) for _ in range(3))
    for m in (0, 1, 2, 3, 6, 9):
        w = orc.conv_window_at(q, k, v, m, K)
        for i in range(K - 1):
            t = m - (K - 1) + i
            for s, x in enumerate((q, k, v)):
                want = x[t] if t >= 0 else np.zeros((H, d), np.float32)
                assert np.array_equal(w[i, s], want), (m, i, s)
    # the window after a whole sequence is the one the token loop returns
    a = rng.uniform(0.5, 1.0, size=(L, H)).astype(np.float32)
    e = rng.uniform(0.0, 1.0, size=(L, H)).astype(np.float32)
    cw = rng.uniform(-0.5, 0.5, size=(3, H, d, K)).astype(np.float32)
    _, _, _, win = orc.gdn_sequence(q, k, v, a, e, cw)
    assert np.array_equal(win, orc.conv_window_at(q, k, v, L, K))
