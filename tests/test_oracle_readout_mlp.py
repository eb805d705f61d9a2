"""Pins of the oracle's selective-readout block: the final pointwise block run
on the questions' last-token rows only (onedev summary "어떻게 쓰나"), read
as a pre-norm SwiGLU MLP with a residual, a final RMSNorm and eq. (1)."""
import math

import numpy as np

from oracle import forkattn as orc


def test_round_to_bf16_bit_patterns():
    u = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0x3F817FFF, 0x3F7FFFFF, 0x7F7F8000, 0xBF80C000,
                  0x00008000], dtype=np.uint32)
    want = np.array([0x3F800000, 0x3F800000, 0x3F820000, 0x3F810000, 0x3F800000, 0x7F800000, 0xBF810000,
                     0x00000000], dtype=np.uint32)
    got = orc.round_to_bf16(u.view(np.float32)).view(np.uint32)
    assert np.array_equal(got, want)  # ties to even, carries into the exponent, overflow to inf
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    r = orc.round_to_bf16(x)
    assert np.array_equal(orc.round_to_bf16(r), r)
    assert np.all(r.view(np.uint32) & 0xFFFF == 0)
    assert np.all(np.abs(r - x) <= np.abs(x) * 2.0 ** -8)


def test_rms_norm_closed_forms():
    g = np.array([0.5, 2.0, -1.0, 1.5], dtype=np.float64)
    for c in (3.0, -0.25):
        y = orc.rms_norm(np.full((1, 4), c), g, eps=0.0, dtype=np.float64)
        assert np.allclose(y[0], np.sign(c) * g, atol=1e-15)
    x = np.random.default_rng(1).standard_normal((5, 64))
    one = np.ones(64)
    y = orc.rms_norm(x, one, eps=0.0, dtype=np.float64)
    assert np.allclose((y * y).mean(axis=1), 1.0, atol=1e-13)
    assert np.allclose(orc.rms_norm(7.5 * x, one, eps=0.0, dtype=np.float64), y, atol=1e-13)


def test_mlp_block_worked_example():
    # D = 2, F = 1, g1 = 1: worked by hand with scalar steps
    h = np.array([[3.0, 4.0]], dtype=np.float32)
    wg = np.array([[1.0, 0.0]], dtype=np.float32)
    wu = np.array([[0.0, 1.0]], dtype=np.float32)
    wd = np.array([[1.0], [2.0]], dtype=np.float32)
    rms = math.sqrt((9.0 + 16.0) / 2.0 + 1e-6)
    n0, n1 = 3.0 / rms, 4.0 / rms            # 0.84852..., 1.13137...
    n0b, n1b = 0.84765625, 1.1328125         # nearest bfloat16 values
    assert abs(n0 - n0b) < 2 ** -9 and abs(n1 - n1b) < 2 ** -8
    gate, up = n0b, n1b
    a = gate / (1.0 + math.exp(-gate)) * up  # 0.6722...
    ab = 0.671875                            # nearest bfloat16
    assert abs(a - ab) < 2 ** -9
    y = orc.mlp_block(h, np.ones(2), wg, wu, wd, dtype=np.float64)
    assert np.allclose(y, [[3.0 + ab, 4.0 + 2.0 * ab]], atol=1e-12)


def test_mlp_block_reductions_and_row_independence():
    rng = np.random.default_rng(2)
    T, D, F = 40, 32, 48
    h = rng.standard_normal((T, D)).astype(np.float32)
    g1 = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wg = (rng.standard_normal((F, D)) / math.sqrt(D)).astype(np.float32)
    wu = (rng.standard_normal((F, D)) / math.sqrt(D)).astype(np.float32)
    wd = (rng.standard_normal((D, F)) / math.sqrt(F)).astype(np.float32)
    assert np.array_equal(orc.mlp_block(h, g1, wg, wu, np.zeros_like(wd)), h)
    assert np.array_equal(orc.mlp_block(h, g1, np.zeros_like(wg), wu, wd), h)
    # selective readout changes no output: the block on every row, then the chosen rows,
    # equals the block on the chosen rows alone
    rows = np.array([3, 17, 18, 39, 0])
    full = orc.mlp_block(h, g1, wg, wu, wd, dtype=np.float64)[rows]
    sel = orc.mlp_block(h[rows], g1, wg, wu, wd, dtype=np.float64)
    assert np.array_equal(full, sel)
    assert not np.allclose(full, h[rows])


def test_readout_mlp_reduces_to_eq1():
    rng = np.random.default_rng(3)
    Nq, D, F = 6, 32, 64
    h = rng.standard_normal((Nq, D)).astype(np.float32)
    n_opt = np.array([2, 3, 1, 4, 2, 5])
    off = np.concatenate([[0], np.cumsum(n_opt)]).astype(np.int32)
    w = (0.2 * rng.standard_normal((off[-1], D))).astype(np.float32)
    g = np.ones(D, dtype=np.float32)
    wg = rng.standard_normal((F, D)).astype(np.float32)
    p = orc.readout_mlp(h, g, wg, wg, np.zeros((D, F), np.float32), g, w, off)
    assert np.allclose(p, orc.readout(orc.rms_norm(h, g), w, off), atol=1e-7)
    for i in range(Nq):
        assert abs(p[off[i]:off[i + 1]].sum() - 1.0) < 1e-6
