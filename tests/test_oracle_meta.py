"""Pins of the oracle's metadata builder: hand-derived arrays and properties."""
import numpy as np
import pytest

from oracle import forkattn as orc
from tests.golden_io import load_meta_cases

CASES = load_meta_cases()
SCALARS = ("R", "Nq", "T_cap", "tile", "desc")


@pytest.mark.parametrize("name", sorted(CASES))
def test_meta_matches_hand_derived(name):
    c = CASES[name]
    R, Nq, T_cap, tile = int(c["R"][0]), int(c["Nq"][0]), int(c["T_cap"][0]), int(c["tile"][0])
    m = orc.meta_ref(c["desc"], R, Nq, T_cap, tile)
    for key, want in c.items():
        if key in SCALARS:
            continue
        got = np.atleast_1d(m[key])
        assert got.tolist() == want.tolist(), key


def _random_desc(rng, R, Nq_max=6):
    P = rng.integers(0, 40, size=R)
    n = rng.integers(0, Nq_max, size=R)
    ql = rng.integers(1, 20, size=int(n.sum()))
    pl = np.array([rng.integers(0, p + 1) if rng.random() < 0.3 else 0 for p in P])
    ck = np.array([rng.integers(pl[j], P[j] + 1) if rng.random() < 0.3 else -1 for j in range(R)])
    return np.concatenate([P, n, ql, pl, ck]).astype(np.int32), P, n, ql, pl, ck


@pytest.mark.parametrize("seed", range(20))
def test_meta_properties(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 7))
    desc, P, n, ql, pl, ck = _random_desc(rng, R)
    Nq = int(n.sum())
    T = int((P - pl).sum() + ql.sum())
    T_cap = T + int(rng.integers(0, 9))
    tile = int(rng.choice([4, 8, 16]))
    m = orc.meta_ref(desc, R, Nq, T_cap, tile)
    assert int(m["T"]) == T
    # every non-pad token belongs to exactly one segment, in stream order
    cover = np.zeros(T_cap, dtype=int)
    for s in range(R + Nq):
        st, L = m["seg_start"][s], m["seg_len"][s]
        cover[st:st + L] += 1
        assert (m["tok_req"][st:st + L] == m["seg_req"][s]).all()
        assert (m["tok_branch"][st:st + L] == m["seg_branch"][s]).all()
        assert (m["tok_pos"][st:st + L] == m["seg_pos0"][s] + np.arange(L)).all()
    assert (cover[:T] == 1).all() and (cover[T:] == 0).all()
    assert (m["tok_req"][T:] == -1).all() and (m["tok_pos"][T:] == -1).all()
    # question positions continue from P; trunk positions start at prefix_len
    for j in range(R):
        assert m["seg_pos0"][j] == pl[j]
        for qi in range(m["req_first_q"][j], m["req_first_q"][j] + n[j]):
            assert m["seg_pos0"][R + qi] == P[j]
            assert m["seg_trunk_start"][R + qi] == m["seg_start"][j]
            assert m["q_last"][qi] == m["seg_start"][R + qi] + m["seg_len"][R + qi] - 1
    # the work list tiles every segment exactly once
    cov2 = np.zeros(T_cap, dtype=int)
    for s, o in zip(m["work_seg"], m["work_off"]):
        L = m["seg_len"][s]
        assert 0 <= o < L and o % tile == 0
        st = m["seg_start"][s]
        cov2[st + o:st + min(o + tile, L)] += 1
    assert (cov2[:T] == 1).all()


def test_visibility_rule_examples():
    # rainbus "方法步骤详情" step 2: same request, trunk or own branch, t_y <= t_x, window.
    assert orc.visible(0, 2, 70, 0, 0, 10)  # question sees its trunk
    assert orc.visible(0, 2, 70, 0, 2, 70)  # and itself
    assert not orc.visible(0, 2, 70, 0, 1, 64)  # not a sibling
    assert not orc.visible(0, 2, 70, 1, 0, 3)  # not another request
    assert not orc.visible(0, 0, 5, 0, 0, 6)  # not the future
    assert not orc.visible(0, 0, 5, 0, 1, 5)  # a trunk token never sees a question
    assert orc.visible(0, 0, 600, 0, 0, 89, window=512)
    assert not orc.visible(0, 0, 600, 0, 0, 88, window=512)
