"""The algorithmic work behind the bench's roofline fractions (CPU).

The attention FLOPs count only visible (q-head, query, key) pairs.  Here the count
is checked against a brute-force pass of the oracle's visibility rule over every
(query, key) pair of small rounds: stream rows from the oracle's metadata, and the
prefix rows of resumed requests (trunk positions 0..prefix_len-1, branch 0).
"""
import numpy as np
import pytest

from oracle import forkattn as orc
from tree_forked_hybrid_gb300 import roofline as RL
from tree_forked_hybrid_gb300 import workloads as wl

A = wl.AttnShape("attn", 4, 2, 16, 0, 10000.0)
G = wl.GdnShape("gdn", 2, 16, 16, 4, 64)


def brute_pairs(rnd, window):
    m = orc.meta_ref(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, 16)
    req, br, pos = m["tok_req"][:rnd.T], m["tok_branch"][:rnd.T], m["tok_pos"][:rnd.T]
    keys = [(int(req[y]), int(br[y]), int(pos[y])) for y in range(rnd.T)]
    for j in range(rnd.R):
        keys += [(j, 0, t) for t in range(int(rnd.prefix_len[j]))]
    total = 0
    for x in range(rnd.T):
        jx, cx, tx = int(req[x]), int(br[x]), int(pos[x])
        total += sum(1 for (jy, cy, ty) in keys if orc.visible(jx, cx, tx, jy, cy, ty, window))
    return total


ROUNDS = [
    ([20, 9, 0, 14], [2, 1, 1, 2], [5, 7, 3, 11, 4, 6], None),
    ([40], [3], [1, 12, 30], None),
    ([30, 25], [2, 1], [6, 9, 4], [12, 0]),  # request 0 resumed: 12 trunk positions outside the stream
]


@pytest.mark.parametrize("case", range(len(ROUNDS)))
@pytest.mark.parametrize("window", [0, 5, 8])
def test_visible_pairs_equal_a_brute_force_count(case, window):
    P, n, ql, pl = ROUNDS[case]
    rnd = wl.custom_round(P, n, ql, attn_shapes=(A,), gdn_shape=G, T_cap=256, seed=case, prefix_len=pl)
    assert RL.visible_pairs(rnd, window) == brute_pairs(rnd, window)


def test_attention_and_layer_work_formulas():
    P, n, ql, pl = ROUNDS[2]
    rnd = wl.custom_round(P, n, ql, attn_shapes=(A,), gdn_shape=G, T_cap=256, seed=7, prefix_len=pl)
    f, b = RL.attn_work(rnd, A)
    assert f == 4 * A.d * A.Hq * brute_pairs(rnd, 0)
    # Q and O per q-head, K and V per kv head, bf16; plus the prefix K/V rows
    assert b == rnd.T * (2 * A.Hq + 2 * A.Hkv) * A.d * 2 + 12 * 2 * A.Hkv * A.d * 2
    w = RL.round_work(rnd)
    assert w["flops"] == f + w["gdn"]["flops"] + w["readout"]["flops"]
    assert w["bytes"] == b + w["gdn"]["bytes"] + w["readout"]["bytes"]
    # the slower of the two limits
    assert RL.roofline_time({"flops": 2e12, "bytes": 1e9}, 1000.0, 1000.0) == pytest.approx(2e-3)
    assert RL.roofline_time({"flops": 1e9, "bytes": 3e9}, 1000.0, 1000.0) == pytest.approx(3e-3)


FORESTS = [
    ([-1, 0, 0, 1, 1, 1, 2, 2, 3, 3, -1], [30, 12, 8, 9, 4, 33, 6, 1, 5, 17, 45]),
    ([-1, 0, 1, 2, 3, 4, 5, 6, 6, 6], [5, 3, 0, 7, 1, 2, 9, 4, 3, 6]),
    ([-1, 0, -1, 1, 2, 1, 4, 4, 0], [0, 6, 10, 3, 20, 2, 1, 8, 5]),
]


@pytest.mark.parametrize("case", range(len(FORESTS)))
@pytest.mark.parametrize("window", [0, 5, 13])
def test_forest_work_counts_the_pairs_of_every_path(case, window):
    """Visible pairs of a forest counted by brute force: each node's sequence (ancestors'
    rows, then its own) built from the tree, every query against every key of it."""
    parent, node_len = FORESTS[case]
    a = wl.AttnShape("attn", 4, 2, 16, window, 10000.0)
    t = wl.make_tree_round(parent, node_len, attn_shapes=(a,), gdn_shape=G, seed=case)
    start = t.node_start
    brute = 0
    for k in range(t.N):
        chain = [k] + t.ancestors(k)[::-1]
        rows = np.concatenate([np.arange(start[c], start[c] + node_len[c]) for c in chain[::-1]])
        n = rows.shape[0]
        for i in range(n - node_len[k], n):
            brute += sum(1 for y in range(n) if y <= i and (window == 0 or i - y < window))
    w = RL.forest_work(t)
    assert w["attn"]["attn"]["flops"] == 4 * a.d * a.Hq * brute
    T = int(np.sum(node_len))
    assert w["T"] == T and w["attn"]["attn"]["bytes"] == T * (2 * a.Hq + 2 * a.Hkv) * a.d * 2
    # states: every node writes its end state; a node with tokens before it reads its parent's
    pos0 = RL.forest_first_positions(t)
    assert pos0.tolist() == [sum(node_len[c] for c in t.ancestors(k)) for k in range(t.N)]
    H, d = G.H, G.dk
    assert w["gdn"]["bytes"] == T * H * (8 * d + 8) + (t.N + int((pos0 > 0).sum())) * H * d * d * 4
    assert w["flops"] == w["attn"]["attn"]["flops"] + w["gdn"]["flops"] + w["readout"]["flops"]
