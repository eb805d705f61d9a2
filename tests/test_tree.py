"""Token trees (branches that fork again): the tree oracle and its decomposition
into one round per depth.

Pins of the tree oracle: a depth-1 tree is a round (the round oracle, pinned
elsewhere); a chain of nodes is one plain sequence; a node's outputs do not
depend on other branches.  The decomposition (own tokens as the trunk,
ancestors' tokens as prefix rows, leaf children as questions) executed level
by level through the round oracle must reproduce the tree oracle bit for bit.
"""
import numpy as np

from oracle import forkattn as orc
from tree_forked_hybrid_gb300 import tree as TR
from tree_forked_hybrid_gb300 import workloads as wl

A1 = wl.AttnShape("attn", 2, 1, 16, 0, 10000.0)
A2 = wl.AttnShape("swa", 2, 1, 16, 6, 10000.0)
G = wl.GdnShape("gdn", 2, 16, 16, 4, 64)


def f32_layers(layers):
    return {n: {f: (wl.bf16_to_f32(v) if v.dtype == np.uint16 else v) for f, v in lay.items()}
            for n, lay in layers.items()}


def tree_oracle(t):
    return orc.run_tree(f32_layers(t.layers), t.parent, t.node_len,
                        [(a.name, a.window, a.rope_theta) for a in t.attn_shapes], t.gdn_shape.name,
                        wl.bf16_to_f32(t.w_opt), t.opt_off)


def forest():
    # two trees of depth 3 and a leaf root: internal nodes with and without leaf children,
    # an empty root, one-token leaves, lengths around the conv width and the window
    parent = [-1, 0, 0, 1, 1, 2, 3, 3, -1, 8, 9, 9, -1]
    node_len = [9, 5, 4, 3, 6, 2, 1, 7, 0, 8, 4, 5, 6]
    return wl.make_tree_round(parent, node_len, attn_shapes=(A1, A2), gdn_shape=G, seed=3)


def run_levels_with_round_oracle(t):
    """Each level's round through the round oracle; outputs scattered back to tree rows."""
    T = int(t.node_len.sum())
    start = t.node_start
    out = {"attn": {a.name: np.zeros((T, a.Hq, a.d), np.float32) for a in t.attn_shapes},
           "gdn": np.zeros((T, G.H, G.dv), np.float32), "p": np.zeros(int(t.opt_off[-1]), np.float32)}
    leaf_index = {k: i for i, k in enumerate(t.leaves())}
    for lv in TR.decompose(t):
        r = lv.round
        pref = f32_layers(r.prefix) if r.prefix is not None else None
        view = orc.RoundView(r.desc(), r.R, r.Nq, r.T_cap, f32_layers(r.layers), prefix=pref)
        res = {a.name: orc.run_attention(view, a.name, window=a.window, rope_theta=a.rope_theta)
               for a in r.attn_shapes}
        g = orc.run_gdn(view, G.name)
        p = orc.run_readout(view, g["o"].reshape(r.T_cap, -1), wl.bf16_to_f32(r.w_opt), r.opt_off)
        for k, rows in TR.node_rows(lv, t):
            for n in res:
                out["attn"][n][start[k]:start[k] + rows.shape[0]] = res[n][rows]
            out["gdn"][start[k]:start[k] + rows.shape[0]] = g["o"][rows]
        for i, k in enumerate(lv.question_nodes):
            li = leaf_index[k]
            out["p"][t.opt_off[li]:t.opt_off[li + 1]] = p[r.opt_off[i]:r.opt_off[i + 1]]
    return out


def test_decomposition_levels():
    t = forest()
    lv = TR.decompose(t)
    assert [l.depth for l in lv] == [0, 1, 2]
    assert lv[0].request_nodes == [0, 8, -1] and lv[0].question_nodes == [12]
    assert lv[1].request_nodes == [1, 2, 9] and lv[1].question_nodes == [4, 5, 10, 11]
    assert lv[1].parent_request == [0, 0, 1]
    assert lv[2].request_nodes == [3] and lv[2].question_nodes == [6, 7] and lv[2].parent_request == [0]
    r2 = lv[2].round
    assert r2.prefix_len.tolist() == [9 + 5] and r2.trunk_len.tolist() == [9 + 5 + 3]
    assert sorted(k for l in lv for k in l.question_nodes) == t.leaves()


def test_depth_one_tree_is_a_round():
    t = wl.make_tree_round([-1, 0, 0, 0], [12, 5, 1, 7], attn_shapes=(A1, A2), gdn_shape=G, seed=4)
    want = tree_oracle(t)
    got = run_levels_with_round_oracle(t)
    assert len(TR.decompose(t)) == 1
    for n in want["attn"]:
        assert np.array_equal(got["attn"][n], want["attn"][n])
    assert np.array_equal(got["gdn"], want["gdn"])
    assert np.array_equal(got["p"], want["p"])


def test_chain_is_one_sequence():
    # the window (6 keys) crosses the node boundaries at rows 6 and 15
    t = wl.make_tree_round([-1, 0, 1], [6, 9, 5], attn_shapes=(A1, A2), gdn_shape=G, seed=5)
    res = tree_oracle(t)
    L = f32_layers(t.layers)
    for name, a in (("attn", A1), ("swa", A2)):
        o = orc.attention_sequence(L[name]["q"][:20], L[name]["k"][:20], L[name]["v"][:20], window=a.window,
                                   rope_theta=a.rope_theta)
        # the tree oracle computes each node's query rows in separate calls: equal up to the
        # summation order of the library matmul
        assert np.abs(res["attn"][name] - o).max() <= 1e-6
    g = L["gdn"]
    o, S, _, _ = orc.gdn_sequence(g["q"][:20], g["k"][:20], g["v"][:20], g["alpha"][:20], g["eta"][:20],
                                  g["conv_w"])
    assert np.array_equal(res["gdn"], o)
    assert np.array_equal(res["S_end"][2], S)
    # every node's end state is the sequence's state after that node's last row
    for k, n in ((0, 6), (1, 15)):
        _, S_k, _, _ = orc.gdn_sequence(g["q"][:n], g["k"][:n], g["v"][:n], g["alpha"][:n], g["eta"][:n],
                                        g["conv_w"])
        assert np.array_equal(res["S_end"][k], S_k), k


def test_node_results_do_not_depend_on_other_branches():
    t = forest()
    base = tree_oracle(t)
    t2 = forest()
    start = t2.node_start
    for n, lay in t2.layers.items():  # perturb the subtree of node 2 (nodes 2 and 5)
        for f, v in lay.items():
            if f == "conv_w":
                continue
            for k in (2, 5):
                v[start[k]:start[k] + t2.node_len[k]] = v[start[k]:start[k] + t2.node_len[k]][::-1].copy()
    pert = tree_oracle(t2)
    for k in (0, 1, 3, 4, 6, 7, 9, 10, 11, 12):
        rows = slice(start[k], start[k] + t.node_len[k])
        assert np.array_equal(base["gdn"][rows], pert["gdn"][rows])
        for n in base["attn"]:
            assert np.array_equal(base["attn"][n][rows], pert["attn"][n][rows])
    assert not np.array_equal(base["gdn"][start[5]:start[5] + 2], pert["gdn"][start[5]:start[5] + 2])


def test_levels_through_round_oracle_reproduce_the_tree():
    t = forest()
    want = tree_oracle(t)
    got = run_levels_with_round_oracle(t)
    for n in want["attn"]:
        assert np.array_equal(got["attn"][n], want["attn"][n]), n
    assert np.array_equal(got["gdn"], want["gdn"])
    assert np.array_equal(got["p"], want["p"])


def random_forest(seed):
    rng = np.random.default_rng(seed)
    parent, node_len = [], []
    for k in range(int(rng.integers(3, 12))):
        if k == 0 or rng.random() < 0.15:
            parent.append(-1)
        else:
            # attach to an earlier node whose depth stays below 4
            cand = [p for p in range(k) if _depth(parent, p) < 3]
            parent.append(int(rng.choice(cand)))
        node_len.append(int(rng.integers(0, 12)))
    leaves = [k for k in range(len(parent)) if k not in parent]
    for k in leaves:
        node_len[k] = max(node_len[k], 1)
    return wl.make_tree_round(parent, node_len, attn_shapes=(A1, A2), gdn_shape=G, seed=seed)


def _depth(parent, k):
    d = 0
    while parent[k] >= 0:
        k = parent[k]
        d += 1
    return d


def test_random_forests_through_round_oracle():
    for seed in range(12):
        t = random_forest(100 + seed)
        want = tree_oracle(t)
        got = run_levels_with_round_oracle(t)
        for n in want["attn"]:
            assert np.array_equal(got["attn"][n], want["attn"][n]), (seed, n)
        assert np.array_equal(got["gdn"], want["gdn"]), seed
        assert np.array_equal(got["p"], want["p"]), seed
        qs = sorted(k for lv in TR.decompose(t) for k in lv.question_nodes)
        assert qs == t.leaves(), seed
