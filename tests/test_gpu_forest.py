"""Token forests as ONE round of one flat stream on the GPU: fork_build_forest_meta,
one fork_attn call per attention layer (FORK_FOREST: a node's queries read every
ancestor's keys in place), one fork_gdn_forest call per depth (a node starts from its
parent's end state, read by state index), fork_readout on the leaves.  Checked against
the tree oracle, which runs every node as its ancestors' tokens followed by its own."""
import dataclasses

import numpy as np
import pytest

from oracle import forkattn as orc
from tests.gpu_util import ATOL_OUT, RTOL_STATE, TV_MAX, require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATTN = (wl.AttnShape("attn", 16, 4, 128, 0, 10000.0), wl.AttnShape("swa", 16, 4, 128, 64, 10000.0))


def oracle_of(t):
    f32 = {n: {f: (wl.bf16_to_f32(v) if v.dtype == np.uint16 else v) for f, v in lay.items()}
           for n, lay in t.layers.items()}
    return orc.run_tree(f32, t.parent, t.node_len, [(a.name, a.window, a.rope_theta) for a in t.attn_shapes],
                        t.gdn_shape.name, wl.bf16_to_f32(t.w_opt), t.opt_off)


def run_forest(t, flags=0):
    import torch
    from tree_forked_hybrid_gb300.runner import ForestRound
    run = ForestRound(t, flags=flags)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == 0, hex(run.status())
    return run


def check_against_oracle(t, run):
    got_attn, got_gdn, got_p, S_end = run.outputs()
    want = oracle_of(t)
    T = int(t.node_len.sum())
    for a in t.attn_shapes:
        err = np.abs(got_attn[a.name] - want["attn"][a.name][:T]).max()
        assert err <= ATOL_OUT, (a.name, err)
    err = np.abs(got_gdn - want["gdn"][:T]).max()
    assert err <= ATOL_OUT, err
    # every node's end state, per (node, head); nodes whose path holds no token end at zero
    for k in range(t.N):
        for h in range(t.gdn_shape.H):
            ref = want["S_end"][k, h]
            nr = np.linalg.norm(ref)
            if nr == 0:
                assert np.abs(S_end[k, h]).max() == 0, (k, h)
            else:
                rel = np.linalg.norm(S_end[k, h] - ref) / nr
                assert rel <= RTOL_STATE, (k, h, rel)
    tv = orc.total_variation(got_p, want["p"], t.opt_off)
    assert tv.max() <= TV_MAX, tv.max()


def test_forest_matches_tree_oracle():
    require_gpu()
    gdn = wl.GdnShape("gdn", 4, 128, 128, 4, 64)
    # two trees (depth 3 and a leaf root): internal nodes with leaf and internal children,
    # a one-token leaf, lengths across chunk and tile boundaries
    parent = [-1, 0, 0, 1, 1, 1, 2, 2, 3, 3, -1]
    node_len = [300, 120, 80, 90, 40, 33, 65, 1, 50, 17, 45]
    t = wl.make_tree_round(parent, node_len, attn_shapes=ATTN, gdn_shape=gdn, seed=8)
    run = run_forest(t)
    assert run.plan.levels == 4
    check_against_oracle(t, run)


def test_forest_deepest_chain_empty_nodes_and_window_across_ancestors():
    require_gpu()
    attn = (wl.AttnShape("attn", 16, 4, 128, 0, 10000.0), wl.AttnShape("swa", 16, 4, 128, 37, 10000.0))
    gdn = wl.GdnShape("gdn", 2, 128, 128, 4, 64)
    # a chain through all 8 levels (short nodes, one empty, so a window and a chunk span
    # several ancestors), leaves on it at several depths; an empty root with a subtree
    parent = [-1, 0, 1, 2, 3, 4, 5, 6, 6, 6, 2, 4, -1, 12, 13]
    node_len = [70, 2, 0, 29, 1, 66, 5, 3, 40, 1, 9, 130, 0, 33, 7]
    t = wl.make_tree_round(parent, node_len, attn_shapes=attn, gdn_shape=gdn, seed=11)
    run = run_forest(t)
    assert run.plan.levels == 8
    check_against_oracle(t, run)


def test_forest_checks_flag_changes_no_bit():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    gdn = wl.GdnShape("gdn", 2, 128, 128, 4, 64)
    parent = [-1, 0, 0, 1, 1, -1]
    node_len = [150, 70, 20, 3, 64, 9]
    t = wl.make_tree_round(parent, node_len, attn_shapes=ATTN, gdn_shape=gdn, seed=12)
    a = run_forest(t)
    b = run_forest(t, flags=F.FORK_CHECKS)
    for n in a.attn_out:
        assert torch.equal(a.attn_out[n], b.attn_out[n])
    assert torch.equal(a.gdn_out, b.gdn_out)
    assert torch.equal(a.node_state, b.node_state)
    assert torch.equal(a.p, b.p)


def test_a_path_gives_the_same_bits_alone_and_inside_its_forest():
    """Composition invariance: the rows of one leaf's path run alone (a forest of that
    path only) give bit for bit the results they give inside the whole forest."""
    torch = require_gpu()
    gdn = wl.GdnShape("gdn", 2, 128, 128, 4, 64)
    parent = [-1, 0, 0, 1, 1, 2, -1]
    node_len = [200, 45, 70, 16, 90, 33, 12]
    t = wl.make_tree_round(parent, node_len, attn_shapes=ATTN, gdn_shape=gdn, seed=13)
    path = [0, 1, 4]  # root -> 1 -> leaf 4
    start = t.node_start
    rows = np.concatenate([np.arange(start[k], start[k] + node_len[k]) for k in path])
    layers = {n: {f: (v if f == "conv_w" else v[rows]) for f, v in lay.items()} for n, lay in t.layers.items()}
    leaf_i = t.leaves().index(4)
    o0, o1 = int(t.opt_off[leaf_i]), int(t.opt_off[leaf_i + 1])
    sub = dataclasses.replace(t, parent=np.array([-1, 0, 1], np.int32), node_len=np.array([200, 45, 90], np.int32),
                              n_opt=np.array([0, 0, o1 - o0], np.int32), layers=layers, w_opt=t.w_opt[o0:o1],
                              opt_off=np.array([0, o1 - o0], np.int32))
    whole, alone = run_forest(t), run_forest(sub)
    r = torch.from_numpy(rows).to(whole.gdn_out.device)
    n = rows.shape[0]
    for name in whole.attn_out:
        assert torch.equal(whole.attn_out[name].index_select(0, r), alone.attn_out[name][:n]), name
    assert torch.equal(whole.gdn_out.index_select(0, r), alone.gdn_out[:n])
    assert torch.equal(whole.p[o0:o1], alone.p[:o1 - o0])
