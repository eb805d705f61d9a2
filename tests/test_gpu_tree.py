"""Token trees of depth 3 on the GPU, one round per depth, against the tree oracle
(every node run as its ancestors' tokens followed by its own)."""
import numpy as np
import pytest

from oracle import forkattn as orc
from tests.gpu_util import ATOL_OUT, require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_tree_levels_match_tree_oracle():
    torch = require_gpu()
    from tree_forked_hybrid_gb300.runner import TreeRunner

    attn = (wl.AttnShape("attn", 16, 4, 128, 0, 10000.0), wl.AttnShape("swa", 16, 4, 128, 64, 10000.0))
    gdn = wl.GdnShape("gdn", 4, 128, 128, 4, 64)
    # two trees (depth 3 and a leaf root): internal nodes with leaf and internal children,
    # a one-token leaf, lengths across chunk and tile boundaries
    parent = [-1, 0, 0, 1, 1, 1, 2, 2, 3, 3, -1]
    node_len = [300, 120, 80, 90, 40, 33, 65, 1, 50, 17, 45]
    t = wl.make_tree_round(parent, node_len, attn_shapes=attn, gdn_shape=gdn, seed=8)
    run = TreeRunner(t)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == 0
    assert len(run.levels) == 3
    got_attn, got_gdn, got_p = run.outputs()

    f32 = {n: {f: (wl.bf16_to_f32(v) if v.dtype == np.uint16 else v) for f, v in lay.items()}
           for n, lay in t.layers.items()}
    want = orc.run_tree(f32, t.parent, t.node_len, [(a.name, a.window, a.rope_theta) for a in attn], gdn.name,
                        wl.bf16_to_f32(t.w_opt), t.opt_off)
    for a in attn:
        err = np.abs(got_attn[a.name] - want["attn"][a.name]).max()
        assert err <= ATOL_OUT, (a.name, err)
    err = np.abs(got_gdn - want["gdn"]).max()
    assert err <= ATOL_OUT, err
    tv = orc.total_variation(got_p, want["p"], t.opt_off)
    assert tv.max() <= 1e-3, tv.max()


def test_tree_with_a_level_without_questions_and_an_empty_root():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import tree as TR
    from tree_forked_hybrid_gb300.runner import TreeRunner

    attn = (wl.AttnShape("attn", 16, 4, 128, 0, 10000.0),)
    gdn = wl.GdnShape("gdn", 2, 128, 128, 4, 64)
    # root 0 -> 1 -> 2 -> leaves 3, 4 (level 1 has no leaf children); empty root 5 -> 6 -> leaf 7
    parent = [-1, 0, 1, 2, 2, -1, 5, 6]
    node_len = [70, 33, 65, 20, 1, 0, 40, 9]
    t = wl.make_tree_round(parent, node_len, attn_shapes=attn, gdn_shape=gdn, seed=9)
    assert any(lv.round.Nq == 0 for lv in TR.decompose(t))
    run = TreeRunner(t)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == 0
    got_attn, got_gdn, got_p = run.outputs()
    f32 = {n: {f: (wl.bf16_to_f32(v) if v.dtype == np.uint16 else v) for f, v in lay.items()}
           for n, lay in t.layers.items()}
    want = orc.run_tree(f32, t.parent, t.node_len, [(a.name, a.window, a.rope_theta) for a in attn], gdn.name,
                        wl.bf16_to_f32(t.w_opt), t.opt_off)
    assert np.abs(got_attn["attn"] - want["attn"]["attn"]).max() <= ATOL_OUT
    assert np.abs(got_gdn - want["gdn"]).max() <= ATOL_OUT
    assert orc.total_variation(got_p, want["p"], t.opt_off).max() <= 1e-3
