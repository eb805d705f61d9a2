"""Flat-graph replay per capacity bucket (GraphPool), against the CPU oracle.

One whole-layer CUDA graph is captured per stream capacity; a round runs in the
smallest bucket that holds it, a round over the largest bucket is split at
request boundaries, and a request too long for every bucket runs eagerly.  Every
output of every case is compared with the oracle at the layer tolerances.  The
metadata built from the fixed-capacity device descriptor equals the one built
from the packed descriptor word for word.
"""
import numpy as np
import pytest

from oracle import forkattn as orc
from tests.gpu_util import ATOL_OUT, TV_MAX, oracle_view, require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

A = wl.AttnShape("attn", 8, 2, 128, 0, 10000.0)
SWA = wl.AttnShape("swa", 8, 2, 128, 96, 10000.0)
G = wl.GdnShape("gdn", 2, 128, 128, 4, 64)


def rnd_of(P, n, ql, seed, T_cap=None):
    T = int(np.sum(P) + np.sum(ql))
    return wl.custom_round(P, n, ql, attn_shapes=(A, SWA), gdn_shape=G, T_cap=T_cap or max(T, 1), seed=seed)


def check_against_oracle(rnd, res):
    view = oracle_view(rnd)
    T = rnd.T
    for a in rnd.attn_shapes:
        want = orc.run_attention(view, a.name, window=a.window, rope_theta=a.rope_theta)[:T]
        d = np.abs(res["attn"][a.name] - want)
        assert np.isfinite(res["attn"][a.name]).all() and d.max() <= ATOL_OUT, f"{a.name}: {d.max():.3e}"
    g = orc.run_gdn(view, rnd.gdn_shape.name)
    d = np.abs(res["gdn"] - g["o"][:T])
    assert d.max() <= ATOL_OUT, f"gdn: {d.max():.3e}"
    p_ref = orc.run_readout(view, g["o"].reshape(rnd.T_cap, -1), rnd.w_opt_f32(), rnd.opt_off)
    tv = orc.total_variation(res["p"], p_ref, rnd.opt_off)
    assert tv.max() <= TV_MAX, f"TV {tv.max():.2e}"


@pytest.fixture(scope="module")
def pool():
    require_gpu()
    from tree_forked_hybrid_gb300.runner import GraphPool
    return GraphPool((A, SWA), G, buckets=(1024, 2048, 4096), max_req=8, max_q=24, max_opts=256)


def test_meta_from_device_counts_equals_packed():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300.runner import CapacityRound
    rnd = rnd_of([300, 0, 57], [2, 1, 3], [40, 7, 64, 1, 20, 9], seed=3, T_cap=1024)
    cr = CapacityRound((A, SWA), G, 1024, 8, 24, 256)
    cr.load(rnd)
    F.fork_build_meta_dev(cr.meta, cr.desc)
    ref = F.Meta(1024, 8, 24, cr.tile_tokens)
    F.fork_build_meta(ref, torch.from_numpy(rnd.desc()).cuda(), rnd.R, rnd.Nq)
    torch.cuda.synchronize()
    assert torch.equal(cr.meta.buf, ref.buf)


def test_three_rounds_of_different_counts_replay_one_bucket(pool):
    torch = require_gpu()
    cases = [rnd_of([700, 300], [3, 1], [40, 12, 64, 33], seed=1),
             rnd_of([400, 350, 120, 77, 5], [1, 4, 2, 1, 2], [16, 1, 48, 20, 31, 2, 64, 9, 17, 40], seed=2),
             rnd_of([900], [6], [12, 30, 64, 1, 50, 22], seed=3)]
    for rnd in cases:
        assert 1024 < rnd.T <= 2048
        res = pool.run(rnd)
        assert pool.last_plan == [("graph", 2048, rnd.R, rnd.Nq)]
        check_against_oracle(rnd, res)


def test_round_over_the_largest_bucket_is_split_at_request_boundaries(pool):
    require_gpu()
    rnd = rnd_of([1500, 1200, 1400, 900], [2, 3, 1, 2], [40, 12, 64, 33, 8, 50, 20, 61], seed=4)
    assert rnd.T > 4096
    res = pool.run(rnd)
    assert len(pool.last_plan) >= 2 and all(kind == "graph" for kind, *_ in pool.last_plan)
    check_against_oracle(rnd, res)


def test_request_longer_than_every_bucket_runs_eagerly(pool):
    require_gpu()
    rnd = rnd_of([4200, 300], [2, 1], [40, 64, 20], seed=5)
    res = pool.run(rnd)
    kinds = sorted(kind for kind, *_ in pool.last_plan)
    assert kinds == ["eager", "graph"]
    check_against_oracle(rnd, res)
