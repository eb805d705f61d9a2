"""The whole layer replayed from one CUDA graph (one graph per capacity bucket).

The graph captured for one round must give the eager path's results bit for
bit, and so must a replay after a second round with the same request and
question counts (other lengths, other values) has been loaded into the
captured buffers.
"""
import numpy as np
import pytest

from tests.gpu_util import require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _snapshot(dr, rnd):
    T, n_opt = rnd.T, int(rnd.opt_off[-1])
    out = {f"attn_{k}": v[:T].float().cpu().numpy() for k, v in dr.attn_out.items()}
    out["gdn"] = dr.gdn_out[:T].float().cpu().numpy()
    out["S_P"] = dr.S_P[:rnd.R].cpu().numpy()
    out["p"] = dr.p[:n_opt].cpu().numpy()
    return out


def _same(a, b):
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_graph_replay_matches_eager_on_two_rounds():
    torch = require_gpu()
    from tree_forked_hybrid_gb300.runner import DeviceRound, GraphRound

    a = wl.make_round(1, seed=11)
    ql = np.random.default_rng(5).integers(16, 48, size=a.Nq, endpoint=True)
    b = wl.make_round(1, seed=12, n_q=a.n_q, q_len=ql, n_opt=a.n_opt)
    assert (b.R, b.Nq) == (a.R, a.Nq) and b.T != a.T

    ea = DeviceRound(a)
    ea.run()
    torch.cuda.synchronize()
    want_a = _snapshot(ea, a)

    g = GraphRound(DeviceRound(a))
    g.replay()
    torch.cuda.synchronize()
    assert g.dr.status() == 0
    _same(_snapshot(g.dr, a), want_a)

    g.load(b)
    g.replay()
    torch.cuda.synchronize()
    assert g.dr.status() == 0
    eb = DeviceRound(b)
    eb.run()
    torch.cuda.synchronize()
    _same(_snapshot(g.dr, b), _snapshot(eb, b))


def test_graph_load_rejects_another_bucket():
    require_gpu()
    from tree_forked_hybrid_gb300.runner import DeviceRound, GraphRound

    g = GraphRound(DeviceRound(wl.make_round(0)))
    with pytest.raises(ValueError):
        g.load(wl.make_round(1, seed=3))
