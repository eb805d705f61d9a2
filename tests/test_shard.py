"""Request-sharded rounds (the multi-GPU path) on CPU.

A round splits at request boundaries with no exchange between ranks (a key is
visible to a query only inside its request, and each request owns its GDN
state).  Two `gloo` ranks each run the oracle on their shard; the gathered
results must equal, bit for bit, the oracle on the whole round.
"""
import os
import socket

import numpy as np
import pytest

from oracle import forkattn as orc
from tree_forked_hybrid_gb300 import shard as S
from tree_forked_hybrid_gb300 import workloads as wl


def small_round():
    a = wl.AttnShape("attn", 2, 1, 16, 0, 10000.0)
    w = wl.AttnShape("swa", 2, 1, 16, 8, 10000.0)
    g = wl.GdnShape("gdn", 2, 16, 16, 4, 64)
    # request 3 has an empty trunk; lengths straddle the conv width and the window
    return wl.custom_round([20, 9, 33, 0, 14], [2, 1, 3, 1, 2], [5, 7, 3, 11, 4, 6, 2, 9, 1],
                           attn_shapes=(a, w), gdn_shape=g, T_cap=160, seed=5)


def view_of(rnd):
    lay = {n: {k: (rnd.f32(n, k) if k != "conv_w" else v[k]) for k in v} for n, v in rnd.layers.items()}
    return orc.RoundView(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, lay)


def oracle_results(rnd):
    """Per question: attention rows of every layer, GDN rows and probabilities; per request: S_P."""
    view = view_of(rnd)
    m = view.meta
    attn = {a.name: orc.run_attention(view, a.name, window=a.window, rope_theta=a.rope_theta)
            for a in rnd.attn_shapes}
    g = orc.run_gdn(view, rnd.gdn_shape.name)
    p = orc.run_readout(view, g["o"].reshape(rnd.T_cap, -1), rnd.w_opt_f32(), rnd.opt_off)
    per_q = []
    for i in range(rnd.Nq):
        st, L = int(m["seg_start"][rnd.R + i]), int(m["seg_len"][rnd.R + i])
        rows = {n: o[st:st + L] for n, o in attn.items()}
        rows["gdn"] = g["o"][st:st + L]
        per_q.append((rows, p[rnd.opt_off[i]:rnd.opt_off[i + 1]]))
    return per_q, g["S_P"], p


def test_assignment_covers_each_request_once_and_balances():
    rnd = small_round()
    tok = S.request_tokens(rnd)
    assert tok.tolist() == [32, 12, 54, 2, 24]
    for world in (1, 2, 3, 5, 7):
        parts = S.assign_requests(tok, world)
        assert len(parts) == world
        flat = sorted(j for p in parts for j in p)
        assert flat == list(range(rnd.R))
        loads = [int(tok[p].sum()) for p in parts]
        assert max(loads) - min(loads) <= int(tok.max())
    assert S.assign_requests(tok, 2) == [[1, 2], [0, 3, 4]]


def test_shard_rows_are_the_round_rows():
    rnd = small_round()
    full = view_of(rnd)
    for part in S.assign_requests(S.request_tokens(rnd), 2):
        sub, qids = S.shard_round(rnd, part)
        sv = view_of(sub)
        assert sub.T == sum(int(S.request_tokens(rnd)[j]) for j in part)
        for jj, j in enumerate(part):
            for name, lay in rnd.layers.items():
                for field in lay:
                    if field == "conv_w":
                        continue
                    a = sv.sequence_rows(name, field, jj, None)
                    b = full.sequence_rows(name, field, j, None)
                    assert np.array_equal(a, b)
                    for k, qi in enumerate(sv.questions_of(jj)):
                        a = sv.sequence_rows(name, field, jj, qi)
                        b = full.sequence_rows(name, field, j, full.questions_of(j)[k])
                        assert np.array_equal(a, b)
        for k, i in enumerate(qids):
            n = int(rnd.n_opt[i])
            assert np.array_equal(sub.w_opt[sub.opt_off[k]:sub.opt_off[k] + n],
                                  rnd.w_opt[rnd.opt_off[i]:rnd.opt_off[i] + n])
        assert np.array_equal(sub.layers["gdn"]["conv_w"], rnd.layers["gdn"]["conv_w"])


def test_shard_rejects_bad_request_lists():
    rnd = small_round()
    for bad in ([1, 0], [0, 0], [5], [-1]):
        with pytest.raises(ValueError):
            S.shard_round(rnd, bad)
    with pytest.raises(ValueError):
        S.shard_round(rnd, [0, 2], T_cap=50)  # 86 tokens


def _rank_main(rank, world, port):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rnd = small_round()
        part = S.assign_requests(S.request_tokens(rnd), world)[rank]
        sub, qids = S.shard_round(rnd, part)
        per_q, S_P, p = oracle_results(sub)
        mine = {"requests": part, "qids": qids, "per_q": per_q, "S_P": S_P, "p": p}
        got = [None] * world
        dist.all_gather_object(got, mine)
        if rank == 0:
            want_q, want_S, want_p = oracle_results(rnd)
            p_all = S.scatter_probabilities(rnd, [(g["qids"], g["p"]) for g in got])
            assert np.array_equal(p_all, want_p)
            for g in got:
                for jj, j in enumerate(g["requests"]):
                    assert np.array_equal(g["S_P"][jj], want_S[j])
                for k, i in enumerate(g["qids"]):
                    rows, pq = g["per_q"][k]
                    wrows, wp = want_q[i]
                    assert np.array_equal(pq, wp)
                    for name in wrows:
                        assert np.array_equal(rows[name], wrows[name]), (name, i)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reproduce_the_whole_round():
    mp = pytest.importorskip("torch.multiprocessing")
    mp.spawn(_rank_main, args=(2, _free_port()), nprocs=2, join=True)


def test_split_to_fit_partitions_requests_under_the_capacity():
    """The graph pool's split of a round over its largest bucket: every request exactly
    once, each group's stream within the capacity, requests longer than the capacity on
    their own (they run without a graph)."""
    rnd = small_round()
    tok = S.request_tokens(rnd)
    for cap in (20, 32, 40, 64, 200):
        groups, big = S.split_to_fit(rnd, cap)
        seen = sorted([j for g in groups for j in g] + list(big))
        assert seen == list(range(rnd.R)), cap
        assert all(int(tok[g].sum()) <= cap for g in groups), cap
        assert sorted(big) == [j for j in range(rnd.R) if tok[j] > cap], cap
        assert all(len(g) > 0 for g in groups)
    # a capacity that holds the whole round gives one group
    groups, big = S.split_to_fit(rnd, int(tok.sum()))
    assert len(groups) == 1 and big == []
    # every request above the capacity: nothing to group
    groups, big = S.split_to_fit(rnd, 1)
    assert groups == [] and sorted(big) == [j for j in range(rnd.R) if tok[j] > 1]


def test_split_to_fit_sub_rounds_keep_every_question():
    """Sub-rounds of the split hold, together, every question of the round once, with the
    same question lengths and option counts."""
    rnd = small_round()
    groups, big = S.split_to_fit(rnd, 40)
    qids = []
    for g in groups + [[j] for j in big]:
        sub, q = S.shard_round(rnd, g, T_cap=rnd.T_cap)
        assert sub.R == len(g) and sub.Nq == len(q)
        assert list(sub.n_opt) == [int(rnd.n_opt[i]) for i in q]
        qids.extend(q)
    assert sorted(qids) == list(range(rnd.Nq))
