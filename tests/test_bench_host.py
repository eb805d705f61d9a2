"""Host logic of bench.py and of request sharding that needs no GPU."""
import numpy as np

import bench
from tree_forked_hybrid_gb300 import shard as S
from tree_forked_hybrid_gb300 import workloads as wl


def test_traffic_is_reported_only_for_the_measured_sources(monkeypatch):
    t = dict(bench.TRAFFIC)
    assert bench._sources_sha256(t["sources"]) == bench._sources_sha256(t["sources"])
    if t["sha256"] is not None:
        assert bench._traffic() == t["bytes"]
    monkeypatch.setitem(bench.TRAFFIC, "sha256", "0" * 64)
    assert bench._traffic() is None
    monkeypatch.setitem(bench.TRAFFIC, "sha256", None)
    assert bench._traffic() is None


def test_more_ranks_than_requests_gives_empty_shards():
    a = wl.AttnShape("attn", 2, 1, 16, 0, 0.0)
    g = wl.GdnShape("gdn", 1, 16, 16, 4, 64)
    rnd = wl.custom_round([5, 3], [1, 2], [2, 4, 1], attn_shapes=(a,), gdn_shape=g, T_cap=64, seed=1)
    parts = S.assign_requests(S.request_tokens(rnd), 4)
    assert sorted(j for p in parts for j in p) == [0, 1]
    assert sum(1 for p in parts if not p) == 2
    sub, qids = S.shard_round(rnd, [])
    assert sub.R == 0 and sub.Nq == 0 and sub.T == 0 and qids == []
    assert np.all(sub.layers["attn"]["q"] == 0)


def _agg_rank(rank, world, port):
    import os

    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, tok = bench.aggregate_over_ranks(torch, dist, "cpu", [12.5, 30.25][rank], [22003, 21711][rank])
        assert ms == 30.25 and tok == 22003 + 21711
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_slowest_time_and_all_tokens():
    import socket

    import pytest
    mp = pytest.importorskip("torch.multiprocessing")
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_agg_rank, args=(2, port), nprocs=2, join=True)
    import torch
    assert bench.aggregate_over_ranks(torch, None, "cpu", 7.0, 5) == (7.0, 5)


def _shard_rank(rank, world, port):
    import os

    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shapes = wl.draw_round_shapes(3, world, seed=3)
        req, P, n, ql, no, qids = S.shard_shapes(*shapes, world, rank)
        # every rank can build its shard as a round of the workload's shapes
        assert int(P.sum() + ql.sum()) <= wl.WORKLOADS[3].T_cap
        p = np.concatenate([np.full(int(k), 1.0 / int(k), np.float32) for k in no]) if len(no) else np.zeros(0)
        parts = [None] * world
        dist.all_gather_object(parts, (qids, p))
        reqs = [None] * world
        dist.all_gather_object(reqs, req)
        if rank == 0:
            assert sorted(j for r in reqs for j in r) == list(range(shapes[0].shape[0]))
            whole = type("W", (), {})()
            whole.Nq, whole.n_opt = int(shapes[2].shape[0]), shapes[3]
            whole.opt_off = np.concatenate([[0], np.cumsum(shapes[3])])
            pall = S.scatter_probabilities(whole, parts)
            assert np.allclose(np.add.reduceat(pall, whole.opt_off[:-1]), 1.0)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_one_round_and_gather_every_question():
    import socket

    import pytest
    mp = pytest.importorskip("torch.multiprocessing")
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_shard_rank, args=(2, port), nprocs=2, join=True)
