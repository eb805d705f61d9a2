"""Request-sharded rounds: one process per GPU, no exchange on the data path.

A key is visible to a query only inside the same request (rainbus summary
"方法步骤详情" step 2: j_y = j_x), and every request owns its GDN state S_P and
conv window.  A round therefore splits at request boundaries into independent
sub-rounds.  Each rank builds its own metadata and runs the whole layer on
its requests; only the option probabilities are gathered afterwards.  The
onedev summary ("어떻게 쓰나") splits rounds that exceed a capacity bucket the
same way.

This module only moves rows between stream layouts; it holds none of the
layer's arithmetic.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

from .workloads import Round


def request_tokens(rnd: Round) -> np.ndarray:
    """Stream tokens of each request: its trunk rows in the stream plus its questions."""
    tok = (rnd.trunk_len - rnd.prefix_len).astype(np.int64)
    first = 0
    for j in range(rnd.R):
        n = int(rnd.n_q[j])
        tok[j] += int(rnd.q_len[first:first + n].sum())
        first += n
    return tok


def assign_requests(tokens: Sequence[int], world: int) -> List[List[int]]:
    """Balance requests over `world` ranks by stream tokens.

    Requests are taken in decreasing token count (ties: lower index first) and
    each goes to the rank with the fewest tokens so far (ties: lower rank).
    Every rank's list is returned in request order.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    tokens = [int(t) for t in tokens]
    order = sorted(range(len(tokens)), key=lambda j: (-tokens[j], j))
    load = [0] * world
    out: List[List[int]] = [[] for _ in range(world)]
    for j in order:
        r = min(range(world), key=lambda i: (load[i], i))
        out[r].append(j)
        load[r] += tokens[j]
    return [sorted(x) for x in out]


def _layout(rnd: Round):
    """Stream row offsets: trunk start per request, question start per question."""
    trunk_rows = (rnd.trunk_len - rnd.prefix_len).astype(np.int64)
    trunk_start = np.concatenate([[0], np.cumsum(trunk_rows)[:-1]]) if rnd.R else np.zeros(0, np.int64)
    q0 = int(trunk_rows.sum())
    q_start = q0 + np.concatenate([[0], np.cumsum(rnd.q_len.astype(np.int64))[:-1]]) if rnd.Nq else \
        np.zeros(0, np.int64)
    first_q = np.concatenate([[0], np.cumsum(rnd.n_q.astype(np.int64))[:-1]]) if rnd.R else np.zeros(0, np.int64)
    prefix_off = np.concatenate([[0], np.cumsum(rnd.prefix_len.astype(np.int64))[:-1]]) if rnd.R else \
        np.zeros(0, np.int64)
    return trunk_rows, trunk_start, q_start, first_q, prefix_off


def shard_rows(rnd: Round, requests: Sequence[int]) -> Tuple[np.ndarray, List[int]]:
    """Stream rows of `rnd` that form the sub-round of `requests` (in its stream order:
    the chosen trunks, then their questions), and the global question indices."""
    trunk_rows, trunk_start, q_start, first_q, _ = _layout(rnd)
    qids: List[int] = []
    for j in requests:
        qids.extend(range(int(first_q[j]), int(first_q[j]) + int(rnd.n_q[j])))
    rows = [np.arange(trunk_start[j], trunk_start[j] + trunk_rows[j]) for j in requests]
    rows += [np.arange(q_start[i], q_start[i] + int(rnd.q_len[i])) for i in qids]
    rows = np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)
    return rows, qids


def shard_round(rnd: Round, requests: Sequence[int], T_cap: int = None) -> Tuple[Round, List[int]]:
    """The sub-round made of `requests` (indices into `rnd`, in request order).

    Returns the sub-round and the global indices of its questions, in the
    sub-round's question order.  Its stream holds the chosen trunks, then
    their questions grouped by request; pad rows at the tail up to `T_cap`
    (default: the round's capacity).  Prefix rows, option weights and layer
    weights are carried along.
    """
    req = [int(j) for j in requests]
    if sorted(req) != req or len(set(req)) != len(req) or any(j < 0 or j >= rnd.R for j in req):
        raise ValueError("requests must be distinct indices in increasing order")
    cap = rnd.T_cap if T_cap is None else int(T_cap)
    prefix_off = _layout(rnd)[4]
    rows, qids = shard_rows(rnd, req)  # stream rows of the sub-round, in order: trunks, then questions
    if rows.shape[0] > cap:
        raise ValueError(f"shard of {rows.shape[0]} tokens exceeds capacity {cap}")

    def move(a: np.ndarray) -> np.ndarray:
        out = np.zeros((cap,) + a.shape[1:], dtype=a.dtype)
        out[:rows.shape[0]] = a[rows]
        return out

    layers = {}
    for name, lay in rnd.layers.items():
        layers[name] = {k: (v.copy() if k == "conv_w" else move(v)) for k, v in lay.items()}
    prefix = None
    if rnd.prefix is not None and int(rnd.prefix_len[req].sum()) > 0:
        prows = np.concatenate([np.arange(prefix_off[j], prefix_off[j] + int(rnd.prefix_len[j])) for j in req])
        prefix = {name: {k: v[prows].copy() for k, v in lay.items()} for name, lay in rnd.prefix.items()}
    opt_rows = [np.arange(rnd.opt_off[i], rnd.opt_off[i + 1]) for i in qids]
    opt_rows = np.concatenate(opt_rows) if opt_rows else np.zeros(0, np.int64)
    n_opt = rnd.n_opt[qids].astype(np.int32)
    opt_off = np.zeros(len(qids) + 1, dtype=np.int32)
    opt_off[1:] = np.cumsum(n_opt)
    sub = Round(rnd.wid, rnd.trunk_len[req].copy(), rnd.n_q[req].copy(), rnd.q_len[qids].copy(),
                rnd.prefix_len[req].copy(), rnd.ckpt_pos[req].copy(), n_opt, cap, rnd.attn_shapes,
                rnd.gdn_shape, layers, rnd.w_opt[opt_rows].copy(), opt_off, prefix=prefix)
    return sub, qids


def split_to_fit(rnd: Round, cap: int) -> Tuple[List[List[int]], List[int]]:
    """Split a round at request boundaries into groups of requests whose streams each
    hold at most `cap` tokens (requests balanced by tokens, largest first, over the
    fewest groups that fit).  Requests longer than `cap` on their own are returned
    apart (they run without a capacity bucket)."""
    tok = request_tokens(rnd)
    big = [j for j in range(rnd.R) if tok[j] > cap]
    rest = [j for j in range(rnd.R) if tok[j] <= cap]
    if not rest:
        return [], big
    n = max(1, -(-int(tok[rest].sum()) // cap))
    while True:
        parts = assign_requests(tok[rest], n)
        groups = [[rest[i] for i in part] for part in parts if part]
        if all(int(tok[g].sum()) <= cap for g in groups):
            return groups, big
        n += 1


def scatter_probabilities(rnd: Round, parts) -> np.ndarray:
    """Option probabilities of the whole round from the ranks' (question ids, p) parts."""
    p = np.zeros(int(rnd.opt_off[-1]), dtype=np.float32)
    seen = np.zeros(rnd.Nq, dtype=bool)
    for qids, pp in parts:
        off = 0
        for i in qids:
            n = int(rnd.n_opt[i])
            if seen[i]:
                raise ValueError(f"question {i} came from two ranks")
            seen[i] = True
            p[rnd.opt_off[i]:rnd.opt_off[i] + n] = pp[off:off + n]
            off += n
    if not seen.all():
        raise ValueError("some questions came from no rank")
    return p


def shard_shapes(P: np.ndarray, n: np.ndarray, ql: np.ndarray, no: np.ndarray, world: int, rank: int):
    """This rank's requests of a round given by its shapes (trunk lengths P, question
    counts n, question lengths ql, option counts no), balanced by stream tokens over
    `world` ranks: (requests, their P, n, question lengths, option counts, global
    question indices)."""
    first = np.concatenate([[0], np.cumsum(n)]).astype(np.int64)
    tok = [int(P[j]) + int(ql[first[j]:first[j + 1]].sum()) for j in range(P.shape[0])]
    req = assign_requests(tok, world)[rank]
    qids = [i for j in req for i in range(int(first[j]), int(first[j + 1]))]
    return (req, P[req].copy(), n[req].copy(), ql[qids].copy(), no[qids].copy(), qids)
