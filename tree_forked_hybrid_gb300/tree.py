"""Token trees (branches that fork again) on the two-call layer, one round per depth.

The rainbus summary ("未来方向" (2)) names trees deeper than trunk + questions
as the method's extension: a tree of draft tokens has the shape of a request
tree and runs in the same flat stream.  The layer's resume path already
carries everything a deeper level needs (prefix rows held outside the stream,
a trunk that starts from a given state and conv window), so a forest runs as
one round per depth:

* a node with children is a request of the round for its depth: its own
  tokens are the trunk, its ancestors' tokens are the trunk's prefix rows,
  and the trunk starts from its parent's end state and conv window (the
  previous round's S_P and conv window of the parent's request);
* its leaf children are the request's questions; its other children are
  requests of the next round;
* a leaf root is a request with an empty trunk and one question.

Every node's result is then that of its own sequence (ancestors' tokens,
then its own).  This module only moves rows and indices.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np

from .workloads import Round, TreeRound


@dataclasses.dataclass
class Level:
    """One round of the decomposition."""

    depth: int
    round: Round
    request_nodes: List[int]   # request j -> tree node (-1: an empty trunk for a leaf root)
    question_nodes: List[int]  # question i -> tree node (a leaf)
    parent_request: List[int]  # request j -> request index of its parent node in the previous level, or -1


def _pad64(n: int) -> int:
    return max(64, (n + 63) // 64 * 64)


def decompose(tree: TreeRound) -> List[Level]:
    N = tree.N
    start = tree.node_start
    depth = [tree.depth(k) for k in range(N)]
    has_children = [not tree.is_leaf(k) for k in range(N)]
    leaf_index = {k: i for i, k in enumerate(tree.leaves())}
    levels: List[Level] = []
    prev_req_of_node: Dict[int, int] = {}
    for d in range(max(depth) + 1 if N else 0):
        reqs = [k for k in range(N) if depth[k] == d and (has_children[k] or (d == 0 and not has_children[k]))]
        if not reqs:
            break
        request_nodes, question_nodes, parent_request = [], [], []
        trunk_len, n_q, prefix_len = [], [], []
        trunk_rows, prefix_rows = [], []
        for k in reqs:
            if has_children[k]:
                anc = tree.ancestors(k)
                pl = int(sum(int(tree.node_len[a]) for a in anc))
                qs = [c for c in tree.children(k) if tree.is_leaf(c)]
                request_nodes.append(k)
                trunk_len.append(pl + int(tree.node_len[k]))
                prefix_len.append(pl)
                trunk_rows.append(np.arange(start[k], start[k] + tree.node_len[k]))
                prefix_rows.append(np.concatenate([np.arange(start[a], start[a] + tree.node_len[a]) for a in anc])
                                   if anc else np.zeros(0, np.int64))
                parent_request.append(prev_req_of_node[int(tree.parent[k])] if tree.parent[k] >= 0 else -1)
            else:  # a leaf root: empty trunk, the root is the question
                qs = [k]
                request_nodes.append(-1)
                trunk_len.append(0)
                prefix_len.append(0)
                trunk_rows.append(np.zeros(0, np.int64))
                prefix_rows.append(np.zeros(0, np.int64))
                parent_request.append(-1)
            n_q.append(len(qs))
            question_nodes.extend(qs)
        q_rows = [np.arange(start[c], start[c] + tree.node_len[c]) for c in question_nodes]
        rows = np.concatenate(trunk_rows + q_rows).astype(np.int64) if (trunk_rows or q_rows) else np.zeros(0, np.int64)
        T_cap = _pad64(rows.shape[0])

        def move(a):
            out = np.zeros((T_cap,) + a.shape[1:], dtype=a.dtype)
            out[:rows.shape[0]] = a[rows]
            return out

        layers = {name: {f: (v.copy() if f == "conv_w" else move(v)) for f, v in lay.items()}
                  for name, lay in tree.layers.items()}
        prows = np.concatenate(prefix_rows).astype(np.int64) if prefix_rows else np.zeros(0, np.int64)
        prefix = None
        if prows.shape[0] > 0:
            prefix = {name: {f: v[prows].copy() for f, v in lay.items() if f != "conv_w"}
                      for name, lay in tree.layers.items()}
        li = [leaf_index[c] for c in question_nodes]
        opt_rows = [np.arange(tree.opt_off[i], tree.opt_off[i + 1]) for i in li]
        opt_rows = np.concatenate(opt_rows).astype(np.int64) if opt_rows else np.zeros(0, np.int64)
        n_opt = np.array([tree.opt_off[i + 1] - tree.opt_off[i] for i in li], dtype=np.int32)
        opt_off = np.zeros(len(li) + 1, dtype=np.int32)
        opt_off[1:] = np.cumsum(n_opt)
        R = len(reqs)
        rnd = Round(-1, np.array(trunk_len, np.int32), np.array(n_q, np.int32),
                    np.array([int(tree.node_len[c]) for c in question_nodes], np.int32),
                    np.array(prefix_len, np.int32), np.full(R, -1, np.int32), n_opt, T_cap, tree.attn_shapes,
                    tree.gdn_shape, layers, tree.w_opt[opt_rows].copy(), opt_off, prefix=prefix)
        levels.append(Level(d, rnd, request_nodes, question_nodes, parent_request))
        prev_req_of_node = {k: j for j, k in enumerate(request_nodes) if k >= 0}
    return levels


def node_rows(level: Level, tree: TreeRound):
    """(tree node, stream rows of that node in the level's round) for every trunk and question."""
    out = []
    r = level.round
    pos = 0
    for j, k in enumerate(level.request_nodes):
        L = int(r.trunk_len[j] - r.prefix_len[j])
        if k >= 0:
            out.append((k, np.arange(pos, pos + L)))
        pos += L
    for i, k in enumerate(level.question_nodes):
        L = int(r.q_len[i])
        out.append((k, np.arange(pos, pos + L)))
        pos += L
    return out
