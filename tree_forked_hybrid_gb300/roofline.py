"""Algorithmic work of one round (only what the method must do).

Attention: 4*d flops per visible (q-head, query, key) pair (QK^T and PV);
bytes = Q, K, V, O once each (+ the prefix K/V rows of a resumed round).
GDN: chunk-form flops 2*T*H*(3*d^2 + 2.5*C*d) (the recurrence minimum
6*T*H*d^2 is reported beside it); bytes = q, k, v, o in bf16 and alpha, eta
in fp32 per token and head, plus S_P written once and read once per request.
Readout: the question rows and the option weights, bf16.
A token forest (``forest_work``) counts the same per row, with positions along each path.
"""
from __future__ import annotations

import numpy as np

from .workloads import Round


def visible_pairs(rnd: Round, window: int) -> int:
    """sum over stream queries of the number of visible keys (per head)."""
    total = 0
    qi = 0
    for j in range(rnd.R):
        P, pl = int(rnd.trunk_len[j]), int(rnd.prefix_len[j])
        t = np.arange(pl, P, dtype=np.int64)  # trunk query positions; keys 0..t
        k = t + 1
        if window:
            k = np.minimum(k, window)
        total += int(k.sum())
        for _ in range(int(rnd.n_q[j])):
            L = int(rnd.q_len[qi])
            qi += 1
            t = P + np.arange(L, dtype=np.int64)
            k = t + 1  # trunk (positions < P) and the question's own prefix
            if window:
                k = np.minimum(k, window)
            total += int(k.sum())
    return total


def attn_work(rnd: Round, a) -> tuple:
    pairs = visible_pairs(rnd, a.window)
    flops = 4 * a.d * a.Hq * pairs
    T = rnd.T
    nbytes = T * (2 * a.Hq + 2 * a.Hkv) * a.d * 2 + int(rnd.prefix_len.sum()) * 2 * a.Hkv * a.d * 2
    return flops, nbytes


def gdn_work(rnd: Round) -> tuple:
    g = rnd.gdn_shape
    T, H, d, C = rnd.T, g.H, g.dk, g.chunk
    flops = 2 * T * H * (3 * d * d + 2.5 * C * d)
    flops_min = 6 * T * H * d * d
    nbytes = T * H * (8 * d + 8) + 2 * rnd.R * H * d * d * 4
    return flops, flops_min, nbytes


def readout_work(rnd: Round) -> tuple:
    D = rnd.D
    return 2 * int(rnd.opt_off[-1]) * D, (rnd.Nq + int(rnd.opt_off[-1])) * D * 2


def round_work(rnd: Round) -> dict:
    out = {"attn": {}, "T": rnd.T}
    F = B = 0
    for a in rnd.attn_shapes:
        f, b = attn_work(rnd, a)
        out["attn"][a.name] = {"flops": f, "bytes": b}
        F += f
        B += b
    gf, gmin, gb = gdn_work(rnd)
    out["gdn"] = {"flops": gf, "flops_min": gmin, "bytes": gb}
    rf, rb = readout_work(rnd)
    out["readout"] = {"flops": rf, "bytes": rb}
    out["flops"] = F + gf + rf
    out["bytes"] = B + gb + rb
    return out


def forest_first_positions(tree) -> np.ndarray:
    """Position of every node's first token: the total length of its ancestors."""
    pos0 = np.zeros(tree.N, dtype=np.int64)
    for k in range(tree.N):  # parents precede their children
        p = int(tree.parent[k])
        pos0[k] = 0 if p < 0 else pos0[p] + int(tree.node_len[p])
    return pos0


def forest_positions(tree) -> np.ndarray:
    """Position of every row of a token forest (node after node): its index in its node's
    sequence (the ancestors' tokens, root first, then the node's own)."""
    pos0 = forest_first_positions(tree)
    return np.concatenate([pos0[k] + np.arange(int(tree.node_len[k]), dtype=np.int64) for k in range(tree.N)]
                          + [np.zeros(0, np.int64)])


def forest_work(tree) -> dict:
    """Algorithmic work of a token forest run as one round: every row is a query once and a
    key/value row read once; a query at position t sees min(t + 1, W) keys of its path; the
    recurrence runs every row once, each node writes its end state once and a node with
    tokens before it reads its parent's once."""
    t = forest_positions(tree)
    T = int(t.shape[0])
    out = {"attn": {}, "T": T}
    F = B = 0
    for a in tree.attn_shapes:
        k = t + 1
        if a.window:
            k = np.minimum(k, a.window)
        f = 4 * a.d * a.Hq * int(k.sum())
        b = T * (2 * a.Hq + 2 * a.Hkv) * a.d * 2
        out["attn"][a.name] = {"flops": f, "bytes": b}
        F += f
        B += b
    g = tree.gdn_shape
    H, d, C = g.H, g.dk, g.chunk
    resumed = int((forest_first_positions(tree) > 0).sum())
    gf = 2 * T * H * (3 * d * d + 2.5 * C * d)
    gb = T * H * (8 * d + 8) + (tree.N + resumed) * H * d * d * 4
    out["gdn"] = {"flops": gf, "bytes": gb}
    n_leaves = len(tree.leaves())
    n_opt = int(tree.opt_off[-1])
    D = H * g.dv
    rf, rb = 2 * n_opt * D, (n_leaves + n_opt) * D * 2
    out["readout"] = {"flops": rf, "bytes": rb}
    out["flops"] = F + gf + rf
    out["bytes"] = B + gb + rb
    return out


def roofline_time(work: dict, peak_tflops: float, peak_gbs: float) -> float:
    """Seconds: the slower of the FLOPs at peak and the bytes at peak."""
    return max(work["flops"] / (peak_tflops * 1e12), work["bytes"] / (peak_gbs * 1e9))
