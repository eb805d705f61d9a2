"""Seeded synthetic rounds for the ForkAttention token-mixing layer.

This module only *draws inputs*: round shapes, per-layer q/k/v rows, gates,
conv weights and option weights.  It holds none of the layer's arithmetic, so
both the CPU oracle (through the tests) and the CUDA path consume the very
same arrays.

Shapes follow the five workloads of the Flide pages (tiny round, short
requests, many questions, long documents, wide fork + incremental resume).
The public datasets the pages measure on (RACE, QuALITY, MultiRC, Decision
Index, SWE-agent trajectories) are not available; these draws stand in for
them with the stated length mixes.

Stream order (Flide, "method steps", step 1; onedev summary, "what differs"):
all trunks of the round in request order, then the questions grouped by
request in question order, no padding between requests, zero rows only at
the tail up to the capacity ``T_cap``.

Draw order, from ``numpy.random.default_rng(seed)``:
  1. trunk lengths P[R]; 2. question counts n[R]; 3. question lengths
  q_len[Nq] in request order; 4. option counts |O_i|[Nq];
  5. per layer, in the order of ``layers``: q, k, v ~ N(0,1) (float32, then
  rounded to bfloat16 by round-to-nearest-even); for a Gated DeltaNet layer
  then alpha = sigmoid(N(2, 0.5)) and eta = sigmoid(N(0,1)) per token and
  head (computed in float64, stored as float32) and the depthwise conv
  weights U(-1/sqrt(K), 1/sqrt(K)) as float32;
  6. option weights w_o ~ N(0, 0.02^2), rounded to bfloat16.
A resumed round (workload 4, round B) continues from the same generator.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

# ----------------------------------------------------------------------------
# bfloat16 storage helpers (data format only)
# ----------------------------------------------------------------------------


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> the exactly equal float32 values."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# Workload shapes
# ----------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class AttnShape:
    name: str
    Hq: int
    Hkv: int
    d: int
    window: int  # 0 = full attention
    rope_theta: float  # 0 = no rotary embedding


@dataclasses.dataclass(frozen=True)
class GdnShape:
    name: str
    H: int
    dk: int
    dv: int
    K: int  # causal conv width
    chunk: int


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int
    title: str
    T_cap: int
    attn: tuple  # AttnShape, in layer order
    gdn: GdnShape
    n_opt_range: tuple  # inclusive (lo, hi)


ROPE = 10000.0

WORKLOADS: Dict[int, Workload] = {
    0: Workload(0, "tiny round: 1 request, P=64, questions 8/12/16, d=64", 128,
                (AttnShape("attn", 1, 1, 64, 0, 0.0),),
                GdnShape("gdn", 1, 64, 64, 4, 64), (2, 4)),
    1: Workload(1, "short requests: R=32, P~U[256,512], n~U{1..4}, |q|~U[16,48]", 16384,
                (AttnShape("attn", 16, 4, 128, 0, ROPE),),
                GdnShape("gdn", 16, 128, 128, 4, 64), (2, 8)),
    2: Workload(2, "many questions: R=8, P~U[256,400], n=48, |q|~U[12,32], SWA W=512", 16384,
                (AttnShape("attn", 16, 4, 128, 0, ROPE), AttnShape("swa", 16, 4, 128, 512, ROPE)),
                GdnShape("gdn", 16, 128, 128, 4, 64), (2, 8)),
    3: Workload(3, "long documents: R=4, P~U[4096,6144], n~U{8..20}, |q|~U[32,64], SWA W=1024", 32768,
                (AttnShape("attn", 32, 8, 128, 0, ROPE), AttnShape("swa", 32, 8, 128, 1024, ROPE)),
                GdnShape("gdn", 32, 128, 128, 4, 64), (2, 8)),
    4: Workload(4, "wide fork + resume: P=16384, n=64, |q|~U[16,64], checkpoint m=15360", 32768,
                (AttnShape("attn", 32, 8, 128, 0, ROPE), AttnShape("swa", 32, 8, 128, 1024, ROPE)),
                GdnShape("gdn", 32, 128, 128, 4, 64), (2, 8)),
}

RESUME_M = 15360  # checkpoint position of workload 4
RESUME_NEW = 2048  # new trunk tokens of workload 4, round B
RESUME_TCAP_B = 8192


@dataclasses.dataclass
class Round:
    """One round: the descriptor plus every layer's stream-layout inputs.

    bf16 tensors are stored as uint16 bit patterns; ``f32(layer, name)``
    returns the exactly equal float32 values.
    """

    wid: int
    trunk_len: np.ndarray  # [R] total trunk length P_j (prefix included)
    n_q: np.ndarray  # [R]
    q_len: np.ndarray  # [Nq]
    prefix_len: np.ndarray  # [R] trunk tokens held outside the stream (resume)
    ckpt_pos: np.ndarray  # [R] -1 or the trunk position m of a checkpoint
    n_opt: np.ndarray  # [Nq]
    T_cap: int
    attn_shapes: tuple
    gdn_shape: GdnShape
    layers: Dict[str, Dict[str, np.ndarray]]
    w_opt: np.ndarray  # [sum O, D] uint16
    opt_off: np.ndarray  # [Nq + 1] int32
    # Rows of the trunk that live outside the stream (resume): per layer the
    # same arrays as ``layers`` but for trunk positions [0, prefix_len).
    prefix: Optional[Dict[str, Dict[str, np.ndarray]]] = None

    @property
    def R(self) -> int:
        return int(self.trunk_len.shape[0])

    @property
    def Nq(self) -> int:
        return int(self.q_len.shape[0])

    @property
    def T(self) -> int:
        return int((self.trunk_len - self.prefix_len).sum() + self.q_len.sum())

    @property
    def D(self) -> int:
        return self.gdn_shape.H * self.gdn_shape.dv

    def desc(self) -> np.ndarray:
        """Packed descriptor [R trunk_len | R n_q | Nq q_len | R prefix_len | R ckpt_pos]."""
        return np.concatenate([self.trunk_len, self.n_q, self.q_len, self.prefix_len,
                               self.ckpt_pos]).astype(np.int32)

    def f32(self, layer: str, name: str) -> np.ndarray:
        a = self.layers[layer][name]
        return bf16_to_f32(a) if a.dtype == np.uint16 else a

    def prefix_f32(self, layer: str, name: str) -> np.ndarray:
        a = self.prefix[layer][name]
        return bf16_to_f32(a) if a.dtype == np.uint16 else a

    def w_opt_f32(self) -> np.ndarray:
        return bf16_to_f32(self.w_opt)


def _sigmoid64(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x.astype(np.float64)))


def _draw_layers(rng, T: int, T_cap: int, attn_shapes, gdn: GdnShape):
    layers = {}

    def normal_bf16(shape_rows, tail):
        x = np.zeros((T_cap,) + tail, dtype=np.uint16)
        x[:shape_rows] = bf16_bits(rng.standard_normal((shape_rows,) + tail, dtype=np.float32))
        return x

    for a in attn_shapes:
        layers[a.name] = {
            "q": normal_bf16(T, (a.Hq, a.d)),
            "k": normal_bf16(T, (a.Hkv, a.d)),
            "v": normal_bf16(T, (a.Hkv, a.d)),
        }
    g = gdn
    lay = {
        "q": normal_bf16(T, (g.H, g.dk)),
        "k": normal_bf16(T, (g.H, g.dk)),
        "v": normal_bf16(T, (g.H, g.dv)),
    }
    alpha = np.zeros((T_cap, g.H), dtype=np.float32)
    eta = np.zeros((T_cap, g.H), dtype=np.float32)
    alpha[:T] = _sigmoid64(rng.normal(2.0, 0.5, size=(T, g.H))).astype(np.float32)
    eta[:T] = _sigmoid64(rng.normal(0.0, 1.0, size=(T, g.H))).astype(np.float32)
    lay["alpha"] = alpha
    lay["eta"] = eta
    layers[g.name] = lay
    return layers


def _draw_conv(rng, g: GdnShape) -> np.ndarray:
    lim = 1.0 / math.sqrt(g.K)
    # [3 (q,k,v), H, d, K]; tap K-1 multiplies the current token.
    d = max(g.dk, g.dv)
    return rng.uniform(-lim, lim, size=(3, g.H, d, g.K)).astype(np.float32)


def _draw_wopt(rng, n_opt: np.ndarray, D: int):
    total = int(n_opt.sum())
    w = bf16_bits((rng.standard_normal((total, D), dtype=np.float32) * np.float32(0.02)))
    off = np.zeros(n_opt.shape[0] + 1, dtype=np.int32)
    off[1:] = np.cumsum(n_opt)
    return w, off


def make_round(wid: int, seed: Optional[int] = None, *, trunk_len=None, n_q=None, q_len=None,
               n_opt=None, T_cap: Optional[int] = None, ckpt_pos=None) -> Round:
    """Draw one round of workload ``wid`` (seed defaults to the workload id).

    Keyword overrides replace drawn shape arrays (they are then not drawn,
    which changes the stream of later draws); used by tests for edge cases.
    """
    w = WORKLOADS[wid]
    rng = np.random.default_rng(wid if seed is None else seed)
    if wid == 0:
        P = np.array([64], dtype=np.int32)
        n = np.array([3], dtype=np.int32)
        ql = np.array([8, 12, 16], dtype=np.int32)
        no = np.array([2, 3, 4], dtype=np.int32)
    elif wid == 1:
        P = rng.integers(256, 512, size=32, endpoint=True).astype(np.int32)
        n = rng.integers(1, 4, size=32, endpoint=True).astype(np.int32)
        ql = rng.integers(16, 48, size=int(n.sum()), endpoint=True).astype(np.int32)
        no = rng.integers(2, 8, size=int(n.sum()), endpoint=True).astype(np.int32)
    elif wid == 2:
        P = rng.integers(256, 400, size=8, endpoint=True).astype(np.int32)
        n = np.full(8, 48, dtype=np.int32)
        ql = rng.integers(12, 32, size=int(n.sum()), endpoint=True).astype(np.int32)
        no = rng.integers(2, 8, size=int(n.sum()), endpoint=True).astype(np.int32)
    elif wid == 3:
        P = rng.integers(4096, 6144, size=4, endpoint=True).astype(np.int32)
        n = rng.integers(8, 20, size=4, endpoint=True).astype(np.int32)
        ql = rng.integers(32, 64, size=int(n.sum()), endpoint=True).astype(np.int32)
        no = rng.integers(2, 8, size=int(n.sum()), endpoint=True).astype(np.int32)
    elif wid == 4:
        P = np.array([16384], dtype=np.int32)
        n = np.array([64], dtype=np.int32)
        ql = rng.integers(16, 64, size=64, endpoint=True).astype(np.int32)
        no = rng.integers(2, 8, size=64, endpoint=True).astype(np.int32)
    else:
        raise ValueError(wid)
    if trunk_len is not None:
        P = np.asarray(trunk_len, dtype=np.int32)
    if n_q is not None:
        n = np.asarray(n_q, dtype=np.int32)
    if q_len is not None:
        ql = np.asarray(q_len, dtype=np.int32)
    if n_opt is not None:
        no = np.asarray(n_opt, dtype=np.int32)
    if int(n.sum()) != ql.shape[0] or ql.shape[0] != no.shape[0]:
        raise ValueError("question counts and lengths disagree")
    R = P.shape[0]
    prefix = np.zeros(R, dtype=np.int32)
    ck = np.full(R, -1, dtype=np.int32)
    if wid == 4 and ckpt_pos is None:
        ck[0] = RESUME_M
    if ckpt_pos is not None:
        ck = np.asarray(ckpt_pos, dtype=np.int32)
    cap = w.T_cap if T_cap is None else int(T_cap)
    T = int(P.sum() + ql.sum())
    if T > cap:
        raise ValueError(f"round of {T} tokens exceeds capacity {cap}")
    layers = _draw_layers(rng, T, cap, w.attn, w.gdn)
    layers[w.gdn.name]["conv_w"] = _draw_conv(rng, w.gdn)
    wo, off = _draw_wopt(rng, no, w.gdn.H * w.gdn.dv)
    rnd = Round(wid, P, n, ql, prefix, ck, no, cap, w.attn, w.gdn, layers, wo, off)
    rnd._rng = rng  # continued by make_resume_round
    return rnd


def draw_round_shapes(wid: int, copies: int, seed: int):
    """Request and question shapes of a round of workload ``wid`` with ``copies`` times
    its requests, drawn from the same distributions (trunk lengths, question counts,
    question lengths, option counts); no layer values.  Used to shard one large round
    over several GPUs."""
    rng = np.random.default_rng(seed)
    if wid == 1:
        R, Pr, nr, qr = 32, (256, 512), (1, 4), (16, 48)
    elif wid == 2:
        R, Pr, nr, qr = 8, (256, 400), (48, 48), (12, 32)
    elif wid == 3:
        R, Pr, nr, qr = 4, (4096, 6144), (8, 20), (32, 64)
    else:
        raise ValueError(wid)
    R *= copies
    P = rng.integers(Pr[0], Pr[1], size=R, endpoint=True).astype(np.int32)
    n = rng.integers(nr[0], nr[1], size=R, endpoint=True).astype(np.int32)
    ql = rng.integers(qr[0], qr[1], size=int(n.sum()), endpoint=True).astype(np.int32)
    no = rng.integers(2, 8, size=int(n.sum()), endpoint=True).astype(np.int32)
    return P, n, ql, no


def make_resume_round(round_a: Round, m: int = RESUME_M, n_new: int = RESUME_NEW,
                      n_questions: int = 64, T_cap: int = RESUME_TCAP_B) -> Round:
    """Workload 4, round B: request 0 of ``round_a`` shares its first ``m``
    trunk tokens, adds ``n_new`` fresh trunk tokens and new questions.

    The shared rows are round A's stream rows [0, m) of every layer; they are
    held outside the stream (``prefix``), as a checkpoint at ``m`` would hold
    them.  Draws continue round A's generator.
    """
    if round_a.R != 1 or round_a.prefix_len[0] != 0:
        raise ValueError("resume rounds are built from a one-request round")
    rng = round_a._rng
    w = WORKLOADS[round_a.wid] if round_a.wid in WORKLOADS else None
    ql = rng.integers(16, 64, size=n_questions, endpoint=True).astype(np.int32)
    no = rng.integers(2, 8, size=n_questions, endpoint=True).astype(np.int32)
    P = np.array([m + n_new], dtype=np.int32)
    n = np.array([n_questions], dtype=np.int32)
    prefix = np.array([m], dtype=np.int32)
    ck = np.array([-1], dtype=np.int32)
    T = int(n_new + ql.sum())
    if T > T_cap:
        raise ValueError("resume round exceeds capacity")
    layers = _draw_layers(rng, T, T_cap, round_a.attn_shapes, round_a.gdn_shape)
    g = round_a.gdn_shape
    layers[g.name]["conv_w"] = round_a.layers[g.name]["conv_w"]  # same layer weights
    wo, off = _draw_wopt(rng, no, g.H * g.dv)
    pref = {}
    for name, lay in round_a.layers.items():
        pref[name] = {k: v[:m].copy() for k, v in lay.items() if k != "conv_w"}
    rnd = Round(round_a.wid, P, n, ql, prefix, ck, no, T_cap, round_a.attn_shapes, g, layers,
                wo, off, prefix=pref)
    rnd._rng = rng
    return rnd


def custom_round(trunk_len, n_q, q_len, *, attn_shapes, gdn_shape, T_cap, seed=0, n_opt=None,
                 prefix_len=None, ckpt_pos=None) -> Round:
    """A round with explicit lengths and shapes (tests: edge cases, small sizes).

    ``prefix_len`` > 0 marks trunk tokens held outside the stream; their rows
    are drawn too (into ``prefix``) so an oracle can run the full trunk.
    """
    rng = np.random.default_rng(seed)
    P = np.asarray(trunk_len, dtype=np.int32)
    n = np.asarray(n_q, dtype=np.int32)
    ql = np.asarray(q_len, dtype=np.int32)
    R = P.shape[0]
    if int(n.sum()) != ql.shape[0] or n.shape[0] != R:
        raise ValueError("question counts do not match the question lengths")
    if n_opt is None:
        no = rng.integers(2, 8, size=ql.shape[0], endpoint=True).astype(np.int32)
    else:
        no = np.asarray(n_opt, dtype=np.int32)
    pl = np.zeros(R, dtype=np.int32) if prefix_len is None else np.asarray(prefix_len, dtype=np.int32)
    ck = np.full(R, -1, dtype=np.int32) if ckpt_pos is None else np.asarray(ckpt_pos, dtype=np.int32)
    T = int((P - pl).sum() + ql.sum())
    if T > T_cap:
        raise ValueError("round exceeds capacity")
    layers = _draw_layers(rng, T, T_cap, attn_shapes, gdn_shape)
    layers[gdn_shape.name]["conv_w"] = _draw_conv(rng, gdn_shape)
    wo, off = _draw_wopt(rng, no, gdn_shape.H * gdn_shape.dv)
    pref = None
    if int(pl.sum()) > 0:
        # Prefix rows are stored request after request: rows of request j at
        # [sum(pl[:j]), sum(pl[:j+1])).
        Tp = int(pl.sum())
        pl_layers = _draw_layers(rng, Tp, Tp, attn_shapes, gdn_shape)
        pref = {name: dict(lay) for name, lay in pl_layers.items()}
    rnd = Round(-1, P, n, ql, pl, ck, no, T_cap, tuple(attn_shapes), gdn_shape, layers, wo, off,
                prefix=pref)
    rnd._rng = rng
    return rnd


def readout_block_weights(D: int, F: int, seed: int = 7):
    """Seeded weights of the last layer's pointwise block (selective readout):
    norm gains g1, g2 = 1 + N(0, 0.1^2) (float32); W_gate, W_up [F, D] ~ N(0, 1/D)
    and W_down [D, F] ~ N(0, 1/F), rounded to bfloat16 (uint16 bit patterns)."""
    rng = np.random.default_rng(seed)
    g1 = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    g2 = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wg = bf16_bits(rng.standard_normal((F, D), dtype=np.float32) * np.float32(1.0 / math.sqrt(D)))
    wu = bf16_bits(rng.standard_normal((F, D), dtype=np.float32) * np.float32(1.0 / math.sqrt(D)))
    wd = bf16_bits(rng.standard_normal((D, F), dtype=np.float32) * np.float32(1.0 / math.sqrt(F)))
    return {"g1": g1, "g2": g2, "w_gate": wg, "w_up": wu, "w_down": wd}


@dataclasses.dataclass
class TreeRound:
    """A forest of token trees (requests whose branches fork again).

    Node k has ``parent[k]`` (-1 for a root) and ``node_len[k]`` tokens of its
    own, stored node after node in ``layers`` (rows [node_start[k],
    node_start[k] + node_len[k])).  A node without children is a leaf: a
    question, with at least one token and ``n_opt[k]`` options (option weights
    ``w_opt``, CSR ``opt_off`` over the leaves in node order).  Every node's
    sequence is its ancestors' tokens followed by its own.
    """

    parent: np.ndarray  # [N] int32
    node_len: np.ndarray  # [N] int32
    n_opt: np.ndarray  # [N] int32, 0 for internal nodes
    attn_shapes: tuple
    gdn_shape: GdnShape
    layers: Dict[str, Dict[str, np.ndarray]]
    w_opt: np.ndarray  # [sum O, D] uint16
    opt_off: np.ndarray  # [leaves + 1] int32

    @property
    def N(self) -> int:
        return int(self.parent.shape[0])

    @property
    def node_start(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.node_len)[:-1]]).astype(np.int64)

    def children(self, k: int) -> List[int]:
        return [c for c in range(self.N) if int(self.parent[c]) == k]

    def is_leaf(self, k: int) -> bool:
        return not any(int(p) == k for p in self.parent)

    def leaves(self) -> List[int]:
        return [k for k in range(self.N) if self.is_leaf(k)]

    def depth(self, k: int) -> int:
        d = 0
        while int(self.parent[k]) >= 0:
            k = int(self.parent[k])
            d += 1
        return d

    def ancestors(self, k: int) -> List[int]:
        """Ancestors of node k, root first."""
        out = []
        while int(self.parent[k]) >= 0:
            k = int(self.parent[k])
            out.append(k)
        return out[::-1]


def request_forest(n_req: int, level_len, fanout):
    """Parent and length arrays of n_req identical request trees: a trunk of level_len[0]
    tokens; every node of depth d < len(fanout) has fanout[d] children of level_len[d + 1]
    tokens each.  Nodes are listed tree after tree, depth first (parents before children)."""
    parent, node_len = [], []

    def add(p, d):
        k = len(parent)
        parent.append(p)
        node_len.append(int(level_len[d]))
        if d < len(fanout):
            for _ in range(fanout[d]):
                add(k, d + 1)

    for _ in range(n_req):
        add(-1, 0)
    return np.array(parent, np.int32), np.array(node_len, np.int32)


def make_tree_round(parent, node_len, *, attn_shapes, gdn_shape, seed=0, n_opt=None) -> TreeRound:
    """A forest with explicit structure; rows, gates, conv and option weights drawn
    as for a round (same draw order: layers, conv weights, option weights)."""
    parent = np.asarray(parent, dtype=np.int32)
    node_len = np.asarray(node_len, dtype=np.int32)
    N = parent.shape[0]
    for k in range(N):
        if not (-1 <= parent[k] < k):
            raise ValueError("parents must precede their children")
    rng = np.random.default_rng(seed)
    leaf = np.array([not np.any(parent == k) for k in range(N)])
    if np.any(node_len[leaf] < 1):
        raise ValueError("a leaf (question) needs at least one token")
    if n_opt is None:
        n_opt = np.where(leaf, rng.integers(2, 8, size=N, endpoint=True), 0).astype(np.int32)
    n_opt = np.asarray(n_opt, dtype=np.int32)
    T = int(node_len.sum())
    layers = _draw_layers(rng, T, max(T, 1), attn_shapes, gdn_shape)
    layers[gdn_shape.name]["conv_w"] = _draw_conv(rng, gdn_shape)
    wo, off = _draw_wopt(rng, n_opt[leaf], gdn_shape.H * gdn_shape.dv)
    return TreeRound(parent, node_len, n_opt, tuple(attn_shapes), gdn_shape, layers, wo, off)
