"""One round of the ForkAttention layer on the device.

Holds a round's inputs in device memory, the output and workspace buffers,
and issues the C-ABI calls in order: fork_build_meta, fork_attn for every
attention layer, fork_gdn_trunk, fork_gdn_branches, fork_readout.  All of it
is stream-ordered with no host synchronisation.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np
import torch

from . import fork as F
from .workloads import Round


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def _f32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


class DeviceRound:
    """Device-resident inputs and outputs of one round.

    ``resume_from``: for a round whose trunks start from a checkpoint, the
    DeviceRound of the round that produced it (its S_ckpt / conv_ckpt are the
    initial state and conv window; the prefix K/V rows come from this round's
    ``prefix`` arrays, i.e. the earlier round's attention inputs).
    ``init_state`` / ``init_conv``: the initial states [R, H, d, d] and conv
    windows [R, K-1, 3, H, d] of the resumed trunks, given directly instead.
    """

    def __init__(self, rnd: Round, device="cuda", max_req: Optional[int] = None,
                 max_q: Optional[int] = None, resume_from: Optional["DeviceRound"] = None,
                 flags: int = 0, init_state: Optional[torch.Tensor] = None,
                 init_conv: Optional[torch.Tensor] = None):
        self.rnd = rnd
        self.device = device
        self.flags = flags
        a0 = rnd.attn_shapes[0]
        G = a0.Hq // a0.Hkv
        for a in rnd.attn_shapes:
            if a.Hq // a.Hkv != G:
                raise ValueError("attention layers of one round share the GQA group size")
        # a work item of the tcgen05 attention kernel is two 128-row query tiles
        # (tokens x grouped heads) that share every key tile; the warp-MMA kernel takes one
        self.tile_tokens = (128 if flags & F.FORK_WARP_MMA else 256) // G
        self.max_req = max_req or rnd.R
        self.max_q = rnd.Nq if max_q is None else max_q
        self.meta = F.Meta(rnd.T_cap, self.max_req, self.max_q, self.tile_tokens, device)
        self.desc = torch.from_numpy(rnd.desc()).to(device)
        self.inputs: Dict[str, Dict[str, torch.Tensor]] = {}
        for name, lay in rnd.layers.items():
            self.inputs[name] = {k: (_bf16(v, device) if v.dtype == np.uint16 else _f32(v, device))
                                 for k, v in lay.items()}
        # at least one row, so that a round without questions still passes valid pointers
        self.w_opt = _bf16(rnd.w_opt if rnd.w_opt.shape[0] else np.zeros((1, rnd.D), np.uint16), device)
        self.opt_off = torch.from_numpy(rnd.opt_off.astype(np.int32)).to(device)
        self.prefix_rows = int(rnd.prefix_len.sum())
        self.prefix = {}
        if self.prefix_rows > 0:
            for a in rnd.attn_shapes:
                self.prefix[a.name] = (_bf16(rnd.prefix[a.name]["k"], device),
                                       _bf16(rnd.prefix[a.name]["v"], device))
        # outputs
        T_cap = rnd.T_cap
        self.attn_out = {a.name: torch.zeros((T_cap, a.Hq, a.d), dtype=torch.bfloat16, device=device)
                         for a in rnd.attn_shapes}
        self.attn_ws = {}
        for a in rnd.attn_shapes:
            nb = F.fork_attn_workspace_bytes(T_cap, self.prefix_rows, a.Hq, a.Hkv, a.d, a.rope_theta, flags)
            self.attn_ws[a.name] = torch.empty(max(nb, 16), dtype=torch.uint8, device=device) if nb else None
        g = rnd.gdn_shape
        if g.dk != g.dv:
            raise ValueError("the GDN kernels take d_k == d_v")
        R, H, d, K = self.max_req, g.H, g.dk, g.K
        self.gdn_out = torch.zeros((T_cap, H, d), dtype=torch.bfloat16, device=device)
        self.S_P = torch.zeros((R, H, d, d), dtype=torch.float32, device=device)
        self.conv_win = torch.zeros((R, K - 1, 3, H, d), dtype=torch.bfloat16, device=device)
        self.has_ckpt = bool((rnd.ckpt_pos >= 0).any())
        self.S_ckpt = torch.zeros_like(self.S_P) if self.has_ckpt else None
        self.conv_ckpt = torch.zeros_like(self.conv_win) if self.has_ckpt else None
        self.init_state = self.init_conv = None
        if init_state is not None:
            self.init_state, self.init_conv = init_state.contiguous(), init_conv.contiguous()
        elif self.prefix_rows > 0:
            if resume_from is None or resume_from.S_ckpt is None:
                raise ValueError("a round with prefix rows needs the checkpoint it resumes from")
            self.init_state = resume_from.S_ckpt
            self.init_conv = resume_from.conv_ckpt
        self.p = torch.zeros(max(int(rnd.opt_off[-1]), 1), dtype=torch.float32, device=device)

    # ------------------------------------------------------------------
    def step_meta(self, stream=None):
        F.fork_build_meta(self.meta, self.desc, self.rnd.R, self.rnd.Nq, self.flags, stream)

    def step_attn(self, name: str, stream=None):
        a = [x for x in self.rnd.attn_shapes if x.name == name][0]
        inp = self.inputs[name]
        pk, pv = self.prefix.get(name, (None, None))
        F.fork_attn(self.meta, inp["q"], inp["k"], inp["v"], self.attn_out[name], a.Hq, a.Hkv, a.d,
                    a.window, a.rope_theta, 1.0 / math.sqrt(a.d), pk, pv, self.attn_ws[name],
                    self.flags, stream)

    def step_gdn_trunk(self, stream=None):
        g = self.rnd.gdn_shape
        inp = self.inputs[g.name]
        F.fork_gdn_trunk(self.meta, inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"], inp["conv_w"],
                         g.H, g.dk, g.K, g.chunk, self.S_P, self.conv_win, self.gdn_out,
                         init_state=self.init_state, init_conv=self.init_conv, S_ckpt=self.S_ckpt,
                         conv_ckpt=self.conv_ckpt, flags=self.flags, stream=stream)

    def step_gdn_branches(self, stream=None):
        g = self.rnd.gdn_shape
        inp = self.inputs[g.name]
        F.fork_gdn_branches(self.meta, inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                            inp["conv_w"], g.H, g.dk, g.K, g.chunk, self.S_P, self.conv_win,
                            self.gdn_out, flags=self.flags, stream=stream)

    def step_readout(self, stream=None):
        g = self.rnd.gdn_shape
        F.fork_readout(self.meta, self.gdn_out, g.H * g.dv, self.w_opt, self.opt_off, self.p, self.flags,
                       stream)

    def run(self, stream=None):
        """The whole layer: metadata, attention layers, GDN (two calls), readout."""
        self.step_meta(stream)
        for a in self.rnd.attn_shapes:
            self.step_attn(a.name, stream)
        self.step_gdn_trunk(stream)
        self.step_gdn_branches(stream)
        self.step_readout(stream)

    def status(self) -> int:
        return F.fork_read_status(self.meta)

    def launches_per_round(self) -> int:
        n = 3 if self.flags & F.FORK_CHECKS else 2  # metadata: tables + tokens (+ checks)
        for a in self.rnd.attn_shapes:
            if self.flags & F.FORK_WARP_MMA:
                n += 4 if a.rope_theta else 1  # rotary tables + keys + queries + attention
            else:
                n += 4 if a.rope_theta else 2  # rotary tables + keys, fp16 values, attention
        return n + 3  # gdn trunk, gdn branches, readout


class CapacityRound:
    """Device buffers of the whole layer at fixed capacities, for rounds of one set of
    layer shapes: T_cap stream tokens, max_req requests, max_q questions, max_opts
    options.  The round's counts live in a fixed-capacity device descriptor
    (``fork_build_meta_dev``), so every call depends only on the capacities: the
    layer can be captured once as a CUDA graph and replayed for any round that fits
    (after ``load``).  Rounds with prefix rows (resumed trunks) do not fit."""

    def __init__(self, attn_shapes, gdn_shape, T_cap: int, max_req: int, max_q: int, max_opts: int,
                 device="cuda", flags: int = 0):
        self.attn_shapes, self.gdn_shape = tuple(attn_shapes), gdn_shape
        self.T_cap, self.max_req, self.max_q, self.max_opts = T_cap, max_req, max_q, max_opts
        self.device, self.flags = device, flags
        G = self.attn_shapes[0].Hq // self.attn_shapes[0].Hkv
        self.tile_tokens = (128 if flags & F.FORK_WARP_MMA else 256) // G
        self.meta = F.Meta(T_cap, max_req, max_q, self.tile_tokens, device)
        self.desc = torch.zeros(F.fork_desc_capacity_words(max_req, max_q), dtype=torch.int32, device=device)
        bf = dict(dtype=torch.bfloat16, device=device)
        self.inputs: Dict[str, Dict[str, torch.Tensor]] = {}
        self.attn_out, self.attn_ws = {}, {}
        for a in self.attn_shapes:
            self.inputs[a.name] = {"q": torch.zeros((T_cap, a.Hq, a.d), **bf),
                                   "k": torch.zeros((T_cap, a.Hkv, a.d), **bf),
                                   "v": torch.zeros((T_cap, a.Hkv, a.d), **bf)}
            self.attn_out[a.name] = torch.zeros((T_cap, a.Hq, a.d), **bf)
            nb = F.fork_attn_workspace_bytes(T_cap, 0, a.Hq, a.Hkv, a.d, a.rope_theta, flags)
            self.attn_ws[a.name] = torch.empty(max(nb, 16), dtype=torch.uint8, device=device) if nb else None
        g = gdn_shape
        f32 = dict(dtype=torch.float32, device=device)
        self.inputs[g.name] = {"q": torch.zeros((T_cap, g.H, g.dk), **bf), "k": torch.zeros((T_cap, g.H, g.dk), **bf),
                               "v": torch.zeros((T_cap, g.H, g.dv), **bf), "alpha": torch.ones((T_cap, g.H), **f32),
                               "eta": torch.zeros((T_cap, g.H), **f32),
                               "conv_w": torch.zeros((3, g.H, g.dk, g.K), **f32)}
        self.gdn_out = torch.zeros((T_cap, g.H, g.dv), **bf)
        self.S_P = torch.zeros((max_req, g.H, g.dv, g.dk), **f32)
        self.conv_win = torch.zeros((max_req, g.K - 1, 3, g.H, g.dk), **bf)
        D = g.H * g.dv
        self.w_opt = torch.zeros((max(max_opts, 1), D), **bf)
        self.opt_off = torch.zeros(max_q + 1, dtype=torch.int32, device=device)
        self.p = torch.zeros(max(max_opts, 1), **f32)
        self.rnd: Optional[Round] = None

    def fits(self, rnd: Round) -> bool:
        return (rnd.T <= self.T_cap and rnd.R <= self.max_req and rnd.Nq <= self.max_q and
                int(rnd.opt_off[-1]) <= self.max_opts and int(rnd.prefix_len.sum()) == 0 and
                tuple(rnd.attn_shapes) == self.attn_shapes and rnd.gdn_shape == self.gdn_shape)

    def load(self, rnd: Round):
        """Copy a round's descriptor, inputs and option weights into the buffers."""
        if not self.fits(rnd):
            raise ValueError("the round does not fit these capacities")
        R, Nq, T = rnd.R, rnd.Nq, rnd.T
        d = np.zeros(self.desc.shape[0], dtype=np.int32)
        mr, mq = self.max_req, self.max_q
        d[0], d[1] = R, Nq
        d[2:2 + R] = rnd.trunk_len
        d[2 + mr:2 + mr + R] = rnd.n_q
        d[2 + 2 * mr:2 + 2 * mr + Nq] = rnd.q_len
        d[2 + 2 * mr + mq:2 + 2 * mr + mq + R] = rnd.prefix_len
        d[2 + 3 * mr + mq:2 + 3 * mr + mq + R] = rnd.ckpt_pos
        self.desc.copy_(torch.from_numpy(d))
        for name, lay in rnd.layers.items():
            for k, v in lay.items():
                src = v if k == "conv_w" else v[:T]
                t = _bf16(src, "cpu") if v.dtype == np.uint16 else _f32(src, "cpu")
                self.inputs[name][k][:t.shape[0]].copy_(t)
        nopt = int(rnd.opt_off[-1])
        if nopt:
            self.w_opt[:nopt].copy_(_bf16(rnd.w_opt, "cpu"))
        off = np.full(self.max_q + 1, nopt, dtype=np.int32)
        off[:Nq + 1] = rnd.opt_off
        self.opt_off.copy_(torch.from_numpy(off))
        self.rnd = rnd

    def run(self, stream=None):
        """The whole layer; nothing here depends on the loaded round's counts."""
        F.fork_build_meta_dev(self.meta, self.desc, self.flags, stream)
        for a in self.attn_shapes:
            inp = self.inputs[a.name]
            F.fork_attn(self.meta, inp["q"], inp["k"], inp["v"], self.attn_out[a.name], a.Hq, a.Hkv, a.d,
                        a.window, a.rope_theta, 1.0 / math.sqrt(a.d), None, None, self.attn_ws[a.name],
                        self.flags, stream)
        g = self.gdn_shape
        inp = self.inputs[g.name]
        F.fork_gdn_trunk(self.meta, inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"], inp["conv_w"],
                         g.H, g.dk, g.K, g.chunk, self.S_P, self.conv_win, self.gdn_out, flags=self.flags,
                         stream=stream)
        F.fork_gdn_branches(self.meta, inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                            inp["conv_w"], g.H, g.dk, g.K, g.chunk, self.S_P, self.conv_win, self.gdn_out,
                            flags=self.flags, stream=stream)
        F.fork_readout(self.meta, self.gdn_out, g.H * g.dv, self.w_opt, self.opt_off, self.p, self.flags,
                       stream)

    def status(self) -> int:
        return F.fork_read_status(self.meta)


class GraphPool:
    """The whole layer captured once per capacity bucket, replayed for any round.

    The onedev summary ("어떻게 쓰나") and the rainbus summary ("方法步骤详情" step 3,
    "局限与改进") capture one flat graph per stream capacity and replay the smallest
    that holds the round; a round over the largest capacity is split at request
    boundaries; a single request too long for every bucket runs without a graph.
    ``run`` does exactly that: the smallest bucket whose capacities hold the round
    (tokens, requests, questions, options); else ``shard.split_to_fit`` groups of
    requests, each replayed in the smallest bucket that holds it; requests longer
    than the largest bucket (and rounds with prefix rows) run eagerly through a
    DeviceRound of their own.  Results come back in the round's own layout.
    """

    def __init__(self, attn_shapes, gdn_shape, buckets=(4096, 8192, 16384, 32768), max_req: int = 64,
                 max_q: int = 512, max_opts: int = 4096, device="cuda", flags: int = 0):
        self.device, self.flags = device, flags
        self.buckets = []
        for T_cap in sorted(buckets):
            cr = CapacityRound(attn_shapes, gdn_shape, T_cap, max_req, max_q, max_opts, device, flags)
            side = torch.cuda.Stream(device=device)
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # first calls outside capture (function attributes, entry points)
                cr.run()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="thread_local"):
                cr.run()
            torch.cuda.synchronize()
            self.buckets.append((cr, graph))
        self.last_plan = []

    def bucket_for(self, rnd: Round):
        for cr, graph in self.buckets:
            if cr.fits(rnd):
                return cr, graph
        return None

    def run(self, rnd: Round, outputs: bool = True):
        """Run a round; returns {"p": probabilities (host), and with outputs=True
        "attn": {layer: [T, Hq, d]}, "gdn": [T, H, d] (host float32)} in the round's layout."""
        from . import shard as S
        plan = []
        b = self.bucket_for(rnd)
        if b is not None:
            plan.append(("graph", b, rnd, np.arange(rnd.T), list(range(rnd.Nq))))
        else:
            groups, big = S.split_to_fit(rnd, self.buckets[-1][0].T_cap)
            if int(rnd.prefix_len.sum()) > 0:
                groups, big = [], list(range(rnd.R))
            for g in groups:
                sub, qids = S.shard_round(rnd, g, T_cap=rnd.T_cap)
                rows, _ = S.shard_rows(rnd, g)
                bb = self.bucket_for(sub)
                if bb is None:
                    big.extend(g)
                    continue
                plan.append(("graph", bb, sub, rows, qids))
            for j in sorted(big):
                rows, qids = S.shard_rows(rnd, [j])
                cap = int(rows.shape[0])
                sub, _ = S.shard_round(rnd, [j], T_cap=max(cap, 1))
                plan.append(("eager", None, sub, rows, qids))
        self.last_plan = [(kind, (b[0].T_cap if b else sub.T_cap), sub.R, sub.Nq) for kind, b, sub, _, _ in plan]
        res = {"p": np.zeros(int(rnd.opt_off[-1]), np.float32)}
        if outputs:
            res["attn"] = {a.name: np.zeros((rnd.T, a.Hq, a.d), np.float32) for a in rnd.attn_shapes}
            g = rnd.gdn_shape
            res["gdn"] = np.zeros((rnd.T, g.H, g.dv), np.float32)
        parts = []
        status = 0
        for kind, b, sub, rows, qids in plan:
            if kind == "graph":
                cr, graph = b
                cr.load(sub)
                graph.replay()
                src = cr
            else:
                src = DeviceRound(sub, device=self.device, flags=self.flags)
                src.run()
            torch.cuda.synchronize()
            status |= src.status()
            parts.append((qids, src.p[:int(sub.opt_off[-1])].cpu().numpy()))
            if outputs:
                n = sub.T
                for a in rnd.attn_shapes:
                    res["attn"][a.name][rows] = src.attn_out[a.name][:n].float().cpu().numpy()
                res["gdn"][rows] = src.gdn_out[:n].float().cpu().numpy()
        if status:
            raise RuntimeError(f"device status {status:#x}")
        res["p"] = S.scatter_probabilities(rnd, parts) if rnd.Nq else res["p"]
        return res


class TreeRunner:
    """A forest of token trees (branches that fork again) on the device, one
    round per depth (``tree.decompose``): a level's trunks start from their
    parent requests' S_P and conv windows of the previous level, gathered on
    the device; their prefix K/V rows are the ancestors' rows."""

    def __init__(self, tree, device="cuda", flags: int = 0):
        from . import tree as TR
        self.tree = tree
        self.device = device
        self.flags = flags
        self.levels = TR.decompose(tree)
        self.rounds = []

    def run(self):
        self.rounds = []
        prev = None
        for lv in self.levels:
            r = lv.round
            init_state = init_conv = None
            if int(r.prefix_len.sum()) > 0:
                idx = torch.tensor([max(j, 0) for j in lv.parent_request], dtype=torch.long, device=self.device)
                init_state = prev.S_P.index_select(0, idx)
                init_conv = prev.conv_win.index_select(0, idx)
            dr = DeviceRound(r, device=self.device, flags=self.flags, init_state=init_state, init_conv=init_conv)
            dr.run()
            self.rounds.append(dr)
            prev = dr

    def status(self) -> int:
        st = 0
        for dr in self.rounds:
            st |= dr.status()
        return st

    def outputs(self):
        """Attention and GDN rows in tree layout (node after node) and the leaves' probabilities (host)."""
        from . import tree as TR
        t = self.tree
        T = int(t.node_len.sum())
        start = t.node_start
        attn = {a.name: np.zeros((T, a.Hq, a.d), np.float32) for a in t.attn_shapes}
        g = t.gdn_shape
        gdn = np.zeros((T, g.H, g.dv), np.float32)
        p = np.zeros(int(t.opt_off[-1]), np.float32)
        leaf_index = {k: i for i, k in enumerate(t.leaves())}
        for lv, dr in zip(self.levels, self.rounds):
            a_out = {n: o.float().cpu().numpy() for n, o in dr.attn_out.items()}
            g_out = dr.gdn_out.float().cpu().numpy()
            pp = dr.p.cpu().numpy()
            for k, rows in TR.node_rows(lv, t):
                for n in a_out:
                    attn[n][start[k]:start[k] + rows.shape[0]] = a_out[n][rows]
                gdn[start[k]:start[k] + rows.shape[0]] = g_out[rows]
            for i, k in enumerate(lv.question_nodes):
                li = leaf_index[k]
                p[t.opt_off[li]:t.opt_off[li + 1]] = pp[lv.round.opt_off[i]:lv.round.opt_off[i + 1]]
        return attn, gdn, p


class ForestRound:
    """A forest of token trees as ONE round of one flat stream (rainbus summary "未来方向"
    (2): a draft-token tree has the shape of the request tree and runs in the same
    stream; DFlash-TfM summary "GDN을 위한 롤백 없는 트리 검증": the tree in topological
    order).  The rows stay where the tree stores them (node after node); the metadata
    (``fork_build_forest_meta``) gives every node its ancestors' rows and its parent's
    state index.  Each attention layer is one ``fork_attn`` call (FORK_FOREST): a node's
    queries read its ancestors' keys in place.  The recurrence runs one
    ``fork_gdn_forest`` call per depth: a node starts from its parent's end state and
    conv window (read by index) and leaves its own in ``node_state`` / ``node_conv``
    at its state index.  The leaves are the readout's questions.  Nothing is copied
    between nodes."""

    def __init__(self, tree, device="cuda", flags: int = 0, T_cap: Optional[int] = None):
        self.tree = tree
        self.device = device
        self.flags = flags
        a0 = tree.attn_shapes[0]
        G = a0.Hq // a0.Hkv
        for a in tree.attn_shapes:
            if a.Hq // a.Hkv != G:
                raise ValueError("attention layers of one forest share the GQA group size")
        T = int(tree.node_len.sum())
        self.T = T
        self.T_cap = T_cap or max(T, 1)
        n_leaves = len(tree.leaves())
        self.meta = F.Meta(self.T_cap, tree.N, max(n_leaves, 1), 256 // G, device)
        self.plan: Optional[F.ForestPlan] = None
        bf = dict(dtype=torch.bfloat16, device=device)
        self.inputs: Dict[str, Dict[str, torch.Tensor]] = {}
        for name, lay in tree.layers.items():
            self.inputs[name] = {}
            for k, v in lay.items():
                if k == "conv_w":
                    self.inputs[name][k] = _f32(v, device)
                    continue
                rows = np.zeros((self.T_cap,) + v.shape[1:], dtype=v.dtype)
                n = min(T, v.shape[0])
                rows[:n] = v[:n]
                self.inputs[name][k] = _bf16(rows, device) if v.dtype == np.uint16 else _f32(rows, device)
        self.attn_out = {a.name: torch.zeros((self.T_cap, a.Hq, a.d), **bf) for a in tree.attn_shapes}
        self.attn_ws = {}
        for a in tree.attn_shapes:
            nb = F.fork_attn_workspace_bytes(self.T_cap, 0, a.Hq, a.Hkv, a.d, a.rope_theta, flags)
            self.attn_ws[a.name] = torch.empty(max(nb, 16), dtype=torch.uint8, device=device) if nb else None
        g = tree.gdn_shape
        self.gdn_out = torch.zeros((self.T_cap, g.H, g.dv), **bf)
        self.node_state = torch.zeros((tree.N, g.H, g.dv, g.dk), dtype=torch.float32, device=device)
        self.node_conv = torch.zeros((tree.N, g.K - 1, 3, g.H, g.dk), **bf)
        D = g.H * g.dv
        self.w_opt = _bf16(tree.w_opt if tree.w_opt.shape[0] else np.zeros((1, D), np.uint16), device)
        self.opt_off = torch.from_numpy(tree.opt_off.astype(np.int32)).to(device)
        self.p = torch.zeros(max(int(tree.opt_off[-1]), 1), dtype=torch.float32, device=device)

    def build_meta(self, stream=None):
        """Plan the forest on the host and copy its metadata to the device."""
        self.plan = F.fork_build_forest_meta(self.meta, self.tree.parent, self.tree.node_len, stream)

    def launches_per_run(self) -> int:
        """Kernels of ``run`` (the metadata is a copy, not a kernel)."""
        n = sum(4 if a.rope_theta else 2 for a in self.tree.attn_shapes)  # rotary tables + keys, fp16 values, attention
        return n + self.plan.levels + 1  # one recurrence launch per depth, readout

    def run(self, stream=None, meta: bool = True):
        """The whole layer; ``meta=False`` reuses the metadata of an earlier run."""
        t = self.tree
        if meta or self.plan is None:
            self.build_meta(stream)
        for a in t.attn_shapes:
            inp = self.inputs[a.name]
            F.fork_attn(self.meta, inp["q"], inp["k"], inp["v"], self.attn_out[a.name], a.Hq, a.Hkv, a.d,
                        a.window, a.rope_theta, 1.0 / math.sqrt(a.d), None, None, self.attn_ws[a.name],
                        self.flags | F.FORK_FOREST, stream)
        g = t.gdn_shape
        inp = self.inputs[g.name]
        lf = self.plan.level_first
        for lv in range(self.plan.levels):
            F.fork_gdn_forest(self.meta, int(lf[lv]), int(lf[lv + 1] - lf[lv]), inp["q"], inp["k"], inp["v"],
                              inp["alpha"], inp["eta"], inp["conv_w"], g.H, g.dk, g.K, g.chunk, self.node_state,
                              self.node_conv, self.gdn_out, self.flags, stream)
        F.fork_readout(self.meta, self.gdn_out, g.H * g.dv, self.w_opt, self.opt_off, self.p, self.flags, stream)

    def status(self) -> int:
        return F.fork_read_status(self.meta)

    def outputs(self):
        """Attention and GDN rows (node after node), the leaves' probabilities and every
        node's end state in node order (host float32)."""
        T = self.T
        attn = {n: o[:T].float().cpu().numpy() for n, o in self.attn_out.items()}
        gdn = self.gdn_out[:T].float().cpu().numpy()
        p = self.p[:int(self.tree.opt_off[-1])].cpu().numpy()
        idx = torch.from_numpy(self.plan.state_index).to(self.device)
        S_end = self.node_state.index_select(0, idx).cpu().numpy()
        return attn, gdn, p, S_end
