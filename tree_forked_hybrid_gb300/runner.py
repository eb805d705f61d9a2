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
        n = 2  # metadata: tables + tokens
        for a in self.rnd.attn_shapes:
            # rotary tables + keys (+ queries for the warp-MMA kernel) + attention
            n += (4 if self.flags & F.FORK_WARP_MMA else 3) if a.rope_theta else 1
        return n + 3  # gdn trunk, gdn branches, readout


class GraphRound:
    """The whole layer of one round captured as a single CUDA graph.

    Launch shapes depend only on the capacities and the shape arguments, and
    no call reads the device back, so ``DeviceRound.run`` captures as is: the
    metadata build reads the descriptor from device memory, and every later
    kernel takes its segments from the metadata.  A new round with the same
    request and question counts (other lengths, other values) replays the
    graph after ``load`` has copied its descriptor and inputs into the
    captured buffers.  The onedev summary ("어떻게 쓰나") captures one graph
    per capacity bucket the same way.
    """

    def __init__(self, dr: DeviceRound):
        self.dr = dr
        side = torch.cuda.Stream(device=dr.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # first calls outside capture (function attributes, entry points)
            dr.run()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            dr.run()
        torch.cuda.synchronize()

    def load(self, rnd: Round):
        """Copy another round's descriptor and inputs into the captured buffers."""
        dr = self.dr
        if rnd.R != dr.rnd.R or rnd.Nq != dr.rnd.Nq or rnd.T_cap != dr.rnd.T_cap:
            raise ValueError("the graph was captured for another request/question count or capacity")
        if int(rnd.opt_off[-1]) > dr.p.numel() or rnd.w_opt.shape[0] > dr.w_opt.shape[0]:
            raise ValueError("more options than the captured buffers hold")
        if int(rnd.prefix_len.sum()) != dr.prefix_rows:
            raise ValueError("the graph was captured for another number of prefix rows")
        dr.desc.copy_(torch.from_numpy(rnd.desc()))
        for name, lay in rnd.layers.items():
            for k, v in lay.items():
                src = _bf16(v, "cpu") if v.dtype == np.uint16 else _f32(v, "cpu")
                dr.inputs[name][k].copy_(src)
        dr.w_opt[:rnd.w_opt.shape[0]].copy_(_bf16(rnd.w_opt, "cpu"))
        dr.opt_off.copy_(torch.from_numpy(rnd.opt_off.astype(np.int32)))
        dr.rnd = rnd

    def replay(self):
        self.graph.replay()


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
