"""Composition invariance: a question's output bits do not depend on the round it is in.

The Flide pages offer an optional mode that returns identical bits for a
request under any load (onedev summary, "어떻게 쓰나", end).  Every kernel here
computes each output from segment-aligned query tiles, range-aligned key tiles
and segment-aligned GDN chunks in a fixed order, so the same question placed in
different rounds (other requests, other siblings, other stream offsets, other
T_cap buckets) must give the same bits, with FORK_DETERMINISTIC set or not.
"""
import numpy as np
import pytest

from oracle import forkattn as orc
from tests.gpu_util import require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

A = wl.AttnShape("attn", 16, 4, 128, 0, 10000.0)
S = wl.AttnShape("swa", 16, 4, 128, 96, 10000.0)
G = wl.GdnShape("gdn", 16, 128, 128, 4, 64)
P_T, L_Q = 300, 37  # the target request's trunk and question lengths

# (trunks, questions per request, question lengths, target request, target question index in round, T_cap)
COMPOSITIONS = [
    ([P_T], [3], [20, L_Q, 15], 0, 1, 2048),
    ([150, P_T], [2, 4], [11, 30, 9, 25, L_Q, 12], 1, 4, 4096),
    ([P_T, 77, 500], [1, 3, 2], [L_Q, 5, 64, 33, 40, 2], 0, 0, 8192),
]


def _rows(m, seg):
    st, L = int(m["seg_start"][seg]), int(m["seg_len"][seg])
    return slice(st, st + L)


def _build(comp, src, seed):
    P, n, ql, tj, tq, cap = comp
    rnd = wl.custom_round(P, n, ql, attn_shapes=(A, S), gdn_shape=G, T_cap=cap, seed=seed,
                          n_opt=[4] * len(ql))
    m = orc.meta_ref(rnd.desc(), rnd.R, rnd.Nq, cap, 32)
    if src is not None:
        (ref, rm, rtj, rtq) = src
        for name, lay in rnd.layers.items():
            for f, arr in lay.items():
                if f == "conv_w":
                    arr[...] = ref.layers[name][f]
                    continue
                arr[_rows(m, tj)] = ref.layers[name][f][_rows(rm, rtj)]
                arr[_rows(m, rnd.R + tq)] = ref.layers[name][f][_rows(rm, ref.R + rtq)]
    return rnd, m


@pytest.mark.parametrize("flags", [0, 1])
def test_question_bits_do_not_depend_on_round_composition(flags):
    torch = require_gpu()
    from tree_forked_hybrid_gb300.runner import DeviceRound
    ref, rm = _build(COMPOSITIONS[0], None, 1)
    src = (ref, rm, COMPOSITIONS[0][3], COMPOSITIONS[0][4])
    outs = []
    for i, comp in enumerate(COMPOSITIONS):
        rnd, m = (ref, rm) if i == 0 else _build(comp, src, 10 + i)
        tj, tq = comp[3], comp[4]
        if i > 0:
            # the target question's option rows (same count and weights in every round)
            a, ra = int(rnd.opt_off[tq]), int(ref.opt_off[src[3]])
            rnd.w_opt[a:a + 4] = ref.w_opt[ra:ra + 4]
        dr = DeviceRound(rnd, flags=flags)
        dr.run()
        torch.cuda.synchronize()
        assert dr.status() == 0
        q_rows, t_rows = _rows(m, rnd.R + tq), _rows(m, tj)
        rec = {name: o[q_rows].cpu().view(torch.int16).numpy().copy() for name, o in dr.attn_out.items()}
        rec.update({name + "_trunk": o[t_rows].cpu().view(torch.int16).numpy().copy()
                    for name, o in dr.attn_out.items()})
        rec["gdn"] = dr.gdn_out[q_rows].cpu().view(torch.int16).numpy().copy()
        rec["gdn_trunk"] = dr.gdn_out[t_rows].cpu().view(torch.int16).numpy().copy()
        rec["S_P"] = dr.S_P[tj].cpu().numpy().view(np.int32).copy()
        a, b = int(rnd.opt_off[tq]), int(rnd.opt_off[tq + 1])
        rec["p"] = dr.p[a:b].cpu().numpy().view(np.int32).copy()
        outs.append(rec)
    for rec in outs[1:]:
        for key in outs[0]:
            assert np.array_equal(rec[key], outs[0][key]), key
