"""Host-side reader of a metadata buffer copied back from the device.

Mirrors the word offsets of ``fork::meta_layout`` (csrc/fork_common.cuh): a
32-word header, then every array at an offset rounded up to 32 words.
"""
from __future__ import annotations

import numpy as np

H_WORDS = 32
MIN_TILE = 8
HDR = ("magic", "T_cap", "max_req", "max_q", "max_seg", "max_work", "R", "Nq", "T", "nseg", "tile",
       "n_work", "status", "prefix_total", "valid", "forest")


def _align(w: int) -> int:
    return (w + 31) & ~31


def offsets(T_cap: int, max_req: int, max_q: int):
    max_seg = max_req + max_q
    max_work = (T_cap + MIN_TILE - 1) // MIN_TILE + max_seg
    o = H_WORDS
    out = {}
    plan = [("tok_req", T_cap), ("tok_branch", T_cap), ("tok_pos", T_cap)]
    plan += [(k, max_seg) for k in ("seg_start", "seg_len", "seg_pos0", "seg_req", "seg_branch",
                                    "seg_trunk_start", "seg_trunk_len", "seg_state_idx")]
    plan += [(k, max_req) for k in ("req_trunk_len", "req_prefix_len", "req_prefix_off", "req_ckpt_pos",
                                    "req_trunk_start", "req_first_q", "req_n_q")]
    plan += [("q_last", max(max_q, 1)), ("work_seg", max_work), ("work_off", max_work), ("work_order", max_work)]
    for name, n in plan:
        out[name] = (o, n)
        o = _align(o + n)
    return out, o


def unpack(words: np.ndarray, T_cap: int, max_req: int, max_q: int) -> dict:
    words = np.asarray(words, dtype=np.int32)
    offs, total = offsets(T_cap, max_req, max_q)
    res = {k: int(words[i]) for i, k in enumerate(HDR)}
    T, R, Nq, nseg, nw = res["T"], res["R"], res["Nq"], res["nseg"], res["n_work"]
    lens = {"tok": T_cap, "seg": nseg, "req": R, "q_last": Nq, "work": nw}
    for name, (o, n) in offs.items():
        key = name.split("_")[0]
        m = lens.get(key, lens.get(name, n))
        res[name] = words[o:o + min(m, n)].copy()
    return res
