"""CUDA path vs the CPU oracle, through the C-ABI (needs a GB300)."""
import math

import numpy as np
import pytest

from oracle import forkattn as orc
from tests.golden_io import load_meta_cases
from tests.gpu_util import (ATOL_OUT, RTOL_STATE, TV_MAX, assert_close_rows, oracle_view, require_gpu,
                            seg_rows, state_rel_err, to_np)
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

META_KEYS = ("tok_req", "tok_branch", "tok_pos", "seg_start", "seg_len", "seg_pos0", "seg_req",
             "seg_branch", "seg_trunk_start", "seg_trunk_len", "seg_state_idx", "req_trunk_len",
             "req_prefix_len", "req_prefix_off", "req_ckpt_pos", "req_trunk_start", "req_first_q",
             "req_n_q", "q_last", "work_seg", "work_off")


def device_meta(desc, R, Nq, T_cap, tile, max_req=None, max_q=None):
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300 import layout as LY
    meta = F.Meta(T_cap, max_req or max(R, 1), Nq if max_q is None else max_q, tile)
    d = torch.from_numpy(np.asarray(desc, dtype=np.int32)).cuda()
    F.fork_build_meta(meta, d, R, Nq)
    torch.cuda.synchronize()
    return LY.unpack(meta.buf.cpu().numpy(), T_cap, meta.max_req, meta.max_q), meta


def check_meta_equal(desc, R, Nq, T_cap, tile, **kw):
    got, _ = device_meta(desc, R, Nq, T_cap, tile, **kw)
    want = orc.meta_ref(desc, R, Nq, T_cap, tile)
    assert got["T"] == int(want["T"]) and got["nseg"] == int(want["nseg"])
    assert got["status"] == 0
    for k in META_KEYS:
        n = want[k].shape[0]
        assert np.array_equal(got[k][:n], want[k]), k
    assert got["n_work"] == want["work_seg"].shape[0]


@pytest.mark.parametrize("name", sorted(load_meta_cases()))
def test_meta_golden(name):
    """Hand-derived fixtures: tile-independent fields equal the fixture; the
    work list (the device takes tiles of 8..128 tokens) equals the oracle's."""
    c = load_meta_cases()[name]
    R, Nq, T_cap = int(c["R"][0]), int(c["Nq"][0]), int(c["T_cap"][0])
    tile = max(8, int(c["tile"][0]))
    check_meta_equal(c["desc"], R, Nq, T_cap, tile)
    got, _ = device_meta(c["desc"], R, Nq, T_cap, tile)
    for key, want in c.items():
        if key in ("R", "Nq", "T_cap", "tile", "desc") or key.startswith("work_"):
            continue
        if key == "T":
            assert got["T"] == int(want[0])
            continue
        assert got[key][:want.shape[0]].tolist() == want.tolist(), key


@pytest.mark.parametrize("wid", [0, 1, 2, 3, 4])
def test_meta_workloads(wid):
    rnd = wl.make_round(wid)
    tile = 128 // (rnd.attn_shapes[0].Hq // rnd.attn_shapes[0].Hkv)
    check_meta_equal(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, tile, max_req=rnd.R + 3, max_q=rnd.Nq + 5)


@pytest.mark.parametrize("wid", [1, 3])
def test_work_items_launch_longest_first(wid):
    """The launch order is a permutation of the work list in non-increasing key count
    (position after the item's last query), ties in list order."""
    rnd = wl.make_round(wid)
    tile = 256 // (rnd.attn_shapes[0].Hq // rnd.attn_shapes[0].Hkv)
    got, _ = device_meta(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, tile)
    want = orc.meta_ref(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, tile)
    nw = want["work_seg"].shape[0]
    order = got["work_order"][:nw]
    assert sorted(order.tolist()) == list(range(nw))
    seg, off = want["work_seg"], want["work_off"]
    cost = want["seg_pos0"][seg] + off + np.minimum(tile, want["seg_len"][seg] - off)
    expect = sorted(range(nw), key=lambda w: (-int(cost[w]), w))
    assert order.tolist() == expect


@pytest.mark.parametrize("seed", range(6))
def test_meta_random(seed):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.integers(1, 40))
    P = rng.integers(0, 300, size=R)
    n = rng.integers(0, 9, size=R)
    ql = rng.integers(1, 70, size=int(n.sum()))
    pl = np.array([rng.integers(0, p + 1) if rng.random() < 0.2 else 0 for p in P])
    ck = np.array([rng.integers(pl[j], P[j] + 1) if rng.random() < 0.2 else -1 for j in range(R)])
    desc = np.concatenate([P, n, ql, pl, ck]).astype(np.int32)
    T = int((P - pl).sum() + ql.sum())
    check_meta_equal(desc, R, int(n.sum()), T + int(rng.integers(0, 50)), int(rng.choice([8, 16, 32, 64, 128])))


def test_meta_bad_descriptor_sets_status():
    # q_len 0, negative trunk, checkpoint outside [prefix, P], over capacity
    cases = [([10, 1, 0, 0, -1], 1, 1, 16, 0x1), ([-3, 0, 0, -1], 1, 0, 16, 0x1),
             ([10, 0, 0, 11], 1, 0, 16, 0x4), ([10, 1, 9, 0, -1], 1, 1, 16, 0x2)]
    for desc, R, Nq, T_cap, bit in cases:
        got, meta = device_meta(desc, R, Nq, T_cap, 32)
        assert got["status"] & bit, (desc, got["status"])
        assert got["T"] == 0 and got["n_work"] == 0
        from tree_forked_hybrid_gb300 import fork as F
        assert F.fork_read_status(meta) & bit


# ---------------------------------------------------------------------------
# layer parity
# ---------------------------------------------------------------------------

def run_device(rnd, **kw):
    torch = require_gpu()
    from tree_forked_hybrid_gb300.runner import DeviceRound
    dr = DeviceRound(rnd, **kw)
    dr.run()
    torch.cuda.synchronize()
    assert dr.status() == 0
    return dr


def check_attention(rnd, dr, view, name, questions=None, trunk_rows=None, trunks=None):
    a = [x for x in rnd.attn_shapes if x.name == name][0]
    want = orc.run_attention(view, name, window=a.window, rope_theta=a.rope_theta, questions=questions,
                             trunks=trunks, trunk_rows=trunk_rows)
    got = to_np(dr.attn_out[name])
    m = view.meta
    rows = []
    qs = range(rnd.Nq) if questions is None else questions
    rows.append(seg_rows(view, [rnd.R + q for q in qs]))
    ts = range(rnd.R) if trunks is None else trunks
    for j in ts:
        st = int(m["req_trunk_start"][j])
        if trunk_rows is not None and j in trunk_rows:
            rows.append(st + np.asarray(trunk_rows[j]) - int(rnd.prefix_len[j]))
        else:
            rows.append(seg_rows(view, [j]))
    assert_close_rows(got, want, np.concatenate(rows), what=name)


def check_gdn(rnd, dr, view, questions=None, trunks=None):
    out = orc.run_gdn(view, rnd.gdn_shape.name, questions=questions, trunks=trunks)
    got = to_np(dr.gdn_out)
    qs = range(rnd.Nq) if questions is None else questions
    ts = range(rnd.R) if trunks is None else list(trunks)
    rows = np.concatenate([seg_rows(view, [rnd.R + q for q in qs]), seg_rows(view, ts)])
    assert_close_rows(got, out["o"], rows, what="gdn o")
    sp = to_np(dr.S_P)[:rnd.R]
    assert state_rel_err(sp[ts], out["S_P"][ts]) <= RTOL_STATE
    g = rnd.gdn_shape
    cw = to_np(dr.conv_win)[:rnd.R]
    want_cw = out["conv_win"][:, :, :, :, :g.dk]
    assert np.array_equal(cw[ts], want_cw[ts]), "conv window rows are copies of bf16 inputs"
    if dr.has_ckpt:
        ck = [j for j in ts if rnd.ckpt_pos[j] >= 0]
        assert state_rel_err(to_np(dr.S_ckpt)[ck], out["S_ckpt"][ck]) <= RTOL_STATE
        assert np.array_equal(to_np(dr.conv_ckpt)[ck], out["conv_ckpt"][ck][..., :g.dk])
    return out


def check_readout(rnd, dr, view, questions=None):
    qs = list(range(rnd.Nq)) if questions is None else list(questions)
    off = rnd.opt_off
    p = to_np(dr.p)
    # (a) identical h: the kernel alone
    h_gpu = to_np(dr.gdn_out)
    ref_same_h = orc.run_readout(view, h_gpu, rnd.w_opt_f32(), off)
    tv = orc.total_variation(p, ref_same_h, off)
    assert tv[qs].max() <= TV_MAX, f"readout TV (same h) {tv[qs].max():.2e}"
    for i in qs:
        assert abs(p[off[i]:off[i + 1]].sum() - 1.0) < 1e-5
    return tv


@pytest.mark.parametrize("wid", [0, 1, 2])
def test_layer_parity_small_workloads(wid):
    rnd = wl.make_round(wid)
    dr = run_device(rnd)
    view = oracle_view(rnd)
    for a in rnd.attn_shapes:
        check_attention(rnd, dr, view, a.name)
    out = check_gdn(rnd, dr, view)
    check_readout(rnd, dr, view)
    # end to end: the oracle's own h
    p_ref = orc.run_readout(view, out["o"].reshape(rnd.T_cap, -1), rnd.w_opt_f32(), rnd.opt_off)
    tv = orc.total_variation(to_np(dr.p), p_ref, rnd.opt_off)
    assert tv.max() <= TV_MAX, f"end-to-end TV {tv.max():.2e}"


def test_layer_parity_long_documents_sampled():
    """Full-size long-document round, in the bench's launch configuration;
    the oracle computes sampled trunk rows and a few whole questions."""
    rnd = wl.make_round(3)
    dr = run_device(rnd)
    view = oracle_view(rnd)
    m = view.meta
    qs = [0, int(m["req_first_q"][2]) + 1, rnd.Nq - 1]
    P0 = int(rnd.trunk_len[0])
    trunk_rows = {0: np.r_[0:40, 2000:2033, P0 - 70:P0], 3: np.r_[int(rnd.trunk_len[3]) - 33:int(rnd.trunk_len[3])]}
    for a in rnd.attn_shapes:
        check_attention(rnd, dr, view, a.name, questions=qs, trunk_rows=trunk_rows, trunks=[0, 3])
    out = check_gdn(rnd, dr, view, questions=qs, trunks=[0, 2])
    check_readout(rnd, dr, view, questions=qs)


def test_resume_round_matches_scratch():
    """Wide fork with a checkpoint at m (round A), then a round that resumes it:
    B's outputs match a from-scratch oracle run of its full 17408-token trunk."""
    ra = wl.make_round(4)
    rb = wl.make_resume_round(ra)
    dra = run_device(ra)
    va = oracle_view(ra)
    # round A: checkpoint state and window, sampled attention rows, two questions
    P = int(ra.trunk_len[0])
    check_gdn(ra, dra, va, questions=[0, 63])
    for a in ra.attn_shapes:
        check_attention(ra, dra, va, a.name, questions=[5], trunk_rows={0: np.r_[15300:15400, P - 10:P]})
    drb = run_device(rb, resume_from=dra)
    vb = oracle_view(rb)
    qs = [0, 31, 63]
    for a in rb.attn_shapes:
        check_attention(rb, drb, vb, a.name, questions=qs,
                        trunk_rows={0: np.r_[15360:15420, 17300:17408]})
    check_gdn(rb, drb, vb, questions=qs)
    check_readout(rb, drb, vb, questions=qs)


@pytest.mark.parametrize("d", [64, 128])
def test_edge_cases_round(d):
    """Empty trunk, a request without questions, one-token questions, odd tails,
    a stream that fills the capacity exactly; at d = 128 the tensor-core GDN
    kernel (the d = 64 one is the warp-MMA kernel)."""
    a = wl.AttnShape("attn", 4, 1, d, 0, 10000.0)
    s = wl.AttnShape("swa", 4, 1, d, 5, 10000.0)
    g = wl.GdnShape("gdn", 2, d, d, 4, 64)
    P = [0, 67, 130, 1, 2]
    n = [2, 0, 3, 1, 1]
    ql = [1, 5, 64, 65, 1, 3, 2]
    T = sum(P) + sum(ql)
    rnd = wl.custom_round(P, n, ql, attn_shapes=(a, s), gdn_shape=g, T_cap=T, seed=11)
    dr = run_device(rnd, max_req=8, max_q=16)
    view = oracle_view(rnd)
    for x in rnd.attn_shapes:
        check_attention(rnd, dr, view, x.name)
    check_gdn(rnd, dr, view)
    check_readout(rnd, dr, view)


def test_pad_rows_untouched():
    torch = require_gpu()
    from tree_forked_hybrid_gb300.runner import DeviceRound
    rnd = wl.make_round(0)
    dr = DeviceRound(rnd)
    T = rnd.T
    canary = torch.tensor(float("nan"), dtype=torch.bfloat16, device="cuda")
    for o in list(dr.attn_out.values()) + [dr.gdn_out]:
        o[T:] = canary
    dr.run()
    torch.cuda.synchronize()
    for o in list(dr.attn_out.values()) + [dr.gdn_out]:
        assert torch.isnan(o[T:].float()).all()
        assert torch.isfinite(o[:T].float()).all()


def test_warp_mma_variant_matches_oracle():
    """The warp-level mma.sync kernels (FORK_WARP_MMA: attention and GDN) against the oracle."""
    require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    rnd = wl.make_round(2)
    dr = run_device(rnd, flags=F.FORK_WARP_MMA)
    view = oracle_view(rnd)
    for a in rnd.attn_shapes:
        check_attention(rnd, dr, view, a.name)
    check_gdn(rnd, dr, view)
    check_readout(rnd, dr, view)
