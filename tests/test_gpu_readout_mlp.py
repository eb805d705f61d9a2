"""Selective readout with the last layer's pointwise block (RMSNorm, SwiGLU MLP,
residual, final RMSNorm, eq. (1)) on the question rows only, against the oracle.

Round of 32 requests / 80 questions (two 64-row tiles, the second ragged),
D = 2048, F = 4096; hidden rows drawn N(0, 1) in bf16.  y within the layer-output
tolerance, probabilities within TV 1e-3; two calls give identical bits.
"""
import numpy as np
import pytest

from oracle import forkattn as orc
from tests.gpu_util import ATOL_OUT, require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_readout_mlp_matches_oracle():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300.runner import DeviceRound

    rnd = wl.make_round(1, seed=4)
    D, Fw = rnd.D, 2 * rnd.D
    dr = DeviceRound(rnd)
    dr.step_meta()
    rng = np.random.default_rng(9)
    h = np.zeros((rnd.T_cap, D), dtype=np.uint16)
    h[:rnd.T] = wl.bf16_bits(rng.standard_normal((rnd.T, D), dtype=np.float32))
    wts = wl.readout_block_weights(D, Fw)
    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    h_d = dev(h)
    W = {k: dev(v) for k, v in wts.items()}
    p = torch.zeros(int(rnd.opt_off[-1]), dtype=torch.float32, device="cuda")
    nbytes = F.fork_readout_mlp_workspace_bytes(dr.max_q, D, Fw)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        F.fork_readout_mlp(dr.meta, h_d, D, Fw, W["g1"], W["w_gate"], W["w_up"], W["w_down"], W["g2"],
                           dr.w_opt, dr.opt_off, p, ws)
        torch.cuda.synchronize()
        outs.append(p.cpu().numpy().copy())
    assert F.fork_read_status(dr.meta) == 0
    assert np.array_equal(outs[0], outs[1])

    m = orc.meta_ref(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, 32)
    rows = wl.bf16_to_f32(h[m["q_last"]])
    f32 = {k: (wl.bf16_to_f32(v) if v.dtype == np.uint16 else v) for k, v in wts.items()}
    y_ref = orc.mlp_block(rows, f32["g1"], f32["w_gate"], f32["w_up"], f32["w_down"])
    p_ref = orc.readout_mlp(rows, f32["g1"], f32["w_gate"], f32["w_up"], f32["w_down"], f32["g2"],
                            rnd.w_opt_f32(), rnd.opt_off)
    # y from the workspace: [Mpad, D] float32 after two bf16 arrays
    Mpad = (dr.max_q + 63) // 64 * 64
    al = lambda x: (x + 255) // 256 * 256
    y_off = al(al(Mpad * D * 2) + Mpad * Fw * 2)
    y = ws[y_off:y_off + Mpad * D * 4].view(torch.float32).view(Mpad, D)[:rnd.Nq].cpu().numpy()
    assert np.isfinite(y).all()
    assert np.abs(y - y_ref).max() <= ATOL_OUT, np.abs(y - y_ref).max()
    tv = orc.total_variation(outs[0], p_ref, rnd.opt_off)
    assert tv.max() <= 1e-3, tv.max()


def test_pointwise_block_on_every_row_matches_oracle_and_selective():
    """The same block on every stream row (the cost the selective readout avoids): z on
    every row against the oracle's block, and eq. (1) from the questions' rows of z
    against the oracle (TV 1e-3)."""
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300.runner import DeviceRound

    a = wl.AttnShape("attn", 4, 1, 64, 0, 0.0)
    g = wl.GdnShape("gdn", 4, 64, 64, 4, 64)  # D = 256
    rnd = wl.custom_round([300, 41], [2, 1], [20, 7, 64], attn_shapes=(a,), gdn_shape=g, T_cap=512, seed=6)
    D, Fw = rnd.D, 2 * rnd.D
    dr = DeviceRound(rnd)
    dr.step_meta()
    rng = np.random.default_rng(10)
    h = np.zeros((rnd.T_cap, D), dtype=np.uint16)
    h[:rnd.T] = wl.bf16_bits(rng.standard_normal((rnd.T, D), dtype=np.float32))
    wts = wl.readout_block_weights(D, Fw)
    dev = lambda x: torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).cuda()
    h_d = dev(h)
    W = {k: dev(v) for k, v in wts.items()}
    z = torch.full((rnd.T_cap, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(F.fork_pointwise_rows_workspace_bytes(rnd.T_cap, D, Fw), dtype=torch.uint8, device="cuda")
    F.fork_pointwise_rows(dr.meta, h_d, D, Fw, W["g1"], W["w_gate"], W["w_up"], W["w_down"], W["g2"], z, ws)
    p = torch.zeros(int(rnd.opt_off[-1]), dtype=torch.float32, device="cuda")
    F.fork_readout(dr.meta, z, D, dr.w_opt, dr.opt_off, p)
    torch.cuda.synchronize()
    assert F.fork_read_status(dr.meta) == 0
    zz = z.float().cpu().numpy()
    assert np.isnan(zz[rnd.T:]).all()  # pad rows untouched
    f32 = {k: (wl.bf16_to_f32(v) if v.dtype == np.uint16 else v) for k, v in wts.items()}
    rows = wl.bf16_to_f32(h[:rnd.T])
    y_ref = orc.mlp_block(rows, f32["g1"], f32["w_gate"], f32["w_up"], f32["w_down"])
    z_ref = orc.rms_norm(y_ref, f32["g2"])
    assert np.abs(zz[:rnd.T] - z_ref).max() <= ATOL_OUT, np.abs(zz[:rnd.T] - z_ref).max()
    m = orc.meta_ref(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, 32)
    p_ref = orc.readout_mlp(wl.bf16_to_f32(h[m["q_last"]]), f32["g1"], f32["w_gate"], f32["w_up"], f32["w_down"],
                            f32["g2"], rnd.w_opt_f32(), rnd.opt_off)
    tv = orc.total_variation(p.cpu().numpy(), p_ref, rnd.opt_off)
    assert tv.max() <= 1e-3, tv.max()
