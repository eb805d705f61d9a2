"""Failure handling on the device, through the C-ABI (needs a GB300).

- Bounded waits: with FORK_TEST_STALL one role of every CTA waits on a barrier
  that nothing completes; the wait runs out after fork_meta.wait_us, the call
  reports FORK_STATUS_TIMEOUT, and the next normal call on the same stream is
  correct (the context stays usable, tensor memory was given back).
- FORK_CHECKS: a clean round passes every check with unchanged bits; a
  corrupted segment table and bad option offsets are caught (status bit, the
  work skipped), never trapped.
- Workspaces filled with NaN beforehand change nothing (every value read is
  written first).
"""
import pytest

from tests.gpu_util import require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def small_round(seed=5):
    a = wl.AttnShape("attn", 8, 2, 128, 0, 10000.0)
    g = wl.GdnShape("gdn", 2, 128, 128, 4, 64)
    return wl.custom_round([300, 190], [2, 3], [40, 7, 64, 20, 1], attn_shapes=(a,), gdn_shape=g,
                           T_cap=1024, seed=seed)


def test_stalled_waits_run_out_and_the_next_call_is_correct():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300.runner import DeviceRound
    rnd = small_round()
    ref = DeviceRound(rnd)
    ref.run()
    torch.cuda.synchronize()
    assert ref.status() == 0
    dr = DeviceRound(rnd)
    steps = {"attn": lambda: dr.step_attn("attn"), "gdn_trunk": dr.step_gdn_trunk,
             "gdn_branches": dr.step_gdn_branches}
    for name, step in steps.items():
        dr.step_meta()
        if name == "gdn_branches":
            dr.step_gdn_trunk()  # the branch call's inputs
        dr.meta.set_wait_limit_us(2000)
        dr.flags = F.FORK_TEST_STALL
        step()
        dr.flags = 0
        dr.meta.set_wait_limit_us(0)
        torch.cuda.synchronize()
        assert dr.status() & F.FORK_STATUS_TIMEOUT, name
    # normal calls on the same stream afterwards: bit-identical to the reference run
    dr.run()
    torch.cuda.synchronize()
    assert dr.status() == 0
    assert torch.equal(dr.attn_out["attn"][:rnd.T], ref.attn_out["attn"][:rnd.T])
    assert torch.equal(dr.gdn_out[:rnd.T], ref.gdn_out[:rnd.T])
    assert torch.equal(dr.S_P, ref.S_P)
    assert torch.equal(dr.p, ref.p)


def test_checks_pass_on_a_clean_round_with_unchanged_bits():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300.runner import DeviceRound
    rnd = wl.make_round(1)
    plain = DeviceRound(rnd)
    plain.run()
    checked = DeviceRound(rnd, flags=F.FORK_CHECKS)
    checked.run()
    torch.cuda.synchronize()
    assert plain.status() == 0 and checked.status() == 0
    for name in plain.attn_out:
        assert torch.equal(plain.attn_out[name], checked.attn_out[name])
    assert torch.equal(plain.gdn_out, checked.gdn_out)
    assert torch.equal(plain.S_P, checked.S_P)
    assert torch.equal(plain.p, checked.p)


def test_checks_catch_a_corrupted_segment_and_bad_option_offsets():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300 import layout as LY
    from tree_forked_hybrid_gb300.runner import DeviceRound
    rnd = small_round(7)
    dr = DeviceRound(rnd, flags=F.FORK_CHECKS)
    offs, _ = LY.offsets(rnd.T_cap, dr.max_req, dr.max_q)
    # (a) the tables as built pass; then question 1's segment is made to run past the stream
    dr.step_meta()
    torch.cuda.synchronize()
    assert dr.status() == 0
    seg_len = offs["seg_len"][0] + rnd.R + 1
    dr.meta.buf[seg_len] = rnd.T_cap + 100
    dr.step_attn("attn")
    torch.cuda.synchronize()
    assert dr.status() & F.FORK_STATUS_CHECK
    dr.step_meta()
    dr.step_gdn_trunk()
    torch.cuda.synchronize()
    assert dr.status() == 0
    dr.meta.buf[seg_len] = rnd.T_cap + 100
    dr.step_gdn_branches()
    torch.cuda.synchronize()
    assert dr.status() & F.FORK_STATUS_CHECK
    # (b) option offsets that do not grow
    dr.step_meta()
    dr.step_gdn_trunk()
    dr.step_gdn_branches()
    bad = dr.opt_off.clone()
    bad[2] = bad[1]
    F.fork_readout(dr.meta, dr.gdn_out, rnd.D, dr.w_opt, bad, dr.p, F.FORK_CHECKS)
    torch.cuda.synchronize()
    assert dr.status() & F.FORK_STATUS_CHECK


def test_nan_filled_workspaces_change_nothing():
    torch = require_gpu()
    from tree_forked_hybrid_gb300.runner import DeviceRound
    rnd = wl.make_round(2)
    a = DeviceRound(rnd)
    a.run()
    b = DeviceRound(rnd)
    for ws in b.attn_ws.values():
        if ws is not None:
            ws.fill_(0xFF)  # every bf16/float32 word a NaN
    b.run()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    for name in a.attn_out:
        assert torch.equal(a.attn_out[name][:rnd.T], b.attn_out[name][:rnd.T])
    assert torch.equal(a.gdn_out[:rnd.T], b.gdn_out[:rnd.T])
    assert torch.equal(a.p, b.p)
