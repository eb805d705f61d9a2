"""fork_attn_noalloc, the entry point for callers that may not allocate device memory.

Such callers hold only pointers to their inputs and outputs; the variant takes
its scratch from an array owned by the library.  It runs the same kernels as
fork_attn (which uses a caller workspace), so its output must equal fork_attn's
bit for bit, on two calls in a row (the second one finds the first one's
scratch contents: a stale read would show).  This file is collected last so
that a failure here does not stop the others.
"""
import math

import numpy as np
import pytest

from tests.gpu_util import require_gpu
from tree_forked_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    torch = require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300.runner import DeviceRound

    # 16 q-heads / 4 kv-heads, d 128, full and sliding window, T_cap 4096 (fits the scratch array;
    # so would T_cap 16384)
    a = wl.AttnShape("attn", 16, 4, 128, 0, 10000.0)
    s = wl.AttnShape("swa", 16, 4, 128, 512, 10000.0)
    g = wl.GdnShape("gdn", 2, 64, 64, 4, 64)
    rnd = wl.custom_round([700, 1300, 5], [3, 2, 1], [40, 12, 64, 33, 1, 9], attn_shapes=(a, s), gdn_shape=g,
                          T_cap=4096, seed=21)
    dr = DeviceRound(rnd)
    dr.step_meta()
    T = rnd.T
    for call, a in enumerate(rnd.attn_shapes):  # two calls in a row: full, then window
        inp = dr.inputs[a.name]
        scale = 1.0 / math.sqrt(a.d)
        need = F.fork_attn_workspace_bytes(rnd.T_cap, 0, a.Hq, a.Hkv, a.d, a.rope_theta, 0)
        assert 0 < need <= F.FORK_NOALLOC_SCRATCH_BYTES
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.zeros((rnd.T_cap, a.Hq, a.d), dtype=torch.bfloat16, device="cuda")
        got = torch.zeros_like(ref)
        F.fork_attn(dr.meta, inp["q"], inp["k"], inp["v"], ref, a.Hq, a.Hkv, a.d, a.window, a.rope_theta,
                    scale, None, None, ws)
        F.fork_attn_noalloc(dr.meta, inp["q"], inp["k"], inp["v"], got, a.Hq, a.Hkv, a.d, a.window,
                            a.rope_theta, scale)
        torch.cuda.synchronize()
        assert F.fork_read_status(dr.meta) == 0
        r = ref[:T].float().cpu().numpy()
        g = got[:T].float().cpu().numpy()
        assert np.isfinite(g).all()
        assert torch.equal(ref[:T], got[:T]), f"call {call}: max |delta| {np.abs(g - r).max():.3e}"


def test_noalloc_rejects_rounds_beyond_its_scratch():
    require_gpu()
    from tree_forked_hybrid_gb300 import fork as F
    # long-document capacity, 8 kv-heads: its rotated keys alone take 64 MiB
    meta = F.Meta(32768, 4, 80, 32)
    assert F.fork_attn_workspace_bytes(32768, 0, 32, 8, 128, 10000.0, 0) > F.FORK_NOALLOC_SCRATCH_BYTES
    import torch
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(F.ForkError) as e:
        F.fork_attn_noalloc(meta, x, x, x, x, 32, 8, 128, 0, 10000.0, 0.088)
    assert e.value.code == 2  # FORK_ECAPACITY
