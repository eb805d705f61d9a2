"""Helpers of the GPU parity tests: oracle views of a round, device runs, comparisons."""
import numpy as np
import pytest

from oracle import forkattn as orc
from tree_forked_hybrid_gb300 import workloads as wl

ATOL_OUT = 2e-2   # layer outputs, unit-variance inputs (max |delta|)
RTOL_STATE = 1e-3  # S_P, relative Frobenius per (request, head)
TV_MAX = 1e-3     # option probabilities, total variation per question


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_forked_hybrid_gb300 import build
    build.build()
    return torch


def oracle_view(rnd: wl.Round, dtype=np.float32):
    lay = {}
    for name, d in rnd.layers.items():
        lay[name] = {k: (rnd.f32(name, k) if k != "conv_w" else d[k]).astype(dtype) for k in d}
    pre = None
    if rnd.prefix is not None:
        pre = {name: {k: rnd.prefix_f32(name, k).astype(dtype) for k in d} for name, d in rnd.prefix.items()}
    return orc.RoundView(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, lay, pre)


def to_np(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def seg_rows(view, segs):
    m = view.meta
    rows = []
    for s in segs:
        st, L = int(m["seg_start"][s]), int(m["seg_len"][s])
        rows.extend(range(st, st + L))
    return np.array(rows, dtype=np.int64)


def assert_close_rows(got, want, rows, atol=ATOL_OUT, what=""):
    if rows.shape[0] == 0:
        return
    d = np.abs(got[rows].astype(np.float64) - want[rows].astype(np.float64))
    assert np.isfinite(got[rows]).all(), f"{what}: non-finite output"
    assert d.max() <= atol, f"{what}: max |delta| {d.max():.3e} > {atol}"


def state_rel_err(got, want):
    num = np.linalg.norm((got.astype(np.float64) - want.astype(np.float64)).reshape(got.shape[0], got.shape[1], -1), axis=-1)
    den = np.linalg.norm(want.astype(np.float64).reshape(want.shape[0], want.shape[1], -1), axis=-1)
    return (num / np.maximum(den, 1e-30)).max()
