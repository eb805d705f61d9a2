"""Python binding of the C ABI in include/forkattn.h (argument marshalling only).

Every function here has the name of the C entry point it calls and passes
device pointers of torch tensors plus the current CUDA stream (the token-forest
planner takes host arrays).  No arithmetic of the layer happens here: if the
library cannot be loaded, the call fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from . import build as _build

STATUS = {0: "FORK_OK", 1: "FORK_EINVAL", 2: "FORK_ECAPACITY", 3: "FORK_EUNSUPPORTED", 4: "FORK_ECUDA"}
STATUS_BITS = {0x1: "BAD_DESC", 0x2: "CAPACITY", 0x4: "BAD_CKPT", 0x8: "TIMEOUT", 0x10: "BAD_PREFIX",
               0x20: "CHECK"}
FORK_STATUS_TIMEOUT = 0x8
FORK_STATUS_CHECK = 0x20
FORK_DETERMINISTIC = 0x1
FORK_CHECKS = 0x2
FORK_WARP_MMA = 0x4
FORK_FOREST = 0x8
FORK_TEST_STALL = 0x100
FORK_FOREST_MAX_DEPTH = 7  # ancestors of a forest node, at most (include/forkattn.h)
FORK_FOREST_MAX_LEVELS = FORK_FOREST_MAX_DEPTH + 1
FORK_NOALLOC_SCRATCH_BYTES = 32 << 20  # size of the library's scratch array (include/forkattn.h)

_lib = None


class ForkError(RuntimeError):
    def __init__(self, fn: str, code: int, cuda_error: int = 0):
        extra = f" (CUDA error {cuda_error})" if code == 4 and cuda_error else ""
        super().__init__(f"{fn} returned {STATUS.get(code, code)}{extra}")
        self.code = code
        self.cuda_error = cuda_error


class fork_meta(ctypes.Structure):
    _fields_ = [("d_buf", ctypes.c_void_p), ("bytes", ctypes.c_size_t), ("T_cap", ctypes.c_int32),
                ("max_req", ctypes.c_int32), ("max_q", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("wait_us", ctypes.c_uint32)]


def lib_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libforkattn.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: run tree_forked_hybrid_gb300.build.build() first")
    L = ctypes.CDLL(p)
    vp, i32, u32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
    MP = ctypes.POINTER(fork_meta)
    sig = {
        "fork_meta_bytes": (sz, [i32, i32, i32]),
        "fork_meta_init": (ctypes.c_int, [MP, vp, sz, i32, i32, i32, i32]),
        "fork_build_meta": (ctypes.c_int, [MP, vp, i32, i32, u32, vp]),
        "fork_desc_capacity_words": (sz, [i32, i32]),
        "fork_build_meta_dev": (ctypes.c_int, [MP, vp, u32, vp]),
        "fork_read_status": (ctypes.c_int, [MP, ctypes.POINTER(i32), vp]),
        "fork_last_cuda_error": (ctypes.c_int, []),
        "fork_attn_workspace_bytes": (sz, [i32, i32, i32, i32, i32, f32, u32]),
        "fork_attn": (ctypes.c_int, [MP, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, vp, vp, i32, vp,
                                     sz, u32, vp]),
        "fork_attn_noalloc": (ctypes.c_int, [MP, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, vp, vp, i32,
                                             u32, vp]),
        "fork_gdn_trunk": (ctypes.c_int, [MP, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp,
                                          vp, vp, vp, u32, vp]),
        "fork_gdn_branches": (ctypes.c_int, [MP, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp,
                                             u32, vp]),
        "fork_readout": (ctypes.c_int, [MP, vp, i32, vp, vp, vp, u32, vp]),
        "fork_forest_plan": (ctypes.c_int, [MP, vp, vp, i32, vp, vp]),
        "fork_build_forest_meta": (ctypes.c_int, [MP, vp, vp, i32, vp, vp, vp]),
        "fork_gdn_forest": (ctypes.c_int, [MP, i32, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp,
                                           u32, vp]),
        "fork_readout_mlp_workspace_bytes": (sz, [i32, i32, i32]),
        "fork_readout_mlp": (ctypes.c_int, [MP, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, u32, vp]),
        "fork_pointwise_rows_workspace_bytes": (sz, [i32, i32, i32]),
        "fork_pointwise_rows": (ctypes.c_int, [MP, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, u32, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = L
    return L


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise ForkError(fn, rc, load().fork_last_cuda_error() if rc == 4 else 0)


class Meta:
    """A metadata buffer (device) with its host-side fork_meta handle."""

    def __init__(self, T_cap: int, max_req: int, max_q: int, tile_tokens: int, device="cuda"):
        L = load()
        nbytes = L.fork_meta_bytes(T_cap, max_req, max_q)
        if nbytes == 0:
            raise ValueError("invalid metadata capacities")
        self.buf = torch.zeros(nbytes // 4, dtype=torch.int32, device=device)
        self.handle = fork_meta()
        _check("fork_meta_init", L.fork_meta_init(ctypes.byref(self.handle), ctypes.c_void_p(self.buf.data_ptr()),
                                                  nbytes, T_cap, max_req, max_q, tile_tokens))
        self.T_cap, self.max_req, self.max_q, self.tile_tokens = T_cap, max_req, max_q, tile_tokens

    def set_wait_limit_us(self, us: int):
        """Limit of the kernels' bounded waits for later calls (0 = the default 2 s)."""
        self.handle.wait_us = int(us)

    @property
    def ref(self):
        return ctypes.byref(self.handle)


def fork_meta_bytes(T_cap: int, max_req: int, max_q: int) -> int:
    return load().fork_meta_bytes(T_cap, max_req, max_q)


def fork_build_meta(meta: Meta, desc: torch.Tensor, R: int, Nq: int, flags: int = 0, stream=None):
    _check("fork_build_meta", load().fork_build_meta(meta.ref, _ptr(desc), R, Nq, flags, _stream(stream)))


def fork_desc_capacity_words(max_req: int, max_q: int) -> int:
    return load().fork_desc_capacity_words(max_req, max_q)


def fork_build_meta_dev(meta: Meta, desc: torch.Tensor, flags: int = 0, stream=None):
    """Metadata from a fixed-capacity device descriptor (counts read on the device)."""
    _check("fork_build_meta_dev", load().fork_build_meta_dev(meta.ref, _ptr(desc), flags, _stream(stream)))


def fork_read_status(meta: Meta, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("fork_read_status", load().fork_read_status(meta.ref, ctypes.byref(out), _stream(stream)))
    return out.value


def fork_attn_workspace_bytes(T_cap: int, prefix_rows: int, Hq: int, Hkv: int, d: int, rope_theta: float,
                              flags: int = 0) -> int:
    return load().fork_attn_workspace_bytes(T_cap, prefix_rows, Hq, Hkv, d, rope_theta, flags)


def fork_attn(meta: Meta, q, k, v, o, Hq: int, Hkv: int, d: int, window: int, rope_theta: float,
              scale: float, prefix_k=None, prefix_v=None, workspace=None, flags: int = 0, stream=None):
    prefix_rows = 0 if prefix_k is None else int(prefix_k.shape[0])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("fork_attn", load().fork_attn(meta.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(o), Hq, Hkv, d, window,
                                         rope_theta, scale, _ptr(prefix_k), _ptr(prefix_v), prefix_rows,
                                         _ptr(workspace), ws_bytes, flags, _stream(stream)))


def fork_attn_noalloc(meta: Meta, q, k, v, o, Hq: int, Hkv: int, d: int, window: int, rope_theta: float,
                      scale: float, prefix_k=None, prefix_v=None, flags: int = 0, stream=None):
    """fork_attn without a workspace argument (the library's own scratch array)."""
    prefix_rows = 0 if prefix_k is None else int(prefix_k.shape[0])
    _check("fork_attn_noalloc", load().fork_attn_noalloc(
        meta.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(o), Hq, Hkv, d, window, rope_theta, scale,
        _ptr(prefix_k), _ptr(prefix_v), prefix_rows, flags, _stream(stream)))


def fork_gdn_trunk(meta: Meta, q, k, v, alpha, eta, conv_w, H: int, d: int, K: int, chunk: int,
                   S_P, conv_win, o, init_state=None, init_conv=None, S_ckpt=None, conv_ckpt=None,
                   flags: int = 0, stream=None):
    _check("fork_gdn_trunk", load().fork_gdn_trunk(
        meta.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), _ptr(conv_w), H, d, K, chunk,
        _ptr(init_state), _ptr(init_conv), _ptr(S_P), _ptr(conv_win), _ptr(S_ckpt), _ptr(conv_ckpt),
        _ptr(o), flags, _stream(stream)))


def fork_gdn_branches(meta: Meta, q, k, v, alpha, eta, conv_w, H: int, d: int, K: int, chunk: int,
                      S_P, conv_win, o, flags: int = 0, stream=None):
    _check("fork_gdn_branches", load().fork_gdn_branches(
        meta.ref, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), _ptr(conv_w), H, d, K, chunk,
        _ptr(S_P), _ptr(conv_win), _ptr(o), flags, _stream(stream)))


class ForestPlan:
    """The plan that fork_forest_plan writes next to the metadata image: the levels (first
    state index of each depth, and the end) and each node's state index."""

    def __init__(self, words, N: int):
        w = np.asarray(words)
        self.levels = int(w[0])
        self.level_first = w[1:2 + self.levels].astype(np.int64)
        self.state_index = w[2 + FORK_FOREST_MAX_LEVELS:2 + FORK_FOREST_MAX_LEVELS + N].astype(np.int64)


def _host_ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _forest_arrays(parent, node_len, nbytes: int):
    """int32 host arrays of a forest call: parents, lengths, the metadata image, the plan."""
    par = np.ascontiguousarray(parent, dtype=np.int32)
    ln = np.ascontiguousarray(node_len, dtype=np.int32)
    img = np.zeros(nbytes // 4, dtype=np.int32)
    plan = np.zeros(par.shape[0] + 2 + FORK_FOREST_MAX_LEVELS, dtype=np.int32)
    return par, ln, img, plan


def fork_forest_plan(T_cap: int, max_req: int, max_q: int, tile_tokens: int, parent, node_len):
    """Host-only plan of a token forest (no device involved): (metadata image, ForestPlan).
    The handle passed to the C call describes the capacities; its buffer is the image."""
    L = load()
    nbytes = L.fork_meta_bytes(T_cap, max_req, max_q)
    if nbytes == 0:
        raise ValueError("invalid metadata capacities")
    par, ln, img, plan = _forest_arrays(parent, node_len, nbytes)
    h = fork_meta()
    _check("fork_meta_init", L.fork_meta_init(ctypes.byref(h), _host_ptr(img), nbytes, T_cap, max_req, max_q,
                                              tile_tokens))
    _check("fork_forest_plan", L.fork_forest_plan(ctypes.byref(h), _host_ptr(par), _host_ptr(ln), int(par.shape[0]),
                                                  _host_ptr(img), _host_ptr(plan)))
    return img, ForestPlan(plan, int(par.shape[0]))


def fork_build_forest_meta(meta: Meta, parent, node_len, stream=None) -> ForestPlan:
    """Plan a token forest on the host and copy its metadata into meta's device buffer."""
    nbytes = meta.buf.numel() * 4
    par, ln, img, plan = _forest_arrays(parent, node_len, nbytes)
    _check("fork_build_forest_meta", load().fork_build_forest_meta(
        meta.ref, _host_ptr(par), _host_ptr(ln), int(par.shape[0]), _host_ptr(img), _host_ptr(plan),
        _stream(stream)))
    return ForestPlan(plan, int(par.shape[0]))


def fork_gdn_forest(meta: Meta, first: int, count: int, q, k, v, alpha, eta, conv_w, H: int, d: int, K: int,
                    chunk: int, node_state, node_conv, o, flags: int = 0, stream=None):
    _check("fork_gdn_forest", load().fork_gdn_forest(
        meta.ref, first, count, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), _ptr(conv_w), H, d, K, chunk,
        _ptr(node_state), _ptr(node_conv), _ptr(o), flags, _stream(stream)))


def fork_readout(meta: Meta, h, D: int, w_opt, opt_off, p, flags: int = 0, stream=None):
    _check("fork_readout", load().fork_readout(meta.ref, _ptr(h), D, _ptr(w_opt), _ptr(opt_off), _ptr(p),
                                               flags, _stream(stream)))


def fork_readout_mlp_workspace_bytes(max_q: int, D: int, F: int) -> int:
    return load().fork_readout_mlp_workspace_bytes(max_q, D, F)


def fork_readout_mlp(meta: Meta, h, D: int, F: int, g1, w_gate, w_up, w_down, g2, w_opt, opt_off, p,
                     workspace, flags: int = 0, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("fork_readout_mlp", load().fork_readout_mlp(
        meta.ref, _ptr(h), D, F, _ptr(g1), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(g2), _ptr(w_opt),
        _ptr(opt_off), _ptr(p), _ptr(workspace), ws_bytes, flags, _stream(stream)))


def fork_pointwise_rows_workspace_bytes(T_cap: int, D: int, F: int) -> int:
    return load().fork_pointwise_rows_workspace_bytes(T_cap, D, F)


def fork_pointwise_rows(meta: Meta, h, D: int, F: int, g1, w_gate, w_up, w_down, g2, z, workspace, flags: int = 0,
                        stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("fork_pointwise_rows", load().fork_pointwise_rows(
        meta.ref, _ptr(h), D, F, _ptr(g1), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(g2), _ptr(z),
        _ptr(workspace), ws_bytes, flags, _stream(stream)))
