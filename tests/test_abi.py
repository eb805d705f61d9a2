"""The C-ABI library builds for sm_103a, loads, and exports every declared entry point.

No compute call is made here: only host-side argument checks, which return
before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from tree_forked_hybrid_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "forkattn.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t)\s+(fork_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    from tree_forked_hybrid_gb300 import fork as F
    return F.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("fork_build_meta", "fork_attn", "fork_gdn_trunk", "fork_gdn_branches", "fork_readout",
                 "fork_meta_bytes", "fork_meta_init", "fork_read_status", "fork_attn_workspace_bytes",
                 "fork_forest_plan", "fork_build_forest_meta", "fork_gdn_forest"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_meta_sizes_and_handle_checks(lib):
    from tree_forked_hybrid_gb300 import fork as F
    assert lib.fork_meta_bytes(0, 1, 1) == 0
    assert lib.fork_meta_bytes(16, 0, 1) == 0
    n = lib.fork_meta_bytes(128, 4, 8)
    assert n > 0 and n % 4 == 0
    assert lib.fork_meta_bytes(256, 4, 8) > n
    h = F.fork_meta()
    buf = ctypes.create_string_buffer(n + 16)
    addr = (ctypes.addressof(buf) + 15) & ~15
    assert lib.fork_meta_init(ctypes.byref(h), ctypes.c_void_p(addr), n, 128, 4, 8, 32) == 0
    assert h.T_cap == 128 and h.tile_tokens == 32
    assert lib.fork_meta_init(ctypes.byref(h), ctypes.c_void_p(addr), n - 4, 128, 4, 8, 32) == 1
    assert lib.fork_meta_init(ctypes.byref(h), ctypes.c_void_p(addr), n, 128, 4, 8, 24) == 1
    assert lib.fork_meta_init(ctypes.byref(h), ctypes.c_void_p(addr + 4), n, 128, 4, 8, 32) == 1
    assert lib.fork_meta_init(None, ctypes.c_void_p(addr), n, 128, 4, 8, 32) == 1


def test_argument_errors_return_before_any_launch(lib):
    from tree_forked_hybrid_gb300 import fork as F
    n = lib.fork_meta_bytes(128, 4, 8)
    buf = ctypes.create_string_buffer(n + 16)
    addr = (ctypes.addressof(buf) + 15) & ~15
    h = F.fork_meta()
    assert lib.fork_meta_init(ctypes.byref(h), ctypes.c_void_p(addr), n, 128, 4, 8, 32) == 0
    ref = ctypes.byref(h)
    fake = ctypes.c_void_p(0x1000)
    # capacity: more requests than the handle allows
    assert lib.fork_build_meta(ref, fake, 5, 0, 0, None) == 2
    assert lib.fork_build_meta(ref, fake, 2, 9, 0, None) == 2
    assert lib.fork_build_meta(ref, fake, -1, 0, 0, None) == 1
    assert lib.fork_build_meta(ref, None, 1, 0, 0, None) == 1
    # attention: null tensors, bad head dim, GQA group not matching the tile, misalignment
    assert lib.fork_attn(ref, None, fake, fake, fake, 4, 1, 128, 0, 0.0, 0.1, None, None, 0, None, 0, 0, None) == 1
    assert lib.fork_attn(ref, fake, fake, fake, fake, 4, 1, 96, 0, 0.0, 0.1, None, None, 0, None, 0, 0, None) == 1
    # 16 q-heads per kv head x 32-token tiles = 512 rows: neither one nor two 128-row tiles
    assert lib.fork_attn(ref, fake, fake, fake, fake, 16, 1, 128, 0, 0.0, 0.1, None, None, 0, None, 0, 0, None) == 1
    # two 128-row tiles per work item are for the tcgen05 kernel only
    assert lib.fork_attn(ref, fake, fake, fake, fake, 8, 1, 128, 0, 0.0, 0.1, None, None, 0, None, 0, 4, None) == 1
    assert lib.fork_attn(ref, fake, fake, fake, fake, 6, 4, 128, 0, 0.0, 0.1, None, None, 0, None, 0, 0, None) == 1
    odd = ctypes.c_void_p(0x1002)
    assert lib.fork_attn(ref, odd, fake, fake, fake, 4, 1, 128, 0, 0.0, 0.1, None, None, 0, None, 0, 0, None) == 1
    assert lib.fork_attn(ref, fake, fake, fake, fake, 4, 1, 128, -1, 0.0, 0.1, None, None, 0, None, 0, 0, None) == 1
    # rope on without a workspace
    assert lib.fork_attn(ref, fake, fake, fake, fake, 4, 1, 128, 0, 10000.0, 0.1, None, None, 0, None, 0, 0,
                         None) in (1, 3, 4)
    # gdn: only chunk 64, width 4, d in {64,128}
    assert lib.fork_gdn_trunk(ref, fake, fake, fake, fake, fake, fake, 2, 128, 4, 32, None, None, fake, fake,
                              None, None, fake, 0, None) == 1
    assert lib.fork_gdn_trunk(ref, fake, fake, fake, fake, fake, fake, 2, 128, 3, 64, None, None, fake, fake,
                              None, None, fake, 0, None) == 1
    assert lib.fork_gdn_trunk(ref, fake, fake, fake, fake, fake, fake, 2, 128, 4, 64, None, None, fake, fake,
                              fake, None, fake, 0, None) == 1
    assert lib.fork_gdn_branches(ref, fake, fake, fake, fake, fake, fake, 2, 32, 4, 64, fake, fake, fake, 0,
                                 None) == 1
    assert lib.fork_readout(ref, fake, 100, fake, fake, fake, 0, None) == 1
    assert lib.fork_readout(ref, None, 128, fake, fake, fake, 0, None) == 1
    # token forests: attention only at d = 128, without prefix rows, not on the warp-MMA kernel
    forest = F.FORK_FOREST
    assert lib.fork_attn(ref, fake, fake, fake, fake, 4, 1, 64, 0, 0.0, 0.1, None, None, 0, None, 0, forest,
                         None) == 1
    assert lib.fork_attn(ref, fake, fake, fake, fake, 4, 1, 128, 0, 0.0, 0.1, fake, fake, 8, None, 0, forest,
                         None) == 1
    assert lib.fork_attn(ref, fake, fake, fake, fake, 4, 1, 128, 0, 0.0, 0.1, None, None, 0, None, 0,
                         forest | F.FORK_WARP_MMA, None) == 1
    # forest levels: d = 128, a node range inside the capacity, both state arrays
    gf = lambda first, count, d, st, flags=0: lib.fork_gdn_forest(  # noqa: E731
        ref, first, count, fake, fake, fake, fake, fake, fake, 2, d, 4, 64, st, fake, fake, flags, None)
    assert gf(0, 2, 64, fake) == 1
    assert gf(0, 2, 128, None) == 1
    assert gf(-1, 2, 128, fake) == 1
    assert gf(0, -1, 128, fake) == 1
    assert gf(3, 2, 128, fake) == 1       # past max_req = 4
    assert gf(0, 2, 128, fake, F.FORK_WARP_MMA) == 1


def test_readout_mlp_argument_errors_and_workspace_size(lib):
    from tree_forked_hybrid_gb300 import fork as F
    n = lib.fork_meta_bytes(128, 4, 8)
    buf = ctypes.create_string_buffer(n + 16)
    addr = (ctypes.addressof(buf) + 15) & ~15
    h = F.fork_meta()
    assert lib.fork_meta_init(ctypes.byref(h), ctypes.c_void_p(addr), n, 128, 4, 8, 32) == 0
    ref = ctypes.byref(h)
    fake = ctypes.c_void_p(0x1000)
    ws_bytes = lib.fork_readout_mlp_workspace_bytes(8, 256, 512)
    # Mpad = 64 rows: normalised rows (bf16), activations (bf16), y (float32), and for the
    # tensor-core products (D a multiple of 128, F of 256) the partial products, max(2F, 4D)
    # float32 values per row
    assert ws_bytes == 64 * 256 * 2 + 64 * 512 * 2 + 64 * 256 * 4 + 64 * max(2 * 512, 4 * 256) * 4
    # shapes the tensor-core tiles do not divide: no partial products
    assert lib.fork_readout_mlp_workspace_bytes(8, 192, 512) == 64 * 192 * 2 + 64 * 512 * 2 + 64 * 192 * 4
    assert lib.fork_readout_mlp_workspace_bytes(8, 100, 512) == 0     # D not a multiple of 64
    assert lib.fork_readout_mlp_workspace_bytes(8, 256, 96) == 0      # F not a multiple of 64
    assert lib.fork_readout_mlp_workspace_bytes(8, 16384, 512) == 0   # D above 8192
    args = [ref, fake, 256, 512, fake, fake, fake, fake, fake, fake, fake, fake, fake, ws_bytes, 0, None]
    good = list(args)
    for i in (1, 4, 5, 6, 7, 8, 9, 10, 11, 12):  # each pointer null in turn
        a = list(good)
        a[i] = None
        assert lib.fork_readout_mlp(*a) == 1
    a = list(good)
    a[2] = 200  # D
    assert lib.fork_readout_mlp(*a) == 1
    a = list(good)
    a[13] = ws_bytes - 1  # short workspace
    assert lib.fork_readout_mlp(*a) == 1
    a = list(good)
    a[5] = ctypes.c_void_p(0x1008)  # misaligned weights
    assert lib.fork_readout_mlp(*a) == 1
    for i in (4, 8):  # gains read as 16-byte vectors
        a = list(good)
        a[i] = ctypes.c_void_p(0x1004)
        assert lib.fork_readout_mlp(*a) == 1
