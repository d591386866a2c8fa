"""The C-ABI library without a GPU: it loads, exports every function the header
declares, rejects bad arguments on the host (nothing reaches CUDA), and its
byte-count helpers give the figures the pages print."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from attention_cached_kv_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load_library()


@pytest.fixture
def fake_ptrs(lib):
    """The rejection tests pass fake device addresses that only a call failing on
    the host never touches.  Where a GPU is visible a call that unexpectedly
    passed every check would launch on them, so these tests run without one."""
    try:
        import torch
        visible = torch.cuda.is_available()
    except Exception:  # pragma: no cover - torch is part of the environment
        visible = False
    if visible:
        pytest.skip("fake device addresses: host-only test")
    return lib


def header_functions():
    text = open(os.path.join(ROOT, "include", "gist_attn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(gist_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = header_functions()
    assert set(binding.EXPORTS) == set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_byte_helpers_match_page_figures(lib, golden):
    for row in golden["bytes_per_position"]:
        assert binding.kv_bytes_per_position(row["L"], row["Hkv"], row["d"], row["b"]) == row["bytes"]
    for row in golden["bytes_per_item"]:
        assert binding.kv_bytes_per_item(row["L"], row["Hkv"], row["d"], row["k"], row["b"]) == row["bytes"]
    for row in golden["request_kv"]:
        got = binding.kv_bytes_batch(row["B"], row["L"], row["S"], 32, row["H"] // 32, row["b"])
        assert got / 2 ** 30 == row["printed_GB"]
    assert binding.kv_bytes_per_position(-1, 2, 64, 2) == 0


BASE = dict(num_pairs=4, n_new=8, num_q_heads=14, num_kv_heads=2, head_dim=64, block_len=8,
            blocks_per_pair=1, num_blocks=16, num_layers=2, layer=1, rope_theta=1e4,
            softmax_scale=0.0)
P16 = 0x10000  # fake, 16-byte aligned device addresses: never dereferenced on a failing call


def call(lib, dims=BASE, q=P16, k=P16, v=P16, pool=P16, ids=P16, table=None, pos=None, out=P16,
         null_dims=False):
    D = None if null_dims else ctypes.byref(binding.make_dims(dims))
    V = ctypes.c_void_p
    return lib.gist_attn_fwd(V(q) if q else None, V(k) if k else None, V(v) if v else None,
                             V(pool) if pool else None, V(ids) if ids else None,
                             V(table) if table else None, V(pos) if pos else None,
                             V(out) if out else None, D, None)


@pytest.mark.parametrize("case,code", [
    (dict(null_dims=True), binding.ERR_NULL),
    (dict(q=0), binding.ERR_NULL),
    (dict(out=0), binding.ERR_NULL),
    (dict(pool=0), binding.ERR_NULL),
    (dict(ids=0), binding.ERR_NULL),
    (dict(table=P16), binding.ERR_DIMS),                       # both index arrays
    (dict(dims=dict(BASE, blocks_per_pair=2)), binding.ERR_DIMS),  # item ids need one block
    (dict(dims=dict(BASE, n_new=0)), binding.ERR_DIMS),
    (dict(dims=dict(BASE, num_kv_heads=3)), binding.ERR_DIMS),
    (dict(dims=dict(BASE, layer=2)), binding.ERR_DIMS),
    (dict(dims=dict(BASE, num_pairs=-1)), binding.ERR_DIMS),
    (dict(dims=dict(BASE, num_blocks=0)), binding.ERR_DIMS),
    (dict(dims=dict(BASE, rope_theta=0.0)), binding.ERR_DIMS),
    (dict(dims=dict(BASE, softmax_scale=-1.0)), binding.ERR_DIMS),
    (dict(dims=dict(BASE, softmax_scale=float("nan"))), binding.ERR_DIMS),
    (dict(dims=dict(BASE, head_dim=96)), binding.ERR_UNSUPPORTED),
    (dict(dims=dict(BASE, num_q_heads=600, num_kv_heads=2)), binding.ERR_UNSUPPORTED),
    (dict(q=P16 + 2), binding.ERR_ALIGN),
    (dict(out=P16 + 8), binding.ERR_ALIGN),
    (dict(pool=P16 + 4), binding.ERR_ALIGN),
    (dict(ids=P16 + 2), binding.ERR_ALIGN),
    (dict(pos=P16 + 1), binding.ERR_ALIGN),
])
def test_host_rejects_bad_arguments(fake_ptrs, case, code):
    lib = fake_ptrs
    assert call(lib, **case) == code


def test_empty_batch_launches_nothing(fake_ptrs):
    lib = fake_ptrs
    assert call(lib, dims=dict(BASE, num_pairs=0), q=0, k=0, v=0, out=0) == binding.OK


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, 1, 2, 3):
        assert binding.status_string(code)
    assert "block" in binding.status_string(binding.STATUS_BAD_BLOCK)
    assert "fp32" in binding.status_string(binding.STATUS_RANGE)


def test_gather_debug_rejects_bad_arguments(fake_ptrs):
    lib = fake_ptrs
    V = ctypes.c_void_p
    D = ctypes.byref(binding.make_dims(BASE))
    assert lib.gist_attn_gather_debug(V(P16), V(P16), None, None, D, None) == binding.ERR_NULL
    assert lib.gist_attn_gather_debug(V(P16), V(P16), None, V(P16 + 2), D, None) == binding.ERR_ALIGN
    assert lib.gist_attn_gather_debug(V(P16), None, None, V(P16), D, None) == binding.ERR_NULL


def test_gist_mask_rejects_bad_arguments(fake_ptrs):
    lib = fake_ptrs
    V = ctypes.c_void_p
    D0 = dict(BASE, block_len=0, blocks_per_pair=0, num_blocks=0)
    D = ctypes.byref(binding.make_dims(D0))
    f = lib.gist_attn_fwd_gist_mask
    # gist_start is required; gist_len must not be negative; alignment of gist_start
    assert f(V(P16), V(P16), V(P16), None, None, None, None, None, 4, V(P16), D, None) == binding.ERR_NULL
    assert f(V(P16), V(P16), V(P16), None, None, None, None, V(P16), -1, V(P16), D, None) == binding.ERR_DIMS
    assert f(V(P16), V(P16), V(P16), None, None, None, None, V(P16 + 2), 4, V(P16), D, None) == binding.ERR_ALIGN
    Dg = ctypes.byref(binding.make_dims(dict(D0, num_q_heads=130, num_kv_heads=1)))
    assert f(V(P16), V(P16), V(P16), None, None, None, None, V(P16), 4, V(P16), Dg, None) == binding.ERR_UNSUPPORTED


def test_kv_store_rejects_bad_arguments(fake_ptrs):
    lib = fake_ptrs
    V = ctypes.c_void_p
    f = lib.gist_kv_store
    ok = dict(BASE, n_new=12, block_len=8, blocks_per_pair=1)
    D = ctypes.byref(binding.make_dims(ok))
    assert f(V(P16), V(P16), V(P16), V(P16), None, None, D, None) == binding.ERR_NULL
    assert f(V(P16), V(P16), None, V(P16), V(P16), None, D, None) == binding.ERR_NULL
    assert f(V(P16), V(P16), V(P16), V(P16), V(P16 + 1), None, D, None) == binding.ERR_ALIGN
    for bad in (dict(ok, blocks_per_pair=2), dict(ok, block_len=13), dict(ok, block_len=0)):
        Db = ctypes.byref(binding.make_dims(bad))
        assert f(V(P16), V(P16), V(P16), V(P16), V(P16), None, Db, None) == binding.ERR_DIMS
    Dz = ctypes.byref(binding.make_dims(dict(ok, num_pairs=0)))
    assert f(None, None, None, None, None, None, Dz, None) == binding.OK


def test_projections_reject_bad_arguments(fake_ptrs):
    lib = fake_ptrs
    V = ctypes.c_void_p
    D = ctypes.byref(binding.make_dims(dict(BASE, n_new=64)))
    q = lib.gist_qkv_rope
    assert q(None, V(P16), None, V(P16), V(P16), V(P16), 256, D, None) == binding.ERR_NULL
    assert q(V(P16), V(P16), None, V(P16), V(P16), V(P16), 0, D, None) == binding.ERR_DIMS
    assert q(V(P16 + 2), V(P16), None, V(P16), V(P16), V(P16), 256, D, None) == binding.ERR_ALIGN
    pre = ctypes.byref(binding.make_dims(dict(BASE, n_new=64, flags=binding.FLAG_PREROTATED)))
    assert q(V(P16), V(P16), None, V(P16), V(P16), V(P16), 256, pre, None) == binding.ERR_DIMS
    odd = ctypes.byref(binding.make_dims(dict(BASE, n_new=64, num_q_heads=3, num_kv_heads=1)))
    assert q(V(P16), V(P16), None, V(P16), V(P16), V(P16), 256, odd, None) == binding.ERR_UNSUPPORTED
    short = ctypes.byref(binding.make_dims(dict(BASE, n_new=4)))
    assert q(V(P16), V(P16), None, V(P16), V(P16), V(P16), 256, short, None) == binding.ERR_UNSUPPORTED
    # the table of token angles must fit shared memory: l <= 1904 (d = 64), l <= 936 (d = 128)
    for dd in (dict(BASE, n_new=1905), dict(BASE, n_new=937, head_dim=128, num_q_heads=8)):
        long_ = ctypes.byref(binding.make_dims(dd))
        assert q(V(P16), V(P16), None, V(P16), V(P16), V(P16), 256, long_, None) == binding.ERR_UNSUPPORTED
    o = lib.gist_out_proj
    assert o(V(P16), None, V(P16), 256, D, None) == binding.ERR_NULL
    assert o(V(P16), V(P16), V(P16), 200, D, None) == binding.ERR_UNSUPPORTED  # not a multiple of 128
    bad_flags = ctypes.byref(binding.make_dims(dict(BASE, flags=4)))
    assert lib.gist_attn_fwd(V(P16), V(P16), V(P16), V(P16), V(P16), None, None, V(P16), bad_flags,
                             None) == binding.ERR_DIMS


def _dims(**kw):
    d = dict(num_pairs=12800, n_new=256, num_q_heads=14, num_kv_heads=2, head_dim=64, block_len=8,
             blocks_per_pair=1, num_blocks=100000, num_layers=2, layer=0, rope_theta=1e4,
             softmax_scale=0.0)
    d.update(kw)
    return d


def test_workspace_bytes(lib):
    """The staged path's workspace: the angles of q (a (cos, sin) pair per
    frequency for every pair and every new-token index) plus the [cached; new]
    key and value sequences of every pair, each part rounded up to 256 bytes; 0
    where a shape runs without one, and for invalid dimensions."""
    def up(x):
        return (x + 255) // 256 * 256

    for P, l, Hq, Hkv, C in [(12800, 300, 14, 2, 8), (3, 250, 7, 1, 64), (5, 300, 16, 2, 1)]:
        d = _dims(num_pairs=P, n_new=l, num_q_heads=Hq, num_kv_heads=Hkv, block_len=C)
        want = up(P * 32 * 8) + up(l * 32 * 8) + 2 * up(P * (C + l) * Hkv * 64 * 2)
        assert binding.workspace_bytes(d) == want, (P, l, C)
    assert binding.workspace_bytes(_dims(n_new=64)) == 0            # 72 keys: single-pass kernel
    assert binding.workspace_bytes(_dims()) == 0                    # 264 keys: single pass, 512 TMEM columns
    assert binding.workspace_bytes(_dims(n_new=1)) == 0             # decode
    assert binding.workspace_bytes(_dims(head_dim=128)) == 0        # d = 128: streaming kernel
    assert binding.workspace_bytes(_dims(num_pairs=0)) == 0
    assert binding.workspace_bytes(_dims(num_kv_heads=3)) == 0      # invalid: 14 % 3
    assert binding.workspace_bytes(_dims(block_len=0, blocks_per_pair=0, flags=1)) == 0  # pre-rotated, no cache
    assert binding.workspace_bytes(_dims(n_new=300, block_len=0, blocks_per_pair=0)) > 0  # raw inputs, no cache
