"""gist_attn_fwd_noalloc: the staged attention for callers that cannot allocate
device memory where they call it (a plugin whose host program owns every
device allocation and hands it no workspace, or a latency-critical loop that
must not pay cudaMalloc's implicit synchronisation).  Its scratch is a fixed
device array inside the library, so these tests check that two calls in a row
-- the second one reading an array the first one left full -- give what
gist_attn_fwd_ws gives with a caller-owned workspace, within the parity
tolerance.  The file is named to be collected last."""
from __future__ import annotations

import ctypes

import pytest
import torch

from attention_cached_kv_gb300 import binding, workloads
from parity_utils import compare

DEV = "cuda"

# (P, l, Hq, Hkv, block_len, blocks_per_pair, num_blocks, random_pos): both take
# the staged path (d = 64, more than 288 keys), the second through a block table
CASES = [(4, 300, 14, 2, 8, 1, 20, False), (3, 290, 16, 2, 16, 2, 11, True)]


def _with_workspace(wl):
    n = binding.workspace_bytes(wl.dims)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    return binding.gist_attn_fwd_ws(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids,
                                    wl.block_table, wl.pos_offset, None, ws, dims=wl.dims)


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    for i, (P, l, Hq, Hkv, bl, bpp, nb, rpos) in enumerate(CASES):
        wl = workloads.make_custom(P, l, Hq, Hkv, 64, bl, bpp, nb, device=DEV, seed=40 + i,
                                   random_pos=rpos)
        need = binding.workspace_bytes(wl.dims)
        assert 0 < need <= binding.NOALLOC_SCRATCH_BYTES
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = torch.empty_like(wl.q)
        got = binding.gist_attn_fwd_noalloc(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids,
                                            wl.block_table, wl.pos_offset, out, dims=wl.dims,
                                            status=status)
        ref = _with_workspace(wl)
        torch.cuda.synchronize()
        assert got.data_ptr() == out.data_ptr()
        assert int(status.item()) == 0
        compare(got, ref.double().cpu().numpy(), f"no-alloc call {i + 1}")


def test_too_much_scratch_is_rejected_on_the_host():
    """Dimensions whose staged path needs more than the fixed array return
    GIST_ATTN_ERR_SCRATCH before anything reaches CUDA (fake device addresses,
    never dereferenced; host-only, so skipped where a GPU is visible)."""
    if torch.cuda.is_available():
        pytest.skip("fake device addresses: host-only test")
    lib = binding.load_library()
    dims = dict(num_pairs=1024, n_new=300, num_q_heads=14, num_kv_heads=2, head_dim=64,
                block_len=8, blocks_per_pair=1, num_blocks=16, num_layers=1, layer=0,
                rope_theta=1e4, softmax_scale=0.0)
    assert binding.workspace_bytes(dims) > binding.NOALLOC_SCRATCH_BYTES
    V, fake = ctypes.c_void_p, ctypes.c_void_p(0x10000)
    D = binding.make_dims(dims)
    rc = lib.gist_attn_fwd_noalloc(fake, fake, fake, fake, fake, None, None, fake, ctypes.byref(D),
                                   None)
    assert rc == binding.ERR_SCRATCH
    assert "scratch" in binding.status_string(rc)
    # invalid dimensions keep their usual codes
    D = binding.make_dims(dict(dims, n_new=0))
    assert lib.gist_attn_fwd_noalloc(fake, fake, fake, fake, fake, None, None, fake,
                                     ctypes.byref(D), None) == binding.ERR_DIMS
    assert lib.gist_attn_fwd_noalloc(fake, fake, fake, fake, fake, None, None, fake, None,
                                     None) == binding.ERR_NULL
