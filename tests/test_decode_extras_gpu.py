"""GPU parity of the decode-step extras: per-block attention mass (the
eviction statistic of the suffix-cache page, §5 第三步) and the KV append of
the KV page's decode step, against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_cached_kv_gb300 import binding, workloads
from parity_utils import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


def _paged(P, H, d, bl, bpp, nb, seed, L=2, layer=1, random_pos=False, G=1):
    return workloads.make_custom(P, 1, H * G, H, d, bl, bpp, nb, num_layers=L, layer=layer, device=DEV,
                                 seed=seed, random_pos=random_pos, use_table=True)


@pytest.mark.parametrize("G", [1, 7, 16])
@pytest.mark.parametrize("d,bl,bpp,random_pos", [(128, 256, 4, False), (64, 16, 9, True), (128, 32, 7, True)])
def test_block_mass(d, bl, bpp, random_pos, G):
    """One mass per query head and block, for MHA (G = 1) and GQA groups of 7
    and 16 query heads per KV head."""
    wl = _paged(5, 4 if G == 1 else 2, d, bl, bpp, 11, seed=bl + bpp + G, random_pos=random_pos, G=G)
    dims = dict(wl.dims, layer=1)
    out, mass = binding.gist_attn_fwd_block_mass(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.block_table,
                                                 wl.pos_offset, dims=dims)
    torch.cuda.synchronize()
    pool1 = wl.kv_pool[:, 1:2].contiguous()
    ref, w = oracle.gist_attn(wl.q, wl.k_new, wl.v_new, pool1, block_table=wl.block_table,
                              pos_offset=wl.pos_offset, dims=dict(dims, num_layers=1, layer=0),
                              want_weights=True)
    compare(out, ref, "decode output")
    want = oracle.block_mass(w, bpp, bl)
    got = mass.double().cpu().numpy()
    assert np.all(np.abs(got - want) <= 1e-4 + 1e-3 * np.abs(want)), np.abs(got - want).max()
    assert np.all(got.sum(-1) < 1.0)


def test_append_then_next_step():
    """Step t attends with its own k_t/v_t, appends them; step t+1 reads them
    from the cache as its last cached row."""
    P, H, d, bl, nb, L = 4, 2, 64, 16, 12, 3
    wl = _paged(P, H, d, bl, 3, nb, seed=7, L=L, layer=2)
    table = wl.block_table
    t = 2 * bl + 5  # the new token's position == its slot
    slot = torch.full((P,), t, dtype=torch.int32, device=DEV)
    dims = dict(wl.dims, layer=2)
    before = wl.kv_pool.clone()
    binding.gist_kv_append(wl.k_new, wl.v_new, wl.kv_pool, table, slot, None, dims=dims)
    torch.cuda.synchronize()
    want, rc = oracle.kv_append(wl.k_new, wl.v_new, before, table, slot, dims=dims)
    assert rc == 0
    got = oracle.bf16_bits(wl.kv_pool)
    # V rows and every untouched element bit-exact; K rows within one bf16 ulp
    diff = got != want
    assert not diff[:, :, 1].any()
    k_got = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).double()
    k_want = torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).double()
    ulp = torch.maximum(k_want.abs(), torch.full_like(k_want, 2.0 ** -126)) * 2.0 ** -7
    assert bool(((k_got - k_want).abs() <= ulp)[:, :, 0].all())
    touched = np.zeros_like(diff)
    for p in range(P):
        blk = int(table[p, t // bl])
        touched[blk, 2, 0, :, t % bl] = True
    assert not (diff & ~touched).any()
    # the next step: a cache of t+1 rows (the appended row included), new token at t+1
    nxt = workloads.make_custom(P, 1, H, H, d, bl, 3, nb, num_layers=L, layer=2, device=DEV, seed=8,
                                use_table=True)
    pos = torch.full((P,), t + 1, dtype=torch.int32, device=DEV)
    out = binding.gist_attn_fwd(nxt.q, nxt.k_new, nxt.v_new, wl.kv_pool, None, table, pos,
                                dims=dict(dims, blocks_per_pair=3))
    ref = oracle.gist_attn(nxt.q, nxt.k_new, nxt.v_new, torch.from_numpy(want.view(np.int16)).view(torch.bfloat16),
                           block_table=table, pos_offset=pos, dims=dict(dims, blocks_per_pair=3))
    compare(out, ref, "next step on the appended cache")


def test_append_rejects_bad_slot():
    wl = _paged(3, 2, 64, 16, 2, 5, seed=9)
    slot = torch.tensor([0, 32, 5], dtype=torch.int32, device=DEV)  # 32 is past the table
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    before = wl.kv_pool.clone()
    binding.gist_kv_append(wl.k_new, wl.v_new, wl.kv_pool, wl.block_table, slot, None, dims=wl.dims,
                           status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.STATUS_BAD_BLOCK
    changed_blocks = torch.nonzero((wl.kv_pool != before).flatten(1).any(1)).flatten().tolist()
    allowed = {int(wl.block_table[0, 0]), int(wl.block_table[2, 0])}
    assert set(changed_blocks) <= allowed


def test_a_wait_that_runs_out_reports_timeout_and_leaves_the_context_usable():
    """GIST_ATTN_FLAG_TEST_WITHHOLD makes the paged decode withhold its first
    chunk's copy (nothing faults: a flag that nothing sets): every CTA's bounded
    wait runs out after 20 ms, it waits for the copies it did issue and reports
    GIST_ATTN_STATUS_TIMEOUT.  The call ends in bounded time and the next call on
    the same context is correct."""
    import time
    wl = _paged(4, 4, 128, 64, 3, 9, seed=21)
    dims = dict(wl.dims, layer=1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.time()
    binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, wl.block_table, None,
                          dims=dict(dims, flags=binding.FLAG_TEST_WITHHOLD), status=status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) & binding.STATUS_TIMEOUT
    assert elapsed < 5.0, elapsed
    status.zero_()
    out = binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, wl.block_table, None,
                                dims=dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pool1 = wl.kv_pool[:, 1:2].contiguous()
    ref = oracle.gist_attn(wl.q, wl.k_new, wl.v_new, pool1, block_table=wl.block_table,
                           dims=dict(dims, num_layers=1, layer=0))
    compare(out, ref, "after the timeout")
