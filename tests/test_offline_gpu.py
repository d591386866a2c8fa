"""GPU parity of the streaming prefill (caches longer than one tensor-memory
tile, whole sequences with no cache), the gist-masked forward and the store of
compressed items, against the fp64 oracle.

Gist page ("把 item 压成 KV：gist 能不能用在相关性任务上"), 论文做了什么 and
在线的一次 attention: the item is forwarded once, offline, over [prompt; gist];
each layer keeps the K/V at the gist positions; online, the query attends to
that entry.  Under the training mask the same query rows come out of one
forward over [prompt; gist; query]."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_cached_kv_gb300 import binding, workloads
from parity_utils import compare, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


# (P, l, Hq, Hkv, d, block_len, blocks_per_pair, num_blocks): all beyond the
# tensor-memory kernel (more than 128 keys, or groups above 128 rows per tile)
LONG = [
    (2, 600, 14, 2, 64, 0, 0, 0),        # offline pass over [prompt; gist], no cache
    (1, 1000, 4, 4, 64, 0, 0, 0),        # MHA, long causal self-attention
    (2, 300, 32, 8, 128, 0, 0, 0),       # wide model, no cache
    (3, 40, 14, 2, 64, 256, 4, 12),      # 1024-row paged cache, 40 new tokens
    (2, 3, 14, 2, 64, 256, 16, 34),      # 4096-row cache, 3 new tokens
    (2, 300, 32, 8, 128, 8, 1, 5),       # gist item + long query
    (2, 7, 64, 1, 64, 100, 2, 5),        # group of 64: one token per tile
    (2, 33, 6, 1, 128, 130, 1, 4),       # group of 6: 60-row tiles, ragged everything
    (3, 129, 14, 2, 64, 0, 0, 0),        # one key past a tile edge
]


@pytest.mark.parametrize("shape", LONG, ids=lambda s: "P{}_l{}_Hq{}_Hkv{}_d{}_bl{}_b{}".format(*s[:7]))
@pytest.mark.parametrize("random_pos", [False, True])
def test_streaming_shapes_every_pair(shape, random_pos):
    P, l, Hq, Hkv, d, bl, bpp, nb = shape
    wl = workloads.make_custom(P, l, Hq, Hkv, d, bl, bpp, nb, num_layers=2, layer=1, device=DEV,
                               seed=sum(shape) % 997, random_pos=random_pos)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, layer=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref(wl, layer=1), str(shape))


def test_streaming_bad_block_zero_rows():
    P, l, bl, bpp, nb = 3, 20, 64, 4, 6
    wl = workloads.make_custom(P, l, 14, 2, 64, bl, bpp, nb, device=DEV, seed=3, use_table=True)
    wl.block_table[1, 2] = nb  # out of range
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.STATUS_BAD_BLOCK
    assert bool((got[1] == 0).all())
    keep = np.array([0, 2])
    compare(got[torch.from_numpy(keep).to(DEV)], oracle_ref(wl, pairs=keep), "good pairs")


def _masked_case(P, n, Hq, Hkv, d, k, seed, starts, pos=None):
    wl = workloads.make_custom(P, n, Hq, Hkv, d, 0, 0, 0, device=DEV, seed=seed)
    gs = torch.tensor(starts, dtype=torch.int32, device=DEV)
    posv = None if pos is None else torch.tensor(pos, dtype=torch.int32, device=DEV)
    return wl, gs, posv


@pytest.mark.parametrize("P,n,Hq,Hkv,d,k,starts,pos", [
    (3, 200, 14, 2, 64, 8, [0, 57, 150], None),
    (2, 333, 16, 4, 128, 16, [100, 3], [0, 4000]),
    (4, 90, 6, 6, 64, 1, [10, 0, 88, 45], None),
])
def test_gist_mask_forward(P, n, Hq, Hkv, d, k, starts, pos):
    wl, gs, posv = _masked_case(P, n, Hq, Hkv, d, k, 11 + n, starts, pos)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_gist_mask(wl.q, wl.k_new, wl.v_new, None, None, None, posv, gs, k,
                                          dims=wl.dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.gist_attn(wl.q, wl.k_new, wl.v_new, None, pos_offset=posv, dims=wl.dims,
                           gist_start=gs, gist_len=k)
    compare(got, ref, "gist mask")


def test_gist_mask_with_a_cache():
    """The mask over [cached; new] keys: a cached prefix counts as prompt."""
    P, l, bl, bpp, nb, k = 2, 50, 16, 2, 5, 4
    wl = workloads.make_custom(P, l, 14, 2, 64, bl, bpp, nb, device=DEV, seed=21, use_table=True)
    gs = torch.tensor([20, 32], dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_gist_mask(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, wl.block_table,
                                          None, gs, k, dims=wl.dims)
    ref = oracle.gist_attn(wl.q, wl.k_new, wl.v_new, wl.kv_pool, block_table=wl.block_table,
                           dims=wl.dims, gist_start=gs, gist_len=k)
    compare(got, ref, "gist mask over a cache")


def _bf16_from_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def test_kv_store_matches_oracle():
    P, n, Hkv, d, k, nb, L = 5, 40, 2, 128, 8, 9, 3
    wl = workloads.make_custom(P, n, Hkv, Hkv, d, k, 1, nb, num_layers=L, layer=2, device=DEV, seed=31)
    ids = torch.tensor([8, 0, 3, 5, 1], dtype=torch.int32, device=DEV)
    first = torch.tensor([32, 0, 7, 19, 25], dtype=torch.int32, device=DEV)
    spos = torch.tensor([32, 0, 7, 5000, 0], dtype=torch.int32, device=DEV)
    dims = dict(wl.dims, layer=2)
    for sp in (spos, None):
        pool = wl.kv_pool.clone()
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        binding.gist_kv_store(wl.k_new, wl.v_new, pool, ids, first, sp, dims=dims, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        want, rc = oracle.kv_store(wl.k_new, wl.v_new, wl.kv_pool, ids, first, sp, dims=dims)
        assert rc == 0
        got = oracle.bf16_bits(pool)
        diff = got != want
        assert not diff[:, :, 1].any()           # values bit for bit
        touched = np.zeros_like(diff)
        touched[ids.cpu().numpy(), 2, 0] = True
        assert not (diff & ~touched).any()        # nothing else written
        kg, kw = _bf16_from_bits(got).double(), _bf16_from_bits(want).double()
        ulp = torch.maximum(kw.abs(), torch.full_like(kw, 2.0 ** -126)) * 2.0 ** -7
        assert bool(((kg - kw).abs() <= ulp).all())  # keys within one bf16 ulp


def test_kv_store_rejects_rows_past_the_end():
    P, n, Hkv, d, k, nb = 3, 20, 2, 64, 8, 4
    wl = workloads.make_custom(P, n, Hkv, Hkv, d, k, 1, nb, device=DEV, seed=33)
    ids = torch.tensor([0, 1, 7], dtype=torch.int32, device=DEV)     # 7: bad block
    first = torch.tensor([12, 13, 0], dtype=torch.int32, device=DEV)  # 13 + 8 > 20
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    before = wl.kv_pool.clone()
    binding.gist_kv_store(wl.k_new, wl.v_new, wl.kv_pool, ids, first, None, dims=wl.dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.STATUS_BAD_BLOCK
    changed = torch.nonzero((wl.kv_pool != before).flatten(1).any(1)).flatten().tolist()
    assert changed == [0]


def test_offline_store_then_online_equals_masked_forward():
    """One layer end to end on the GPU.  Sequences [prompt j_p; gist k; query lq],
    right-padded: (a) the gist-masked forward; (b) the offline store of the gist
    rows (rotated at their own positions j_p .. j_p+k-1) into the pool; (c) the
    online pass of the query alone, numbered from j_p + k, against that entry.
    (c) equals (a) on the query rows up to the bf16 rounding of stored keys."""
    P, Hq, Hkv, d, k, lq = 4, 14, 2, 64, 8, 16
    js = [37, 120, 5, 200]
    n = max(js) + k + lq
    wl = workloads.make_custom(P, n, Hq, Hkv, d, 0, 0, 0, device=DEV, seed=41)
    gs = torch.tensor(js, dtype=torch.int32, device=DEV)
    full = binding.gist_attn_fwd_gist_mask(wl.q, wl.k_new, wl.v_new, None, None, None, None, gs, k,
                                           dims=wl.dims)
    pool = torch.zeros((P, 1, 2, Hkv, k, d), dtype=torch.bfloat16, device=DEV)
    ids = torch.arange(P, dtype=torch.int32, device=DEV)
    sdims = dict(wl.dims, block_len=k, blocks_per_pair=1, num_blocks=P)
    binding.gist_kv_store(wl.k_new, wl.v_new, pool, ids, gs, gs, dims=sdims)
    rows = torch.stack([torch.arange(j + k, j + k + lq, device=DEV) for j in js])  # [P, lq]

    def take(t):
        return torch.stack([t[p, rows[p]] for p in range(P)]).contiguous()

    q, kn, vn = take(wl.q), take(wl.k_new), take(wl.v_new)
    pos = gs + k
    odims = dict(wl.dims, n_new=lq, block_len=k, blocks_per_pair=1, num_blocks=P)
    online = binding.gist_attn_fwd(q, kn, vn, pool, ids, None, pos, dims=odims)
    torch.cuda.synchronize()
    # each against the oracle on its own inputs
    compare(full, oracle.gist_attn(wl.q, wl.k_new, wl.v_new, None, dims=wl.dims, gist_start=gs,
                                   gist_len=k), "masked forward")
    compare(online, oracle.gist_attn(q, kn, vn, pool, item_ids=ids, pos_offset=pos, dims=odims),
            "online pass")
    # and with each other on the query rows
    gap = (online.float() - take(full).float()).abs().max().item()
    assert gap < 2e-2, gap
