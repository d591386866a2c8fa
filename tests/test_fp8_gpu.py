"""GPU parity of the E4M3 (fp8) KV pool path against the fp64 oracle, which
dequantises every cached element exactly (e4m3 value times its block's scale)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from attention_cached_kv_gb300 import binding, workloads
from parity_utils import compare, oracle_ref_fp8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    yield
    torch.cuda.empty_cache()


@pytest.mark.parametrize("d,bl,bpp,random_pos", [(128, 256, 2, False), (64, 16, 5, True),
                                                 (128, 32, 3, True), (64, 64, 1, False)])
def test_fp8_decode_every_sequence(d, bl, bpp, random_pos):
    wl = workloads.make_custom(6, 1, 8, 8, d, bl, bpp, 9, num_layers=3, layer=2, device=DEV,
                               seed=bl + bpp, random_pos=random_pos, use_table=True)
    pool8, scale = workloads.make_fp8_pool(wl, seed=bl)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, None, wl.block_table,
                                      wl.pos_offset, dims=dict(wl.dims, layer=2), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref_fp8(wl, pool8, scale, layer=2), f"fp8 d={d} bl={bl}")


@pytest.mark.parametrize("P,Hq,Hkv,d,bl,bpp,rpos", [
    (9, 14, 2, 64, 8, 2, False),    # the query-gisted shape: 7 heads, 16 cached keys
    (5, 32, 2, 64, 8, 4, True),     # 16 heads, 32 cached keys
    (6, 16, 4, 128, 8, 3, True),    # d = 128, 24 cached keys
    (7, 14, 2, 64, 16, 1, False),   # item ids, one 16-row block
])
def test_fp8_short_decode_every_pair(P, Hq, Hkv, d, bl, bpp, rpos):
    """E4M3 pools behind the short decode (GQA groups, caches of at most 32 keys)."""
    wl = workloads.make_custom(P, 1, Hq, Hkv, d, bl, bpp, 11, num_layers=2, layer=1, device=DEV,
                               seed=P + bl, random_pos=rpos)
    pool8, scale = workloads.make_fp8_pool(wl, seed=P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, wl.item_ids,
                                      wl.block_table, wl.pos_offset, dims=dict(wl.dims, layer=1),
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref_fp8(wl, pool8, scale, layer=1), f"fp8 short G={Hq // Hkv} d={d}")


@pytest.mark.parametrize("shape", ["short", "paged", "gqa", "prefill"])
@pytest.mark.parametrize("magnitude", [1e-2, 1e-4])
def test_fp8_small_scales(shape, magnitude):
    """Scales near amax / 448 of real activations (1e-2, 1e-4), spread over two
    decades per block: the weights must not lose precision to them."""
    if shape == "short":
        wl = workloads.make_custom(6, 1, 14, 2, 64, 8, 2, 9, device=DEV, seed=4)
    elif shape == "gqa":
        wl = workloads.make_custom(4, 1, 16, 4, 128, 32, 3, 9, device=DEV, seed=4, use_table=True)
    elif shape == "prefill":
        wl = workloads.make_custom(4, 12, 14, 2, 64, 8, 2, 9, device=DEV, seed=4, use_table=True)
    else:
        wl = workloads.make_custom(4, 1, 8, 8, 128, 32, 3, 9, device=DEV, seed=4, use_table=True)
    pool8, scale = workloads.make_fp8_pool(wl, seed=3)
    g = torch.Generator(device=DEV).manual_seed(5)
    scale = scale * magnitude * torch.pow(10.0, -2.0 * torch.rand(scale.shape, generator=g, device=DEV))
    # values large enough that the result is not just the new token's own value
    wl.q.mul_(1.0 / magnitude ** 0.5)
    wl.k_new.mul_(magnitude ** 0.5)
    wl.v_new.mul_(magnitude)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, None, wl.block_table,
                                      None, dims=wl.dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle_ref_fp8(wl, pool8, scale)
    # the tolerance is relative to the output's scale: compare in units of it
    s = float(np.abs(ref).max())
    compare(got / s, ref / s, f"fp8 {shape} scales ~{magnitude}")


def test_fp8_qgist_workload_sampled():
    """The query-gisted workload (25,000 pairs, l = 1 against 8 + 8 cached keys)
    read from an E4M3 pool, as the benchmark's --kv fp8 row times it."""
    wl = workloads.make("qgist", device=DEV, num_layers=2)
    pool8, scale = workloads.make_fp8_pool(wl)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, None, wl.block_table,
                                      None, dims=dict(wl.dims, layer=1), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.sort(np.random.default_rng(1).choice(wl.dims["num_pairs"], 400, replace=False))
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref_fp8(wl, pool8, scale, layer=1, pairs=sel),
            "fp8 qgist")
    del wl, pool8, got
    torch.cuda.empty_cache()


@pytest.mark.parametrize("P,Hq,Hkv,d,bl,bpp,rpos", [
    (4, 32, 8, 128, 256, 2, False),   # GQA 4:1 over two 256-token blocks
    (3, 14, 2, 64, 32, 3, True),      # the gist model's 7:1 groups, 96 keys
    (2, 32, 2, 128, 16, 5, True),     # 16 heads per KV head
    (3, 32, 8, 128, 16, 21, True),    # 21 chunks over eight warps: a ragged last round
    (2, 16, 4, 64, 16, 13, False),    # d = 64, two stages per warp, 13 chunks
])
def test_fp8_gqa_paged_decode(P, Hq, Hkv, d, bl, bpp, rpos):
    """E4M3 pools behind the long GQA decode (more than 32 cached keys, groups
    of 2..16 query heads)."""
    wl = workloads.make_custom(P, 1, Hq, Hkv, d, bl, bpp, 9, num_layers=2, layer=1, device=DEV,
                               seed=bl + bpp, random_pos=rpos, use_table=True)
    pool8, scale = workloads.make_fp8_pool(wl, seed=bl)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, None, wl.block_table,
                                      wl.pos_offset, dims=dict(wl.dims, layer=1), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref_fp8(wl, pool8, scale, layer=1), f"fp8 gqa G={Hq // Hkv} d={d}")


def test_fp8_paged_workload_sampled():
    wl = workloads.make("paged", device=DEV, num_layers=4)
    pool8, scale = workloads.make_fp8_pool(wl)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, None, wl.block_table,
                                      None, dims=dict(wl.dims, layer=3))
    sel = np.arange(0, 32, 3)
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref_fp8(wl, pool8, scale, layer=3, pairs=sel),
            "fp8 paged")


def test_fp8_paged_gqa_workload_sampled():
    """The paged GQA workload (32 sequences x 4096 cached tokens, 32 / 8 heads,
    d = 128) from an E4M3 pool, in the launch configuration the benchmark's
    --kv fp8 row times; the oracle checks every fourth sequence."""
    wl = workloads.make("paged_gqa", device=DEV, num_layers=2)
    pool8, scale = workloads.make_fp8_pool(wl)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, None, wl.block_table,
                                      None, dims=dict(wl.dims, layer=1), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.arange(1, 32, 4)
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref_fp8(wl, pool8, scale, layer=1, pairs=sel),
            "fp8 paged gqa")
    assert torch.isfinite(got.float()).all()
    del wl, pool8, got
    torch.cuda.empty_cache()


def test_fp8_unsupported_shapes_are_refused():
    """Four new tokens behind 320 cached keys: more keys than a tensor-core tile
    holds, and not a decode step."""
    wl = workloads.make_custom(2, 4, 8, 2, 64, 160, 2, 3, device=DEV)
    pool8, scale = workloads.make_fp8_pool(wl)
    with pytest.raises(binding.GistAttnError) as e:
        binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, wl.item_ids,
                                    wl.block_table, None, dims=wl.dims)
    assert e.value.code == binding.ERR_UNSUPPORTED


# l >= 2: the tensor-core prefill dequantises the cached rows in its K/V warps
PREFILL = [
    (4, 12, 14, 2, 64, 8, 1, True),     # the gist model: 8 item-gist keys, 12 new tokens
    (3, 20, 32, 8, 128, 8, 1, False),   # the wide model's heads
    (3, 40, 14, 2, 64, 16, 3, True),    # three 16-row blocks, several tiles per unit
    (3, 16, 14, 2, 64, 32, 2, False),   # one tile per unit (three K/V warps), 80 keys
    (2, 64, 14, 2, 64, 32, 2, True),    # 128 keys: the two-level angle table
    (2, 256, 14, 2, 64, 8, 4, False),   # 288 keys per tile
]


@pytest.mark.parametrize("P,l,Hq,Hkv,d,bl,bpp,rpos", PREFILL, ids=lambda v: str(v))
def test_fp8_prefill_every_pair(P, l, Hq, Hkv, d, bl, bpp, rpos):
    wl = workloads.make_custom(P, l, Hq, Hkv, d, bl, bpp, 9, num_layers=2, layer=1, device=DEV,
                               seed=l + bl, random_pos=rpos)
    pool8, scale = workloads.make_fp8_pool(wl, seed=l)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, wl.item_ids,
                                      wl.block_table, wl.pos_offset, dims=dict(wl.dims, layer=1),
                                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref_fp8(wl, pool8, scale, layer=1), f"fp8 prefill l={l} C={bl * bpp} d={d}")


def test_fp8_prefill_prerotated():
    """q and k_new that arrive rotated (GIST_ATTN_FLAG_PREROTATED, the fused
    projection's output): S runs in bf16, so the cached keys dequantise to bf16."""
    wl = workloads.make_custom(3, 20, 14, 2, 64, 16, 2, 7, num_layers=2, layer=1, device=DEV, seed=23,
                               random_pos=True)
    pool8, scale = workloads.make_fp8_pool(wl, seed=23)
    wl.dims = dict(wl.dims, layer=1, flags=binding.FLAG_PREROTATED)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, wl.item_ids,
                                      wl.block_table, wl.pos_offset, dims=wl.dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref_fp8(wl, pool8, scale, layer=1), "fp8 prefill pre-rotated")


def test_fp8_prefill_keys_past_the_f16_range():
    """A block whose K scale (1e5) dequantises keys past the f16 range: the rows
    that read them are recomputed in fp32 from the E4M3 bytes and match the
    oracle; the status word stays clear."""
    wl = workloads.make_custom(4, 12, 14, 2, 64, 8, 1, 6, num_layers=2, layer=1, device=DEV, seed=9)
    pool8, scale = workloads.make_fp8_pool(wl, seed=9)
    blk = int(wl.item_ids[1].item())
    scale[blk, 1, 0, 0] = 1.0e5
    wl.q.mul_(1.0e-5)  # logits against that block stay of order one
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, wl.item_ids, None, None,
                                      dims=dict(wl.dims, layer=1), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref_fp8(wl, pool8, scale, layer=1), "fp8 prefill keys past f16")


def test_fp8_gist_workload_sampled():
    """The gist workload (12,800 pairs, l = 64 against 8 cached keys) read from
    an E4M3 pool, as the benchmark's --workload gist --kv fp8 row times it."""
    wl = workloads.make("gist", device=DEV, num_layers=2)
    pool8, scale = workloads.make_fp8_pool(wl)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, wl.item_ids, None, None,
                                      dims=dict(wl.dims, layer=1), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.sort(np.random.default_rng(2).choice(wl.dims["num_pairs"], 60, replace=False))
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref_fp8(wl, pool8, scale, layer=1, pairs=sel),
            "fp8 gist")
    del wl, pool8, got
    torch.cuda.empty_cache()


def test_fp8_bad_block_zeroes_and_flags():
    wl = workloads.make_custom(4, 1, 8, 8, 128, 32, 3, 6, device=DEV, seed=2, use_table=True)
    pool8, scale = workloads.make_fp8_pool(wl)
    wl.block_table[1, 2] = 99
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_fp8kv(wl.q, wl.k_new, wl.v_new, pool8, scale, None, wl.block_table,
                                      None, dims=wl.dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.STATUS_BAD_BLOCK
    assert not got[1].float().abs().any()
    ok = np.array([0, 2, 3])
    compare(got[torch.from_numpy(ok).to(DEV)], oracle_ref_fp8(wl, pool8, scale, pairs=ok), "fp8 good")
