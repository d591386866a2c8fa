"""GPU parity: the CUDA library against the fp64 oracle on the same seeded
inputs, element by element, |d| <= 1e-2 + 1e-2 |ref| (bf16 in and out); the
gather bit-exact.  Small cases run on every pair; the full-size workloads (in
the launch configuration the benchmark times) on a seeded sample of pairs."""
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


def sample(P, n, seed=0):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(P, size=min(n, P), replace=False))


def test_tiny_every_pair():
    wl = workloads.make("tiny", device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref(wl), "tiny")


# (P, l, Hq, Hkv, d, block_len, blocks_per_pair, num_blocks)
EDGE = [
    (5, 1, 14, 2, 64, 8, 1, 7),        # decode, gist
    (4, 2, 14, 2, 64, 8, 1, 7),        # smallest prefill
    (3, 3, 7, 1, 64, 5, 2, 9),         # ragged everything
    (6, 17, 4, 4, 128, 3, 3, 11),      # MHA, d=128, odd sizes
    (3, 64, 14, 2, 64, 1, 1, 4),       # k = 1
    (2, 100, 14, 2, 64, 19, 1, 5),     # two chunks, ragged tail
    (2, 256, 14, 2, 64, 64, 1, 3),     # longest sweep corner
    (2, 256, 14, 2, 64, 1, 1, 3),
    (3, 64, 32, 8, 128, 8, 1, 9),      # wide model
    (2, 130, 32, 8, 128, 16, 2, 5),    # wide, 3 chunks
    (4, 1, 32, 32, 128, 256, 2, 6),    # paged decode, short
    (3, 1, 16, 1, 64, 7, 3, 5),        # decode, group of 16
    (2, 9, 20, 1, 64, 4, 1, 3),        # group of 20 (prefill path)
    (3, 5, 6, 2, 64, 0, 0, 0),         # empty cache: causal self-attention only
    (3, 1, 6, 2, 128, 0, 0, 0),        # empty cache, one token: o = v_new
]


@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "P{}_l{}_Hq{}_Hkv{}_d{}_bl{}_b{}".format(*s[:7]))
@pytest.mark.parametrize("random_pos", [False, True])
def test_edge_shapes_every_pair(shape, random_pos):
    P, l, Hq, Hkv, d, bl, bpp, nb = shape
    wl = workloads.make_custom(P, l, Hq, Hkv, d, bl, bpp, nb, num_layers=2, layer=1, device=DEV,
                               seed=hash(shape) % 1000, random_pos=random_pos)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, layer=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref(wl, layer=1), str(shape))


# l = 1 shapes of the short decode (at most 32 cached keys in blocks of 8-row
# multiples): one or two 8-head tiles, one or two 16-key tiles
SHORT = [
    (7, 14, 2, 64, 8, 2),     # the query-gisted shape: 7 heads, 16 keys
    (6, 14, 2, 64, 8, 1),     # 8 cached keys
    (5, 16, 2, 128, 8, 2),    # G = 8: a full head tile, d = 128
    (4, 32, 2, 64, 8, 4),     # G = 16, 32 cached keys
    (5, 24, 2, 64, 16, 2),    # G = 12, 16-row blocks
    (6, 9, 3, 64, 8, 3),      # odd KV heads, 24 keys
    (4, 16, 4, 128, 16, 1),   # item ids, d = 128
    (3, 8, 8, 64, 24, 1),     # MHA, one 24-row block
]


@pytest.mark.parametrize("P,Hq,Hkv,d,bl,bpp", SHORT, ids=lambda v: str(v))
@pytest.mark.parametrize("random_pos", [False, True])
def test_short_decode_shapes(P, Hq, Hkv, d, bl, bpp, random_pos):
    wl = workloads.make_custom(P, 1, Hq, Hkv, d, bl, bpp, 9, num_layers=2, layer=1, device=DEV,
                               seed=P * bl + bpp, random_pos=random_pos)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, layer=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref(wl, layer=1), f"short decode G={Hq // Hkv} C={bl * bpp}")


# l = 1 with groups of 2..16 query heads and caches past 32 keys in blocks of
# 16-row multiples: the long GQA decode
GQA = [
    (3, 32, 8, 128, 256, 2),   # paged, 4 heads per KV head
    (2, 14, 2, 64, 16, 5),     # the gist model's groups, 80 keys
    (2, 32, 2, 64, 32, 3),     # 16 heads per KV head
    (3, 16, 4, 128, 64, 3),    # 4 heads, 192 keys
    (2, 6, 3, 64, 48, 1),      # item ids, 2 heads, one 48-row block
]


@pytest.mark.parametrize("P,Hq,Hkv,d,bl,bpp", GQA, ids=lambda v: str(v))
@pytest.mark.parametrize("random_pos", [False, True])
def test_gqa_decode_shapes(P, Hq, Hkv, d, bl, bpp, random_pos):
    wl = workloads.make_custom(P, 1, Hq, Hkv, d, bl, bpp, 9, num_layers=2, layer=1, device=DEV,
                               seed=P * bl + bpp, random_pos=random_pos)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, layer=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref(wl, layer=1), f"gqa decode G={Hq // Hkv} C={bl * bpp}")


@pytest.mark.parametrize("k", [1, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("l", [16, 64, 256])
def test_sweep_shapes(k, l):
    """The k x l sweep of the gist setting, on 48 pairs of a 300-item pool."""
    wl = workloads.make(workloads.sweep_spec(k, l), device=DEV, queries=4, candidates=12,
                        pool_items=300, num_layers=2)
    got = run_gpu(wl, layer=1)
    compare(got, oracle_ref(wl, layer=1), f"k={k} l={l}")


@pytest.mark.parametrize("name,n_sample,layer", [
    ("gist", 160, 17), ("qgist", 600, 9), ("wide", 96, 27), ("paged", 32, 31), ("paged_gqa", 32, 27)])
def test_full_size_workloads_sampled(name, n_sample, layer):
    """The benchmark's workloads at full size; the oracle checks a sample."""
    wl = workloads.make(name, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, layer=layer, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = sample(wl.dims["num_pairs"], n_sample, seed=layer)
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref(wl, layer=layer, pairs=sel), name)
    # every output row is a convex combination of value rows: finite everywhere
    assert torch.isfinite(got.float()).all()
    del wl, got
    torch.cuda.empty_cache()


@pytest.mark.parametrize("k,l", [(32, 64), (64, 16), (8, 256), (32, 256)])
def test_sweep_points_full_size_sampled(k, l):
    """Sweep points of the gist workload at full size (12,800 Zipf pairs): k = 32
    runs with two q stages so that two CTAs share an SM; k = 64, l = 16 is the
    widest cache of the sweep's single-pass shapes."""
    wl = workloads.make(workloads.sweep_spec(k, l), device=DEV, num_layers=2)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_gpu(wl, layer=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = sample(wl.dims["num_pairs"], 120, seed=k + l)
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref(wl, layer=1, pairs=sel), f"k={k} l={l}")
    del wl, got
    torch.cuda.empty_cache()


def test_shift_invariance_on_gpu():
    """Gist page, 在线的一次 attention: the same relative distances give the same
    output, whether the gist sits at 0..k-1 (query from k) or at j..j+k-1 (query
    from j+k).  The pool holds the gist K rotated at each layout's positions."""
    P, l, Hq, Hkv, d, k, j = 8, 16, 14, 2, 64, 8, 300
    base = workloads.make_custom(P, l, Hq, Hkv, d, k, 1, P, device=DEV, seed=5)
    raw = base.kv_pool[:, 0, 0].double().cpu().numpy()  # [P, Hkv, k, d], pre-rotation
    pools = []
    for start in (0, j):
        rot = np.empty_like(raw)
        for b in range(P):
            for g in range(Hkv):
                for t in range(k):
                    rot[b, g, t] = oracle.rope(raw[b, g, t], start + t)
        pool = base.kv_pool.clone()
        pool[:, 0, 0] = torch.from_numpy(rot).to(DEV).to(torch.bfloat16)
        pools.append(pool)
    ids = torch.arange(P, dtype=torch.int32, device=DEV)
    outs = []
    for pool, pos in zip(pools, (k, j + k)):
        posv = torch.full((P,), pos, dtype=torch.int32, device=DEV)
        outs.append(binding.gist_attn_fwd(base.q, base.k_new, base.v_new, pool, ids, None, posv,
                                          dims=dict(base.dims, num_blocks=P)))
    # both agree with the oracle on their own inputs, hence with each other
    for pool, pos, got in zip(pools, (k, j + k), outs):
        posv = np.full(P, pos, dtype=np.int32)
        ref = oracle.gist_attn(base.q, base.k_new, base.v_new, pool, item_ids=np.arange(P, dtype=np.int32),
                               pos_offset=posv, dims=dict(base.dims, num_blocks=P))
        compare(got, ref, f"layout pos={pos}")
    diff = (outs[0].float() - outs[1].float()).abs().max().item()
    assert diff < 0.05


@pytest.mark.parametrize("name", ["tiny", "qgist_small", "paged_small"])
def test_gather_bit_exact(name):
    if name == "tiny":
        wl = workloads.make("tiny", device=DEV)
    elif name == "qgist_small":
        wl = workloads.make("qgist", device=DEV, queries=20, pool_items=3000)
    else:
        wl = workloads.make("paged", device=DEV, paged_seqs=4, paged_pool_blocks=80, num_layers=3)
    layer = wl.dims["num_layers"] - 1
    dims = dict(wl.dims, layer=layer)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_gather_debug(wl.kv_pool, wl.item_ids, wl.block_table, dims=dims, status=status)
    torch.cuda.synchronize()
    want, rc = oracle.gather(wl.kv_pool, wl.item_ids, wl.block_table, dims=dims)
    assert rc == 0 and int(status.item()) == 0
    assert np.array_equal(oracle.bf16_bits(got), want)


def test_bad_block_zeroes_that_pair_and_sets_status():
    for l in (1, 8):
        wl = workloads.make_custom(6, l, 14, 2, 64, 8, 2, 10, device=DEV, seed=3)
        wl.block_table[2, 1] = 10          # one past the end
        wl.block_table[4, 0] = -7
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        got = run_gpu(wl, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & binding.STATUS_BAD_BLOCK
        assert not got[2].float().abs().any() and not got[4].float().abs().any()
        ok = np.array([0, 1, 3, 5])
        compare(got[torch.from_numpy(ok).to(DEV)], oracle_ref(wl, pairs=ok), f"l={l} good pairs")


def test_explicit_scale_and_default_positions():
    wl = workloads.make_custom(4, 12, 14, 2, 64, 8, 1, 6, device=DEV, seed=9)
    d = wl.dims["head_dim"]
    a = run_gpu(wl)
    wl.pos_offset = torch.full((4,), 8, dtype=torch.int32, device=DEV)  # the default, explicit
    b = run_gpu(wl)
    assert torch.equal(a, b)
    # an explicit scale (2.4 / sqrt(d)); test_range_gpu covers every kernel
    wl.dims = dict(wl.dims, softmax_scale=0.3)
    c = run_gpu(wl)
    compare(c, oracle_ref(wl), "scale 0.3")
    assert (c.float() - a.float()).abs().max().item() > 1e-2


def test_deterministic():
    wl = workloads.make("tiny", device=DEV)
    a, b = run_gpu(wl), run_gpu(wl)
    assert torch.equal(a, b)


def test_empty_batch_is_a_no_op():
    wl = workloads.make_custom(3, 4, 14, 2, 64, 8, 1, 5, device=DEV)
    out = torch.full_like(wl.q, 7.0)
    binding.gist_attn_fwd(wl.q[:0], wl.k_new[:0], wl.v_new[:0], wl.kv_pool, wl.item_ids[:0], None,
                          None, out[:0], dims=dict(wl.dims, num_pairs=0))
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
