"""GPU parity of the staged path (gist_attn_fwd_ws): more than 128 keys on
d = 64 with a cached segment in front, or a whole sequence on pre-RoPE inputs.
A pre-pass writes each pair's [cached; new] key sequence (keys rotated) and the
angles of q into the caller's workspace, then the long-sequence tensor-core
kernel runs on it and rotates q itself ([Gist page, "在线的一次 attention"]:
K = cat(cache[item].K[layer], K_new), the new tokens numbered after the cached
positions, causal inside the new block).
Every case is checked element by element against the float64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


def run_ws(wl, layer=0, status=None):
    dims = dict(wl.dims, layer=layer)
    n = binding.workspace_bytes(dims)
    assert n > 0, "shape should take the staged path"
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    return binding.gist_attn_fwd_ws(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids, wl.block_table,
                                    wl.pos_offset, None, ws, dims=dims, status=status)


SHAPES = [
    # P, l, Hq, Hkv, block_len, blocks_per_pair, num_blocks, random_pos
    (4, 300, 14, 2, 8, 1, 20, False),    # gist k = 8, 308 keys
    (3, 256, 14, 2, 64, 1, 9, True),     # the widest gist of the sweep
    (5, 300, 14, 2, 1, 1, 7, True),      # one cached position, ragged tiles
    (3, 290, 16, 2, 16, 2, 11, True),    # two cached blocks through a table, G = 8
    (2, 300, 4, 4, 32, 1, 5, False),     # MHA: 128 tokens per tile
    (2, 290, 128, 1, 8, 1, 4, False),    # G = 128: one token per tile
    (3, 300, 14, 2, 0, 0, 0, True),      # no cache: the offline pass on pre-RoPE inputs
    (64, 290, 14, 2, 16, 1, 40, True),   # 2,176 tiles: several per persistent CTA
]


@pytest.mark.parametrize("P,l,Hq,Hkv,bl,bpp,nb,rpos", SHAPES,
                         ids=lambda v: str(v))
def test_staged_matches_oracle(P, l, Hq, Hkv, bl, bpp, nb, rpos):
    wl = workloads.make_custom(P, l, Hq, Hkv, 64, bl, bpp, nb, num_layers=2, layer=1, device=DEV,
                               seed=P + l + bl, random_pos=rpos)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_ws(wl, layer=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref(wl, layer=1), f"staged P={P} l={l} C={bl * bpp} G={Hq // Hkv}")


def test_without_workspace_the_call_is_gist_attn_fwd():
    """No workspace (or one too small): the same dispatch as gist_attn_fwd."""
    wl = workloads.make_custom(3, 200, 14, 2, 64, 8, 1, 6, device=DEV, seed=3)
    a = binding.gist_attn_fwd_ws(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids, None, None, None,
                                 None, dims=wl.dims)
    small = torch.empty(1024, dtype=torch.uint8, device=DEV)
    b = binding.gist_attn_fwd_ws(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids, None, None, None,
                                 small, dims=wl.dims)
    c = run_gpu(wl)
    torch.cuda.synchronize()
    assert torch.equal(a, c) and torch.equal(b, c)
    compare(a, oracle_ref(wl), "no workspace")


def test_staged_bad_block_zeroes_that_pair_and_sets_status():
    wl = workloads.make_custom(4, 290, 14, 2, 64, 8, 1, 6, device=DEV, seed=8)
    wl.item_ids[2] = 6  # one past the pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_ws(wl, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.STATUS_BAD_BLOCK
    assert torch.count_nonzero(got[2]).item() == 0
    keep = np.array([0, 1, 3])
    compare(got[torch.from_numpy(keep).to(DEV)], oracle_ref(wl, pairs=keep), "good pairs")


def test_staged_value_past_f16_range_matches_oracle():
    """A query element past the f16 range (the staged path forms q.K in f16):
    the rows that meet it are recomputed in fp32 and every pair matches the
    oracle."""
    wl = workloads.make_custom(2, 290, 14, 2, 64, 8, 1, 4, device=DEV, seed=9)
    wl.q[1, 5, 3, 7] = 1.0e5
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_ws(wl, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    compare(got, oracle_ref(wl), "staged, 1e5 in q")


def test_staged_is_deterministic():
    wl = workloads.make_custom(3, 290, 14, 2, 64, 16, 1, 5, device=DEV, seed=10)
    a, b = run_ws(wl), run_ws(wl)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_sweep_point_k64_l256_full_size_sampled():
    """The widest sweep point, k = 64, l = 256 (320 keys), at its full size
    (12,800 Zipf pairs), as the benchmark times it; the oracle checks a sample."""
    wl = workloads.make(workloads.sweep_spec(64, 256), device=DEV, num_layers=2)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run_ws(wl, layer=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.sort(np.random.default_rng(7).choice(wl.dims["num_pairs"], size=40, replace=False))
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref(wl, layer=1, pairs=sel), "k=64 l=256")
    assert torch.isfinite(got.float()).all()
    del wl, got
    torch.cuda.empty_cache()


def test_staged_prerotated_inputs_with_a_cache():
    """Pre-rotated q and k_new (GIST_ATTN_FLAG_PREROTATED) behind a cache: the
    pre-pass only converts (every angle is 0) and the result is the oracle's
    prerotated attention."""
    wl = workloads.make_custom(3, 290, 14, 2, 64, 16, 1, 5, device=DEV, seed=12, random_pos=True)
    dims = dict(wl.dims, flags=binding.FLAG_PREROTATED)
    n = binding.workspace_bytes(dims)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd_ws(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids, None, wl.pos_offset,
                                   None, ws, dims=dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    wl.dims = dims
    compare(got, oracle_ref(wl), "staged, pre-rotated inputs")
