"""GPU parity of the long-sequence tensor-core kernel: causal attention over
whole pre-rotated sequences with no cached segment (the offline gist pass of
Gist page "论文做了什么" in the fused pipeline, where the QKV projection's
epilogue has already rotated q and k_new), against the float64 oracle, on
sequences longer than the 128 keys of the single-pass kernel."""
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


@pytest.mark.parametrize("P,l,Hq,Hkv", [
    (2, 300, 14, 2),    # the gist model's heads, 3 key blocks, ragged last tile
    (1, 1000, 4, 4),    # MHA (G = 1): 128 tokens per tile, 8 key blocks
    (2, 257, 16, 2),    # G = 8, a key block of 1
    (3, 129, 7, 1),     # one token past the single-pass kernel's limit
    (1, 150, 128, 1),   # G = 128: one token per tile
    (1, 1008, 14, 2),   # the offline pass's length (1000 prompt + 8 gist tokens)
])
def test_long_prerotated_causal_matches_oracle(P, l, Hq, Hkv):
    wl = workloads.make_custom(P, l, Hq, Hkv, 64, 0, 0, 0, device=DEV, seed=l + Hq)
    dims = dict(wl.dims, flags=binding.FLAG_PREROTATED)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, None, None, dims=dims,
                                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.gist_attn(wl.q, wl.k_new, wl.v_new, wl.kv_pool, dims=dims)
    compare(got, ref, f"l={l} G={Hq // Hkv}")


def test_long_kernel_is_deterministic_and_layer_independent():
    wl = workloads.make_custom(2, 400, 14, 2, 64, 0, 0, 0, device=DEV, seed=5)
    dims = dict(wl.dims, flags=binding.FLAG_PREROTATED)
    a = binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, None, None, dims=dims)
    b = binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, None, None, dims=dims)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("P,l,Hq,Hkv", [
    (64, 200, 14, 2),   # 1,536 row tiles: several per persistent CTA
    (40, 300, 4, 4),    # G = 1: 480 tiles, the last CTAs take two
    (40, 140, 128, 1),  # G = 128: 5,600 one-token tiles, ~18 per CTA
])
def test_long_many_tiles_per_cta_every_pair(P, l, Hq, Hkv):
    """Grids where each persistent CTA walks several row tiles (the tile walk,
    the two q stages and the K/V streams across tile boundaries)."""
    wl = workloads.make_custom(P, l, Hq, Hkv, 64, 0, 0, 0, device=DEV, seed=P + l)
    dims = dict(wl.dims, flags=binding.FLAG_PREROTATED)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, None, None, dims=dims,
                                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.gist_attn(wl.q, wl.k_new, wl.v_new, wl.kv_pool, dims=dims)
    compare(got, ref, f"P={P} l={l} G={Hq // Hkv}")


def test_long_offline_pass_full_size_sampled():
    """The offline pass as the benchmark times it (128 items of 1000 prompt +
    8 gist tokens, the gist model's heads); the oracle checks a sample of items
    spread over the grid."""
    P, l, Hq, Hkv = 128, 1008, 14, 2
    wl = workloads.make_custom(P, l, Hq, Hkv, 64, 0, 0, 0, device=DEV, seed=21)
    dims = dict(wl.dims, flags=binding.FLAG_PREROTATED)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, None, None, None, dims=dims,
                                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.array([0, 1, 37, 64, 101, 127], dtype=np.int32)
    ref = oracle.gist_attn(wl.q, wl.k_new, wl.v_new, wl.kv_pool, dims=dims, pairs=sel)
    compare(got[torch.from_numpy(sel).long().to(DEV)], ref, "offline pass, sampled items")
    assert torch.isfinite(got.float()).all()
