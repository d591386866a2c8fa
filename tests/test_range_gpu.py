"""GPU parity over the whole legal input range, against the fp64 oracle.

The operation ([Gist page, "在线的一次 attention"]; [KV page, "Reusable-state"]) is
defined for every bf16 input, every softmax scale and every int32 position, so
each attention kernel is checked, element by element at |d| <= 1e-2 + 1e-2 |ref|,
on:
  * explicit softmax scales well above 1/sqrt(d) (0.3 and 0.5 at d = 64);
  * single values past the f16 range (|x| = 1e5) in q, in a new key and in a
    cached key -- the kernels that form q.K in f16 recompute the rows that meet
    one in fp32 -- and in a value;
  * positions far from 0 (6.5e4, 1e6, 2^30 and the largest that fits), where an
    angle formed as an fp32 product would be off by whole radians;
  * q and keys scaled up together, so that logits spread over tens of nats.
Every case names the kernel its shape selects (the dispatch of gist_attn_fwd)."""
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


# kernel -> (P, l, Hq, Hkv, d, block_len, blocks_per_pair, num_blocks, staged)
SHAPES = {
    "prefill_tc": (4, 12, 14, 2, 64, 8, 1, 6, False),
    "prefill_tc_d128": (3, 20, 32, 8, 128, 8, 1, 5, False),
    "prefill_stream": (3, 40, 14, 2, 64, 128, 2, 7, False),  # 296 keys: past prefill_tc
    "staged": (3, 290, 14, 2, 64, 16, 2, 7, True),
    "prefill_tc_wide_keys": (3, 200, 14, 2, 64, 16, 2, 7, False),
    "decode_short": (5, 1, 14, 2, 64, 8, 2, 9, False),
    "decode_5row_blocks": (4, 1, 14, 2, 64, 5, 3, 9, False),
    "decode_long": (3, 1, 8, 8, 128, 64, 2, 7, False),
    "decode_gqa": (3, 1, 16, 2, 64, 32, 4, 9, False),
    "decode": (3, 1, 16, 2, 64, 20, 4, 9, False),
}


def make(kernel, seed=0, random_pos=False):
    P, l, Hq, Hkv, d, bl, bpp, nb, staged = SHAPES[kernel]
    wl = workloads.make_custom(P, l, Hq, Hkv, d, bl, bpp, nb, device=DEV, seed=seed,
                               random_pos=random_pos)
    return wl, staged


def run(wl, staged, status=None):
    if not staged:
        return run_gpu(wl, status=status)
    n = binding.workspace_bytes(wl.dims)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    return binding.gist_attn_fwd_ws(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids,
                                    wl.block_table, wl.pos_offset, None, ws, dims=wl.dims,
                                    status=status)


def check(wl, staged, what):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = run(wl, staged, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"{what}: status {int(status.item())}"
    return compare(got, oracle_ref(wl), what)


@pytest.mark.parametrize("kernel", sorted(SHAPES))
@pytest.mark.parametrize("scale", [0.3, 0.5])
def test_explicit_scale(kernel, scale):
    """Scales of 2.4 and 4 times 1/sqrt(64): a sharper softmax, larger logits."""
    wl, staged = make(kernel, seed=3, random_pos=True)
    wl.dims = dict(wl.dims, softmax_scale=scale)
    check(wl, staged, f"{kernel} scale {scale}")


def _first_block(wl, p):
    src = wl.block_table if wl.block_table is not None else wl.item_ids.view(-1, 1)
    return int(src[p, 0].item())


@pytest.mark.parametrize("kernel", sorted(SHAPES))
@pytest.mark.parametrize("where", ["q", "k_new", "cached_k", "v_new", "cached_v"])
def test_values_past_the_f16_range(kernel, where):
    """One element of magnitude 1e5 (a legal bf16 value, past f16's 65504) in
    one input; the output still matches the oracle everywhere and the status
    word stays clear."""
    wl, staged = make(kernel, seed=7)
    l = wl.dims["n_new"]
    t = min(l - 1, 3)
    if where == "q":
        wl.q[1, t, 1, 3] = 1.0e5
    elif where == "k_new":
        wl.k_new[1, 0, 0, 5] = -1.0e5
    elif where == "v_new":
        wl.v_new[1, 0, 0, 9] = 1.0e5
    else:
        if wl.dims["block_len"] * wl.dims["blocks_per_pair"] == 0:
            pytest.skip("no cache")
        kv = 0 if where == "cached_k" else 1
        wl.kv_pool[_first_block(wl, 1), 0, kv, 0, 0, 2] = 1.0e5
    check(wl, staged, f"{kernel} 1e5 in {where}")


@pytest.mark.parametrize("kernel", sorted(SHAPES))
def test_positions_far_from_zero(kernel):
    """pos_offset of 65,000, 1,000,003, 2^30 + 7 and the largest position whose
    new tokens still fit int32 (only differences matter to the method, but the
    kernel must rotate at the absolute angle the oracle uses)."""
    wl, staged = make(kernel, seed=11)
    P, l = wl.dims["num_pairs"], wl.dims["n_new"]
    far = [65000, 1000003, (1 << 30) + 7, (1 << 31) - l]
    wl.pos_offset = torch.tensor([far[i % len(far)] for i in range(P)], dtype=torch.int32,
                                 device=DEV)
    check(wl, staged, f"{kernel} far positions")


@pytest.mark.parametrize("kernel", sorted(SHAPES))
@pytest.mark.parametrize("factor", [2.0, 4.0])
def test_large_logits(kernel, factor):
    """q and every key scaled by `factor` (logits by factor^2: a spread of 4 and
    16 times the workloads', up to tens of nats): the kernels that round q and
    the keys to f16 send rows whose largest logit is that large to the fp32
    recomputation, so the output still matches the oracle everywhere."""
    wl, staged = make(kernel, seed=17, random_pos=True)
    wl.q.mul_(factor)
    wl.k_new.mul_(factor)
    wl.kv_pool[:, :, 0].mul_(factor)
    check(wl, staged, f"{kernel} logits x{factor * factor:g}")


def test_masked_key_far_above_the_visible_ones():
    """A later token's key of magnitude 1e4: rows of earlier tokens must not see
    it, although its logit there is tens of thousands of log2 units above every
    key they do see (the tensor-core prefill takes the row maximum over the
    whole tile and recomputes rows whose weights underflow)."""
    wl, staged = make("prefill_tc", seed=13)
    wl.k_new[:, 6] = 1.0e4 * torch.sign(wl.k_new[:, 6].float()).to(torch.bfloat16)
    check(wl, staged, "prefill_tc masked key 1e4")


@pytest.mark.parametrize("scale", [0.3, 0.5])
def test_gist_layer_full_size_explicit_scale(scale):
    """The full-size gist layer (12,800 Zipf pairs, the benchmark's launch) at an
    explicit scale; the oracle checks a sample of pairs."""
    wl = workloads.make("gist", device=DEV)
    dims = dict(wl.dims, layer=5, softmax_scale=scale)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids, None, None,
                                dims=dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.sort(np.random.default_rng(int(scale * 10)).choice(wl.dims["num_pairs"], 80,
                                                                 replace=False))
    wl.dims = dims
    compare(got[torch.from_numpy(sel).to(DEV)], oracle_ref(wl, layer=5, pairs=sel),
            f"gist scale {scale}")
    del wl, got
    torch.cuda.empty_cache()
