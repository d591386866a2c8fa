"""GPU parity of the projections either side of the attention (the QKV
projection with RoPE in its epilogue, and the output projection) and of one
whole layer of them around the attention, against the float64 oracle.

Gist page ("把 item 压成 KV：gist 能不能用在相关性任务上"), 在线的一次 attention:
per layer X is projected to Q, K, V, attends against the cache, and goes
through the output projection.  Weights are synthetic (N(0, 1/fan_in))."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_cached_kv_gb300 import binding, workloads
from oracle import projections as proj
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


def _weights(rows, cols, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn((rows, cols), generator=g, device=DEV) / cols ** 0.5).to(torch.bfloat16)


def _x(P, l, dm, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn((P, l, dm), generator=g, device=DEV).to(torch.bfloat16)


def _dims(P, l, Hq, Hkv, d, bl=8, bpp=1, nb=1, flags=0):
    return dict(num_pairs=P, n_new=l, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_len=bl,
                blocks_per_pair=bpp, num_blocks=nb, num_layers=1, layer=0, rope_theta=1e4,
                softmax_scale=0.0, flags=flags)


@pytest.mark.parametrize("P,l,Hq,Hkv,d,dm,pos", [
    (3, 64, 14, 2, 64, 256, None),       # the gist model's heads, a narrow model width
    (2, 37, 14, 2, 64, 896, "random"),   # ragged rows, the gist model width
    (2, 64, 8, 2, 128, 512, "random"),   # d = 128
    (3, 40, 14, 2, 64, 200, "random"),   # d_model not a multiple of the 64-wide k-block
])
def test_qkv_rope_matches_oracle(P, l, Hq, Hkv, d, dm, pos):
    x, w = _x(P, l, dm, 1), _weights((Hq + 2 * Hkv) * d, dm, 2)
    dims = _dims(P, l, Hq, Hkv, d)
    pos_t = None
    if pos == "random":
        pos_t = torch.from_numpy(np.random.default_rng(3).integers(0, 4000, P).astype(np.int32)).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, k, v = binding.gist_qkv_rope(x, w, pos_t, dims=dims, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rq, rk, rv = proj.qkv_rope(x, w, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, cached=8,
                               pos_offset=None if pos_t is None else pos_t.cpu().numpy())
    compare(q, rq, "q")
    compare(k, rk, "k_new")
    compare(v, rv, "v_new")


def test_projections_with_several_tiles_per_cta():
    """Both GEMMs at a size where each persistent CTA takes two or three output
    tiles (the k-block ring and the two TMEM accumulators carried across
    tiles): 128 pairs x 64 tokens of the gist model (8,192 rows)."""
    P, l, Hq, Hkv, d, dm = 128, 64, 14, 2, 64, 1152
    x, w = _x(P, l, dm, 11), _weights((Hq + 2 * Hkv) * d, dm, 12)
    pos_t = torch.from_numpy(np.random.default_rng(13).integers(0, 4000, P).astype(np.int32)).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, k, v = binding.gist_qkv_rope(x, w, pos_t, dims=_dims(P, l, Hq, Hkv, d), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rq, rk, rv = proj.qkv_rope(x, w, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, cached=8,
                               pos_offset=pos_t.cpu().numpy())
    compare(q, rq, "q")
    compare(k, rk, "k_new")
    compare(v, rv, "v_new")
    wo = _weights(dm, Hq * d, 14)
    y = binding.gist_out_proj(q, wo, dims=_dims(P, l, Hq, Hkv, d))
    torch.cuda.synchronize()
    compare(y, proj.out_proj(q.reshape(P, l, Hq * d), wo), "y")


@pytest.mark.parametrize("P,l,Hq,d,dm", [(3, 50, 14, 64, 256), (2, 64, 14, 64, 896), (1, 200, 8, 128, 384),
                                          (5, 77, 14, 64, 1152)])
def test_out_proj_matches_oracle(P, l, Hq, d, dm):
    a = _x(P, l * Hq, d, 4).reshape(P, l, Hq, d).contiguous()
    w = _weights(dm, Hq * d, 5)
    y = binding.gist_out_proj(a, w, dims=_dims(P, l, Hq, 2 if Hq % 2 == 0 else 1, d))
    torch.cuda.synchronize()
    ref = proj.out_proj(a.reshape(P, l, Hq * d), w)
    compare(y, ref, "y")


def test_one_layer_projections_around_attention():
    """x -> QKV + RoPE -> attention on pre-rotated inputs (gist cache) -> o-proj.
    Each stage against the oracle on the stage's actual inputs, and the whole
    layer against the float64 pipeline."""
    P, l, Hq, Hkv, d, dm, k_gist, nb = 4, 64, 14, 2, 64, 896, 8, 6
    x, wqkv, wo = _x(P, l, dm, 6), _weights((Hq + 2 * Hkv) * d, dm, 7), _weights(dm, Hq * d, 8)
    wl = workloads.make_custom(P, l, Hq, Hkv, d, k_gist, 1, nb, device=DEV, seed=9)
    dims = _dims(P, l, Hq, Hkv, d, bl=k_gist, nb=nb)
    q, kn, vn = binding.gist_qkv_rope(x, wqkv, dims=dims)
    pre = dict(dims, flags=binding.FLAG_PREROTATED)
    attn = binding.gist_attn_fwd(q, kn, vn, wl.kv_pool, wl.item_ids, None, None, dims=pre)
    y = binding.gist_out_proj(attn, wo, dims=dims)
    torch.cuda.synchronize()
    # the attention stage on its own inputs
    ref_attn = oracle.gist_attn(q, kn, vn, wl.kv_pool, item_ids=wl.item_ids, dims=pre)
    compare(attn, ref_attn, "attention on pre-rotated q, k")
    # the output projection on its own input
    compare(y, proj.out_proj(attn.reshape(P, l, Hq * d), wo), "o-proj")
    # the whole layer in float64 (bf16 intermediates on the GPU: a looser bound)
    rq, rk, rv = proj.qkv_rope(x, wqkv, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, cached=k_gist)
    pool = oracle.bf16_bits(wl.kv_pool).astype(np.uint32) << 16
    poolf = pool.view(np.float32).astype(np.float64)
    ra = oracle.gist_attn(rq, rk, rv, poolf, item_ids=wl.item_ids, dims=pre, f64_inputs=True)
    ry = proj.out_proj(ra.reshape(P, l, Hq * d), wo)
    err = np.abs(y.float().cpu().numpy() - ry)
    assert (err <= 5e-2 + 5e-2 * np.abs(ry)).all(), err.max()


@pytest.mark.parametrize("P,l,Hq,Hkv,d,nb", [
    (3, 12, 14, 2, 64, 5),     # tensor-core prefill, two CTAs per SM
    (2, 64, 32, 8, 128, 4),    # tensor-core prefill, d = 128
    (4, 1, 14, 2, 64, 6),      # decode (short cache)
    (3, 200, 14, 2, 64, 4),    # streaming prefill (cache + l > 128 keys)
])
def test_prerotated_flag_skips_rope_in_the_attention(P, l, Hq, Hkv, d, nb):
    """Rotating q and k_new outside (the oracle's rotation, rounded to bf16) and
    passing the flag gives the attention of the unrotated inputs."""
    wl = workloads.make_custom(P, l, Hq, Hkv, d, 8, 1, nb, device=DEV, seed=10)
    pos = 8 + np.arange(l)
    qr = np.stack([proj.rope_rows(oracle_f64(wl.q[p]).transpose(1, 0, 2), pos).transpose(1, 0, 2)
                   for p in range(P)])
    kr = np.stack([proj.rope_rows(oracle_f64(wl.k_new[p]).transpose(1, 0, 2), pos).transpose(1, 0, 2)
                   for p in range(P)])
    qb = torch.from_numpy(qr).to(torch.bfloat16).to(DEV)
    kb = torch.from_numpy(kr).to(torch.bfloat16).to(DEV)
    dims = dict(wl.dims, flags=binding.FLAG_PREROTATED)
    got = binding.gist_attn_fwd(qb, kb, wl.v_new, wl.kv_pool, wl.item_ids, None, None, dims=dims)
    ref = oracle.gist_attn(qb, kb, wl.v_new, wl.kv_pool, item_ids=wl.item_ids, dims=dims)
    compare(got, ref, "pre-rotated")


def oracle_f64(t: torch.Tensor) -> np.ndarray:
    bits = oracle.bf16_bits(t).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)
