"""Pins for the fp64 oracle, against facts that do not come from the oracle.

Pages, cited by title and section:
  gist page   "把 item 压成 KV：gist 能不能用在相关性任务上"
  suffix page icman.com.cn news 64898 (suffix KV-cache reuse)
  KV page     "为什么自回归推理缓存 KV，而不缓存历史 Q？"

Independent references used here: RoPE as a complex rotation (numpy complex
exp), torch's scaled_dot_product_attention in float64 with an explicit boolean
mask, the decode formula written with numpy matrix products, closed forms,
the gist mask built by brute force, a tiny random two-layer model, and the
figures the pages print (tests/golden/page_figures.json).  The last test plants
one mistake at a time in a separate oracle build and checks that some pin
fails for each.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import gist_mask as gm

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


# ---------------------------------------------------------------- helpers ---

def rope_complex(x: np.ndarray, pos, theta: float = 1e4) -> np.ndarray:
    """RoPE written as a complex rotation: (x_j + i x_{j+d/2}) * exp(i pos theta_j)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    z = x[..., :h] + 1j * x[..., h:]
    freq = theta ** (-2.0 * np.arange(h) / d)
    pos = np.asarray(pos, dtype=np.float64)
    z = z * np.exp(1j * pos[..., None] * freq)
    return np.concatenate([z.real, z.imag], axis=-1)


def bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def sdpa_reference(q, k_new, v_new, pool, blocks, pos0, *, Hq, Hkv, layer=0, theta=1e4, scale=None):
    """Full reference through torch SDPA (float64): per pair, keys = cached rows
    (all visible) then rotated new keys (causal), GQA by contiguous groups."""
    q, k_new, v_new, pool = f64(q), f64(k_new), f64(v_new), f64(pool)
    P, l, _, d = q.shape
    G = Hq // Hkv
    out = np.zeros(q.shape)
    for p in range(P):
        pos = pos0[p] + np.arange(l)
        Kc = np.concatenate([pool[b, layer, 0] for b in blocks[p]], axis=1) if len(blocks[p]) else np.zeros((Hkv, 0, d))
        Vc = np.concatenate([pool[b, layer, 1] for b in blocks[p]], axis=1) if len(blocks[p]) else np.zeros((Hkv, 0, d))
        C = Kc.shape[1]
        kn = np.stack([rope_complex(k_new[p, :, g], pos, theta) for g in range(Hkv)])  # [Hkv, l, d]
        K = np.concatenate([Kc, kn], axis=1)
        V = np.concatenate([Vc, v_new[p].transpose(1, 0, 2)], axis=1)
        qr = np.stack([rope_complex(q[p, :, h], pos, theta) for h in range(Hq)])  # [Hq, l, d]
        mask = np.zeros((l, C + l), dtype=bool)
        for i in range(l):
            mask[i, : C + i + 1] = True
        Kx = torch.from_numpy(np.repeat(K, G, axis=0))
        Vx = torch.from_numpy(np.repeat(V, G, axis=0))
        o = F.scaled_dot_product_attention(torch.from_numpy(qr), Kx, Vx,
                                           attn_mask=torch.from_numpy(mask),
                                           scale=scale if scale else 1.0 / math.sqrt(d))
        out[p] = o.numpy().transpose(1, 0, 2)
    return out


def dims(P, l, Hq, Hkv, d, bl, bpp, nb, L=1, layer=0, scale=0.0):
    return dict(num_pairs=P, n_new=l, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                block_len=bl, blocks_per_pair=bpp, num_blocks=nb, num_layers=L, layer=layer,
                rope_theta=1e4, softmax_scale=scale)


def small_case(seed=0, P=3, l=7, Hq=6, Hkv=2, d=16, bl=5, bpp=2, nb=9, L=2, layer=1):
    q = bf16((P, l, Hq, d), seed)
    kn = bf16((P, l, Hkv, d), seed + 1)
    vn = bf16((P, l, Hkv, d), seed + 2)
    pool = bf16((nb, L, 2, Hkv, bl, d), seed + 3)
    rng = np.random.default_rng(seed)
    table = rng.integers(0, nb, size=(P, bpp)).astype(np.int32)
    pos0 = rng.integers(0, 5000, size=P).astype(np.int32)
    return q, kn, vn, pool, table, pos0, dims(P, l, Hq, Hkv, d, bl, bpp, nb, L, layer)


# ------------------------------------------------------------- the checks ---
# Each check returns None when the pin holds, else a short reason; the tests
# below assert on them, and the planted-mistake test runs them on mutants.

def check_rope_complex(plant=0):
    rng = np.random.default_rng(1)
    for d in (16, 64, 128):
        x = rng.standard_normal(d)
        for pos in (0, 1, 7, 4096, 100_000):
            a = oracle.rope(x, pos, plant=plant)
            b = rope_complex(x, pos)
            if not np.allclose(a, b, rtol=0, atol=1e-9 * max(1.0, np.abs(b).max())):
                return f"rope d={d} pos={pos}"
    return None


def check_sdpa_general(plant=0, seed=0):
    q, kn, vn, pool, table, pos0, D = small_case(seed)
    got = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D, plant=plant)
    ref = sdpa_reference(q, kn, vn, pool, table, pos0, Hq=D["num_q_heads"], Hkv=D["num_kv_heads"],
                         layer=D["layer"])
    err = np.abs(got - ref).max()
    return None if err < 1e-11 else f"sdpa max err {err:.3e}"


def check_gqa_equals_repeated_mha(plant=0):
    q, kn, vn, pool, table, pos0, D = small_case(3, Hq=6, Hkv=2)
    G = 3
    got = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D, plant=plant)
    D2 = dict(D, num_kv_heads=6)
    rep = oracle.gist_attn(q, kn.repeat_interleave(G, dim=2), vn.repeat_interleave(G, dim=2),
                           pool.repeat_interleave(G, dim=3), block_table=table, pos_offset=pos0,
                           dims=D2, plant=plant)
    err = np.abs(got - rep).max()
    return None if err < 1e-12 else f"gqa vs repeated mha {err:.3e}"


def check_layer_selection(plant=0):
    q, kn, vn, pool, table, pos0, D = small_case(5, L=3, layer=1)
    got = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D, plant=plant)
    one = pool[:, 1:2].contiguous()
    ref = oracle.gist_attn(q, kn, vn, one, block_table=table, pos_offset=pos0,
                           dims=dict(D, num_layers=1, layer=0), plant=plant)
    err = np.abs(got - ref).max()
    return None if err == 0.0 else f"layer slice {err:.3e}"


def check_closed_forms(plant=0):
    # (a) q = 0: uniform weights, o = mean of the visible values
    q, kn, vn, pool, table, pos0, D = small_case(7)
    zq = torch.zeros_like(q)
    got = oracle.gist_attn(zq, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D, plant=plant)
    P, l, Hq, d = q.shape
    G = Hq // D["num_kv_heads"]
    poolf, vnf = f64(pool), f64(vn)
    for p in range(P):
        Vc = np.concatenate([poolf[b, D["layer"], 1] for b in table[p]], axis=1)
        for h in range(Hq):
            g = h // G
            for i in range(l):
                rows = np.concatenate([Vc[g], vnf[p, : i + 1, g]], axis=0)
                if not np.allclose(got[p, i, h], rows.mean(axis=0), rtol=0, atol=1e-12):
                    return "q=0 mean"
    # (b) constant values: o = c
    c = bf16((d,), 11)
    vconst = c.expand_as(vn).contiguous()
    pconst = pool.clone()
    pconst[:, :, 1] = c
    got = oracle.gist_attn(q, kn, vconst, pconst, block_table=table, pos_offset=pos0, dims=D, plant=plant)
    if not np.allclose(got, np.broadcast_to(f64(c), got.shape), rtol=0, atol=1e-12):
        return "constant V"
    # (c) empty cache, one token: o = v_new
    D0 = dims(P, 1, Hq, D["num_kv_heads"], d, 0, 0, 0)
    got = oracle.gist_attn(q[:, :1].contiguous(), kn[:, :1].contiguous(), vn[:, :1].contiguous(), None,
                           dims=D0, plant=plant)
    want = np.repeat(f64(vn[:, :1]), G, axis=2)
    if not np.allclose(got, want, rtol=0, atol=1e-12):
        return "empty cache l=1"
    return None


def check_rows_sum(plant=0):
    q, kn, vn, pool, table, pos0, D = small_case(9)
    _, w = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D,
                            want_weights=True, plant=plant)
    if not np.allclose(w.sum(axis=-1), 1.0, rtol=0, atol=1e-12):
        return "row sums"
    C = D["blocks_per_pair"] * D["block_len"]
    for i in range(D["n_new"]):
        if np.any(w[:, i, :, C + i + 1:] != 0) or np.any(w[:, i, :, : C + i + 1] <= 0):
            return "support of the weights"
    return None


def check_gist_mask_brute_force(plant=0):
    """gist page, 论文做了什么: the oracle's gist-masked attention over whole
    sequences [prompt j_p; gist k; rest] (right-padded to one length, a
    different j_p per pair) against the brute-force mask, the loop-per-row
    masked attention and the loop-per-element RoPE of oracle/gist_mask.py."""
    P, n, Hq, Hkv, d, k = 3, 13, 4, 2, 8, 3
    G = Hq // Hkv
    q, kn, vn = bf16((P, n, Hq, d), 70), bf16((P, n, Hkv, d), 71), bf16((P, n, Hkv, d), 72)
    starts = np.array([2, 5, 0], dtype=np.int32)
    pos0 = np.array([0, 17, 300], dtype=np.int32)
    got = oracle.gist_attn(q, kn, vn, None, pos_offset=pos0, dims=dims(P, n, Hq, Hkv, d, 0, 0, 0),
                           gist_start=starts, gist_len=k, plant=plant)
    for p in range(P):
        j = int(starts[p])
        allowed = gm.gist_mask(j, k, n - j - k)
        pos = pos0[p] + np.arange(n)
        for h in range(Hq):
            qr = gm.rope_rotate_half(f64(q[p, :, h]), pos)
            kr = gm.rope_rotate_half(f64(kn[p, :, h // G]), pos)
            want = gm.masked_attention(qr, kr, f64(vn[p, :, h // G]), allowed, 1 / math.sqrt(d))
            err = np.abs(got[p, :, h] - want).max()
            if err > 1e-12:
                return f"gist mask pair {p} head {h}: {err:.3e}"
    return None


ALL_CHECKS = [check_rope_complex, check_sdpa_general, check_gqa_equals_repeated_mha,
              check_layer_selection, check_closed_forms, check_rows_sum,
              check_gist_mask_brute_force]


# ------------------------------------------------------------------ tests ---

def test_bf16_widening_is_exact():
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x0080: 2.0 ** -126, 0x3C00: 2.0 ** -7}
    for bits, val in cases.items():
        assert oracle.bf16_to_f64(bits) == val
    assert math.copysign(1.0, oracle.bf16_to_f64(0x8000)) == -1.0


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    assert check() is None


def test_rope_depends_only_on_position_difference():
    """gist page, 在线的一次 attention: RoPE depends only on the difference."""
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    base = np.dot(oracle.rope(q, 19), oracle.rope(k, 3))
    for shift in (1, 100, 4000):
        assert abs(np.dot(oracle.rope(q, 19 + shift), oracle.rope(k, 3 + shift)) - base) < 1e-10


def _shift_case(j, pos_shift_gist, pos_offset, seed=21):
    """f64 inputs: gist keys rotated at pos_shift_gist + 0..k-1, queries at pos_offset."""
    P, l, Hq, Hkv, d, k = 2, 6, 4, 2, 64, 8
    rng = np.random.default_rng(seed)
    graw = rng.standard_normal((P, Hkv, k, d))
    gv = rng.standard_normal((P, Hkv, k, d))
    pool = np.zeros((P, 1, 2, Hkv, k, d))
    for p in range(P):
        for g in range(Hkv):
            pool[p, 0, 0, g] = rope_complex(graw[p, g], pos_shift_gist + np.arange(k))
            pool[p, 0, 1, g] = gv[p, g]
    q = rng.standard_normal((P, l, Hq, d))
    kn = rng.standard_normal((P, l, Hkv, d))
    vn = rng.standard_normal((P, l, Hkv, d))
    D = dims(P, l, Hq, Hkv, d, k, 1, P)
    return oracle.gist_attn(q, kn, vn, pool, item_ids=np.arange(P, dtype=np.int32),
                            pos_offset=np.full(P, pos_offset, dtype=np.int32), dims=D,
                            f64_inputs=True)


def test_shift_invariance_of_positions():
    """gist page, 在线的一次 attention: training puts the gist at j+1..j+k and the
    query after it; inference numbers the query from k+1.  Same relative
    distances, same result."""
    k, j = 8, 37
    infer = _shift_case(j, 0, k)
    train = _shift_case(j, j, j + k)
    assert np.abs(infer - train).max() < 1e-12
    # the failure the page warns about: gist kept at j.., query renumbered from k
    wrong = _shift_case(j, j, k)
    assert np.abs(wrong - train).max() > 1e-3


def test_bf16_and_f64_entries_agree():
    q, kn, vn, pool, table, pos0, D = small_case(13)
    a = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D)
    b = oracle.gist_attn(f64(q), f64(kn), f64(vn), f64(pool), block_table=table, pos_offset=pos0,
                         dims=D, f64_inputs=True)
    assert np.array_equal(a, b)


def test_gist_mask_is_causal_minus_lower_left_block():
    """gist page, 论文做了什么: causal mask with the lower-left block removed."""
    j, k, l = 5, 3, 4
    m = gm.gist_mask(j, k, l)
    n = j + k + l
    for r in range(n):
        for c in range(n):
            if r < j + k:
                assert m[r, c] == (c <= r)
            else:
                assert m[r, c] == (j <= c <= r)
    causal = np.tril(np.ones((n, n), dtype=bool))
    assert (causal & ~m).sum() == l * j


def test_masked_attention_matches_sdpa():
    rng = np.random.default_rng(4)
    j, k, l, d = 4, 3, 5, 8
    n = j + k + l
    q, kk, v = rng.standard_normal((3, n, d))
    m = gm.gist_mask(j, k, l)
    got = gm.masked_attention(q, kk, v, m, 1 / math.sqrt(d))
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None], torch.from_numpy(kk)[None],
                                         torch.from_numpy(v)[None], attn_mask=torch.from_numpy(m)[None])
    assert np.abs(got - ref[0].numpy()).max() < 1e-12


def test_cached_form_equals_full_sequence_with_gist_mask():
    """gist page, 论文做了什么 + 在线的一次 attention: rows after the gist, under
    the gist mask over [prompt; gist; query], equal attention of the query over
    [G; own K/V] with the query numbered after the gist."""
    rng = np.random.default_rng(6)
    j, k, l, Hq, Hkv, d = 6, 4, 5, 4, 2, 16
    G, n = Hq // Hkv, j + k + l
    qs = rng.standard_normal((n, Hq, d))
    ks = rng.standard_normal((n, Hkv, d))
    vs = rng.standard_normal((n, Hkv, d))
    pos = np.arange(n)
    qr = np.stack([rope_complex(qs[:, h], pos) for h in range(Hq)])     # [Hq, n, d]
    kr = np.stack([rope_complex(ks[:, g], pos) for g in range(Hkv)])    # [Hkv, n, d]
    m = torch.from_numpy(gm.gist_mask(j, k, l))
    full = F.scaled_dot_product_attention(
        torch.from_numpy(qr), torch.from_numpy(np.repeat(kr, G, axis=0)),
        torch.from_numpy(np.repeat(vs.transpose(1, 0, 2), G, axis=0)), attn_mask=m).numpy()
    want = full[:, j + k:].transpose(1, 0, 2)  # [l, Hq, d]
    pool = np.zeros((1, 1, 2, Hkv, k, d))
    pool[0, 0, 0] = kr[:, j:j + k]
    pool[0, 0, 1] = vs[j:j + k].transpose(1, 0, 2)
    got = oracle.gist_attn(qs[None, j + k:], ks[None, j + k:], vs[None, j + k:], pool,
                           item_ids=np.zeros(1, np.int32), pos_offset=np.array([j + k], np.int32),
                           dims=dims(1, l, Hq, Hkv, d, k, 1, 1), f64_inputs=True)
    assert np.abs(got[0] - want).max() < 1e-12


class TinyModel:
    """Random two-layer GQA transformer in float64 (no trained weights needed)."""

    def __init__(self, Dm=24, Hq=4, Hkv=2, d=8, L=2, seed=8):
        rng = np.random.default_rng(seed)
        s = 1 / math.sqrt(Dm)
        self.Hq, self.Hkv, self.d, self.L = Hq, Hkv, d, L
        self.W = [dict(q=rng.standard_normal((Dm, Hq * d)) * s, k=rng.standard_normal((Dm, Hkv * d)) * s,
                       v=rng.standard_normal((Dm, Hkv * d)) * s, o=rng.standard_normal((Hq * d, Dm)) * s,
                       m1=rng.standard_normal((Dm, 2 * Dm)) * s, m2=rng.standard_normal((2 * Dm, Dm)) * s)
                  for _ in range(L)]

    def proj(self, li, X):
        W, n = self.W[li], X.shape[0]
        return ((X @ W["q"]).reshape(n, self.Hq, self.d), (X @ W["k"]).reshape(n, self.Hkv, self.d),
                (X @ W["v"]).reshape(n, self.Hkv, self.d))

    def post(self, li, X, attn):  # attn [n, Hq, d]
        W = self.W[li]
        X = X + attn.reshape(X.shape[0], -1) @ W["o"]
        return X + np.tanh(X @ W["m1"]) @ W["m2"]

    def full_forward(self, X, allowed):
        """Whole sequence, positions 0..n-1, under `allowed` (torch SDPA)."""
        n, G = X.shape[0], self.Hq // self.Hkv
        pos = np.arange(n)
        kv_by_layer = []
        for li in range(self.L):
            q, k, v = self.proj(li, X)
            qr = np.stack([rope_complex(q[:, h], pos) for h in range(self.Hq)])
            kr = np.stack([rope_complex(k[:, g], pos) for g in range(self.Hkv)])
            vv = v.transpose(1, 0, 2)
            kv_by_layer.append((kr, vv))
            a = F.scaled_dot_product_attention(torch.from_numpy(qr), torch.from_numpy(np.repeat(kr, G, 0)),
                                               torch.from_numpy(np.repeat(vv, G, 0)),
                                               attn_mask=torch.from_numpy(allowed)).numpy()
            X = self.post(li, X, a.transpose(1, 0, 2))
        return X, kv_by_layer


def test_two_layer_model_offline_gist_then_online_query():
    """gist page, 在线的一次 attention: G of layer i depends on the item's states
    after layers < i, so the offline pass runs every layer and keeps each
    layer's gist K/V; the online pass then runs only the query against them."""
    j, k, l = 7, 3, 4
    tm = TinyModel()
    rng = np.random.default_rng(10)
    X = rng.standard_normal((j + k + l, 24))
    full, _ = tm.full_forward(X, gm.gist_mask(j, k, l))
    # offline: prompt + gist only (the gist mask restricted to these rows is causal)
    _, kv = tm.full_forward(X[: j + k], np.tril(np.ones((j + k, j + k), dtype=bool)))
    pool = np.zeros((1, tm.L, 2, tm.Hkv, k, tm.d))
    for li, (kr, vv) in enumerate(kv):
        pool[0, li, 0] = kr[:, j:j + k]
        pool[0, li, 1] = vv[:, j:j + k]
    # online: query rows only, numbered after the gist
    Xq = X[j + k:].copy()
    for li in range(tm.L):
        q, kk, v = tm.proj(li, Xq)
        a = oracle.gist_attn(q[None], kk[None], v[None], pool, item_ids=np.zeros(1, np.int32),
                             pos_offset=np.array([j + k], np.int32),
                             dims=dims(1, l, tm.Hq, tm.Hkv, tm.d, k, 1, 1, L=tm.L, layer=li),
                             f64_inputs=True)
        Xq = tm.post(li, Xq, a[0])
    assert np.abs(Xq - full[j + k:]).max() < 1e-10
    # storing layer-0 gist K/V for every layer is not the same thing
    bad = pool.copy()
    bad[0, 1] = bad[0, 0]
    Xb = X[j + k:].copy()
    for li in range(tm.L):
        q, kk, v = tm.proj(li, Xb)
        a = oracle.gist_attn(q[None], kk[None], v[None], bad, item_ids=np.zeros(1, np.int32),
                             pos_offset=np.array([j + k], np.int32),
                             dims=dims(1, l, tm.Hq, tm.Hkv, tm.d, k, 1, 1, L=tm.L, layer=li),
                             f64_inputs=True)
        Xb = tm.post(li, Xb, a[0])
    assert np.abs(Xb - full[j + k:]).max() > 1e-3


def test_decode_step_formula():
    """KV page, Reusable-state: o_t = softmax(q_t K_{<=t}^T / sqrt(d_k)) V_{<=t},
    K_{<=t} = [K_{<t}; k_t], here with a paged cache read through a block table."""
    P, Hq, d, bl, bpp, nb = 3, 4, 32, 16, 3, 10
    q, kn, vn = bf16((P, 1, Hq, d), 30), bf16((P, 1, Hq, d), 31), bf16((P, 1, Hq, d), 32)
    pool = bf16((nb, 1, 2, Hq, bl, d), 33)
    table = np.array([[3, 1, 7], [0, 9, 2], [5, 5, 4]], dtype=np.int32)
    got = oracle.gist_attn(q, kn, vn, pool, block_table=table, dims=dims(P, 1, Hq, Hq, d, bl, bpp, nb))
    poolf = f64(pool)
    t = bpp * bl  # default position of the new token
    for p in range(P):
        for h in range(Hq):
            Kc = np.concatenate([poolf[b, 0, 0, h] for b in table[p]])
            Vc = np.concatenate([poolf[b, 0, 1, h] for b in table[p]])
            K = np.vstack([Kc, rope_complex(f64(kn[p, 0, h]), t)])
            V = np.vstack([Vc, f64(vn[p, 0, h])])
            s = K @ rope_complex(f64(q[p, 0, h]), t) / math.sqrt(d)
            w = np.exp(s - s.max())
            o = (w / w.sum()) @ V
            assert np.abs(got[p, 0, h] - o).max() < 1e-12


def test_block_order_does_not_change_the_result():
    q, kn, vn, pool, table, pos0, D = small_case(15, bpp=3)
    a = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D)
    b = oracle.gist_attn(q, kn, vn, pool, block_table=table[:, ::-1].copy(), pos_offset=pos0, dims=D)
    assert np.abs(a - b).max() < 1e-12


def test_item_ids_equal_one_column_table():
    q, kn, vn, pool, table, pos0, D = small_case(17, bpp=1)
    a = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D)
    b = oracle.gist_attn(q, kn, vn, pool, item_ids=table[:, 0].copy(), pos_offset=pos0, dims=D)
    assert np.array_equal(a, b)


def test_explicit_scale():
    q, kn, vn, pool, table, pos0, D = small_case(19)
    d = D["head_dim"]
    a = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D)
    b = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0,
                         dims=dict(D, softmax_scale=1 / math.sqrt(d)))
    c = oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0,
                         dims=dict(D, softmax_scale=2 / math.sqrt(d)))
    assert np.abs(a - b).max() < 1e-15
    assert np.abs(a - c).max() > 1e-3


def test_out_of_range_block_is_rejected():
    q, kn, vn, pool, table, pos0, D = small_case(23)
    table[1, 0] = D["num_blocks"]
    with pytest.raises(ValueError):
        oracle.gist_attn(q, kn, vn, pool, block_table=table, pos_offset=pos0, dims=D)


def test_gather_is_bit_exact():
    q, kn, vn, pool, table, pos0, D = small_case(25, bpp=3)
    got, rc = oracle.gather(pool, block_table=table, dims=D)
    assert rc == 0
    bits = oracle.bf16_bits(pool)
    for p in range(D["num_pairs"]):
        want = np.concatenate([bits[b, D["layer"]] for b in table[p]], axis=2)  # [2, Hkv, C, d]
        assert np.array_equal(got[p], want.transpose(1, 0, 2, 3))
    table[2, 1] = -1
    got, rc = oracle.gather(pool, block_table=table, dims=D)
    assert rc == -2 and not got[2].any() and got[0].any()


# ------------------------------------------------- figures the pages print ---

def test_bytes_per_position_and_item(golden):
    for row in golden["bytes_per_position"]:
        assert oracle.kv_bytes_per_position(row["L"], row["Hkv"], row["d"], row["b"]) == row["bytes"]
    for row in golden["bytes_per_item"]:
        assert oracle.kv_bytes_per_item(row["L"], row["Hkv"], row["d"], row["k"], row["b"]) == row["bytes"]


def test_prefix_and_pool_totals(golden):
    r0, r1 = golden["prefix_item"]
    per_pos = oracle.kv_bytes_per_position(r0["L"], r0["Hkv"], r0["d"], r0["b"])
    assert round(per_pos * r0["tokens"] / 2 ** 20) == r0["printed_MiB"]
    assert round(per_pos * r1["tokens"] * r1["items"] / 1e12, 1) == r1["printed_TB"]
    for row in golden["pool_totals_100k_items_k8"]:
        gib = oracle.kv_bytes_per_item(row["L"], row["Hkv"], row["d"], 8, 2) * 100_000 / 2 ** 30
        if row["rounding"] == "one decimal":
            assert round(gib, 1) == row["printed_GiB"]
        else:
            assert int(gib) == row["printed_GiB"]


def test_shard_counts(golden):
    a, b = golden["shards_10M_items"]
    gib = oracle.kv_bytes_per_item(a["L"], a["Hkv"], a["d"], a["k"], 2) * a["items"] / 2 ** 30
    assert round(gib) == a["printed_GiB"]
    assert math.ceil(gib / a["card_GiB"]) == a["printed_M"]
    gib_b = oracle.kv_bytes_per_item(b["L"], b["Hkv"], b["d"], b["k"], 2) * b["items"] / 2 ** 30
    assert round(gib_b / b["card_GiB"]) == b["printed_M"]


def test_request_kv_formula(golden):
    """suffix page §2: 2 x L x S x H x dtype; KV page, Memory: 2 B L T h_kv d_h b."""
    for row in golden["request_kv"]:
        # hidden H = h_kv * d_h for the page's MHA model (32 heads of 128)
        got = oracle.kv_bytes_batch(row["B"], row["L"], row["S"], 32, row["H"] // 32, row["b"])
        assert got == 2 * row["B"] * row["L"] * row["S"] * row["H"] * row["b"]
        assert got / 2 ** 30 == row["printed_GB"]


def test_flop_share_and_traffic_figures(golden):
    a, b = golden["flop_share"]
    assert round(100 * 2 * a["S"] * a["D"] / (10.5 * a["D"] ** 2), 1) == a["printed_percent"]
    assert a["S"] == a["k"] + a["l"]
    assert round(5.25 * b["D"], -2) == b["printed_break_even_tokens"]
    t = golden["decode_traffic"][0]
    w_kb = t["layers"] * t["weights_MB_per_layer"] * 1e3 / t["batch"]
    assert round(w_kb, -1) == t["printed_weights_KB_per_candidate"]
    kv = t["kv_positions"] * oracle.kv_bytes_per_position(24, 2, 64, 2)
    assert kv == t["printed_kv_KiB"] * 1024
    share = kv / (w_kb * 1e3 + kv)
    assert 0.18 < share < 0.22
    assert round(t["layers"] * t["weights_MB_per_layer"] * 1e6 / kv, -3) == t["printed_break_even_batch"]
    g = golden["query_gisting"][0]
    assert 20 <= (g["N"] * g["l"]) / (g["l"] + g["N"]) < 30


# ------------------------------------------- each planted mistake is caught ---

@pytest.mark.parametrize("plant", range(1, 10))
def test_planted_mistake_is_caught(plant):
    failures = [c.__name__ for c in ALL_CHECKS if c(plant=plant) is not None]
    assert failures, f"planted mistake {plant} slipped through every pin"


# ------------------------------------------------- the fp8 (E4M3) KV pool ---

def test_e4m3_decoder_all_256_patterns():
    """Suffix page §2 / end of §5 (1-byte KV elements): the oracle's E4M3 decoder
    against torch's float8_e4m3fn conversion, every bit pattern."""
    pats = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = pats.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_f64(0x38) == 1.0 and oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9


def _fp8_case(seed, P=3, l=1, Hq=4, Hkv=4, d=32, bl=16, bpp=3, nb=7, L=2, layer=1, pow2=False):
    g = torch.Generator().manual_seed(seed)
    pool8 = torch.randn((nb, L, 2, Hkv, bl, d), generator=g).to(torch.float8_e4m3fn)
    if pow2:
        scale = 2.0 ** torch.randint(-3, 4, (nb, L, 2, Hkv), generator=g).to(torch.float32)
    else:
        scale = torch.rand((nb, L, 2, Hkv), generator=g, dtype=torch.float32) * 1.5 + 0.25
    q, kn, vn = bf16((P, l, Hq, d), seed + 1), bf16((P, l, Hkv, d), seed + 2), bf16((P, l, Hkv, d), seed + 3)
    table = np.random.default_rng(seed).integers(0, nb, size=(P, bpp)).astype(np.int32)
    D = dims(P, l, Hq, Hkv, d, bl, bpp, nb, L, layer)
    deq = pool8.to(torch.float64) * scale.to(torch.float64)[..., None, None]
    return q, kn, vn, pool8, scale, deq, table, D


def test_fp8_pool_equals_f64_oracle_on_dequantised_pool():
    q, kn, vn, pool8, scale, deq, table, D = _fp8_case(40)
    got = oracle.gist_attn_fp8kv(q, kn, vn, pool8, scale, block_table=table, dims=D)
    ref = oracle.gist_attn(f64(q), f64(kn), f64(vn), deq.numpy(), block_table=table, dims=D,
                           f64_inputs=True)
    assert np.array_equal(got, ref)


def test_fp8_pool_with_power_of_two_scales_equals_bf16_path():
    """E4M3 values times powers of two are exact bf16 values: both paths agree."""
    q, kn, vn, pool8, scale, deq, table, D = _fp8_case(41, l=3, Hq=6, Hkv=2, pow2=True)
    got = oracle.gist_attn_fp8kv(q, kn, vn, pool8, scale, block_table=table, dims=D)
    pool_bf16 = deq.to(torch.bfloat16)
    assert torch.equal(pool_bf16.to(torch.float64), deq)
    ref = oracle.gist_attn(q, kn, vn, pool_bf16, block_table=table, dims=D)
    assert np.array_equal(got, ref)


# ---------------------------------- block attention mass and the KV append ---

def test_block_mass_closed_form_and_total():
    """Suffix page §5 第三步 (attention per history block): with q = 0 every key
    weighs 1/(C+1), so a block of bl rows weighs bl/(C+1); the masses plus the new
    token's own weight sum to 1."""
    P, Hq, d, bl, bpp, nb = 2, 3, 16, 4, 3, 5
    kn, vn = bf16((P, 1, Hq, d), 50), bf16((P, 1, Hq, d), 51)
    pool = bf16((nb, 1, 2, Hq, bl, d), 52)
    table = np.array([[0, 3, 1], [4, 2, 2]], dtype=np.int32)
    D = dims(P, 1, Hq, Hq, d, bl, bpp, nb)
    _, w = oracle.gist_attn(torch.zeros((P, 1, Hq, d), dtype=torch.bfloat16), kn, vn, pool,
                            block_table=table, dims=D, want_weights=True)
    mass = oracle.block_mass(w, bpp, bl)
    assert np.allclose(mass, bl / (bpp * bl + 1), rtol=0, atol=1e-15)
    q = bf16((P, 1, Hq, d), 53)
    _, w = oracle.gist_attn(q, kn, vn, pool, block_table=table, dims=D, want_weights=True)
    mass = oracle.block_mass(w, bpp, bl)
    assert np.allclose(mass.sum(-1) + w[:, 0, :, -1], 1.0, rtol=0, atol=1e-12)


def test_kv_append_writes_rotated_key_and_value():
    """KV page, Reusable-state: the new k_t (rotated at its position) and v_t join
    the cache.  The key is checked against the complex-rotation RoPE rounded by
    torch to bf16; the value bit for bit; nothing else changes."""
    P, Hkv, d, bl, bpp, nb, L = 3, 2, 32, 8, 2, 6, 2
    kn, vn = bf16((P, 1, Hkv, d), 60), bf16((P, 1, Hkv, d), 61)
    pool = bf16((nb, L, 2, Hkv, bl, d), 62)
    table = np.array([[1, 4], [0, 5], [3, 2]], dtype=np.int32)
    slot = np.array([3, 8, 15], dtype=np.int32)
    D = dims(P, 1, Hkv, Hkv, d, bl, bpp, nb, L=L, layer=1)
    new, rc = oracle.kv_append(kn, vn, pool, table, slot, dims=D)
    assert rc == 0
    old = oracle.bf16_bits(pool)
    changed = np.argwhere(np.any(new != old, axis=-1))
    for p in range(P):
        blk, t = table[p, slot[p] // bl], slot[p] % bl
        for g in range(Hkv):
            want_k = torch.from_numpy(rope_complex(f64(kn[p, 0, g]), slot[p])).to(torch.bfloat16)
            assert np.array_equal(new[blk, 1, 0, g, t], oracle.bf16_bits(want_k))
            assert np.array_equal(new[blk, 1, 1, g, t], oracle.bf16_bits(vn[p, 0, g]))
    assert len({tuple(c[:3]) + (c[4],) for c in changed}) <= P * 2  # only the written rows
    bad = slot.copy()
    bad[1] = bpp * bl
    _, rc = oracle.kv_append(kn, vn, pool, table, bad, dims=D)
    assert rc == -2


# ------------------------------------------- offline compression: the store ---

def test_kv_store_writes_rotated_gist_rows():
    """gist page, 论文做了什么 / 在线的一次 attention: the item's cache entry is
    each layer's K/V at the k gist positions.  Keys against the complex-rotation
    RoPE rounded by torch to bf16, values bit for bit, other rows untouched."""
    P, n, Hkv, d, k, nb, L = 3, 11, 2, 32, 4, 5, 2
    kn, vn = bf16((P, n, Hkv, d), 80), bf16((P, n, Hkv, d), 81)
    pool = bf16((nb, L, 2, Hkv, k, d), 82)
    ids = np.array([4, 0, 2], dtype=np.int32)
    first = np.array([7, 0, 3], dtype=np.int32)
    spos = np.array([7, 0, 1000], dtype=np.int32)
    D = dims(P, n, Hkv, Hkv, d, k, 1, nb, L=L, layer=1)
    new, rc = oracle.kv_store(kn, vn, pool, ids, first, spos, dims=D)
    assert rc == 0
    old = oracle.bf16_bits(pool)
    for p in range(P):
        for g in range(Hkv):
            for t in range(k):
                r = first[p] + t
                want_k = torch.from_numpy(rope_complex(f64(kn[p, r, g]), spos[p] + t)).to(torch.bfloat16)
                assert np.array_equal(new[ids[p], 1, 0, g, t], oracle.bf16_bits(want_k))
                assert np.array_equal(new[ids[p], 1, 1, g, t], oracle.bf16_bits(vn[p, r, g]))
    untouched = np.ones(nb, dtype=bool)
    untouched[ids] = False
    assert np.array_equal(new[untouched], old[untouched])
    assert np.array_equal(new[:, 0], old[:, 0])  # other layer
    # default positions 0..k-1
    new0, _ = oracle.kv_store(kn, vn, pool, ids, first, None, dims=D)
    want = torch.from_numpy(rope_complex(f64(kn[0, 7 + 2, 1]), 2)).to(torch.bfloat16)
    assert np.array_equal(new0[4, 1, 0, 1, 2], oracle.bf16_bits(want))
    # rows past the sequence end, or a bad id: rejected
    _, rc = oracle.kv_store(kn, vn, pool, ids, np.array([8, 0, 3], np.int32), dims=D)
    assert rc == -2
    _, rc = oracle.kv_store(kn, vn, pool, np.array([4, 5, 2], np.int32), first, dims=D)
    assert rc == -2


def test_offline_pass_store_then_online_equals_masked_forward():
    """gist page, 论文做了什么 + 在线的一次 attention, one layer: the gist-masked
    forward over [prompt; gist; query] gives, on the query rows, what the query
    gets against the stored gist entry (gist rotated at j..j+k-1, query from
    j+k).  Equal up to the bf16 rounding of the stored keys."""
    j, k, l, Hq, Hkv, d = 9, 4, 6, 6, 2, 16
    n = j + k + l
    q, kn, vn = bf16((1, n, Hq, d), 90), bf16((1, n, Hkv, d), 91), bf16((1, n, Hkv, d), 92)
    full = oracle.gist_attn(q, kn, vn, None, dims=dims(1, n, Hq, Hkv, d, 0, 0, 0),
                            gist_start=np.array([j], np.int32), gist_len=k)
    pool0 = torch.zeros((1, 1, 2, Hkv, k, d), dtype=torch.bfloat16)
    store_dims = dims(1, n, Hkv, Hkv, d, k, 1, 1)
    entry, rc = oracle.kv_store(kn, vn, pool0, np.zeros(1, np.int32), np.array([j], np.int32),
                                np.array([j], np.int32), dims=store_dims)
    assert rc == 0
    online = oracle.gist_attn(q[:, j + k:].contiguous(), kn[:, j + k:].contiguous(),
                              vn[:, j + k:].contiguous(), entry, item_ids=np.zeros(1, np.int32),
                              pos_offset=np.array([j + k], np.int32),
                              dims=dims(1, l, Hq, Hkv, d, k, 1, 1))
    assert np.abs(online - full[:, j + k:]).max() < 1e-2
    # the unmasked (plain causal) forward differs on the query rows
    plain = oracle.gist_attn(q, kn, vn, None, dims=dims(1, n, Hq, Hkv, d, 0, 0, 0))
    assert np.abs(plain[:, j + k:] - full[:, j + k:]).max() > 5e-2
    # and the rows before the gist's end are plain causal attention
    assert np.array_equal(plain[:, : j + k], full[:, : j + k])


# ------------------------------- the projections either side of attention ---

from oracle import projections as proj  # noqa: E402


def test_qkv_rope_selects_and_rotates():
    """gist page, 在线的一次 attention (per layer: project, then attend): with a
    one-hot W_qkv the projected heads are chosen coordinates of x; Q and K are
    then rotated at cached + t (complex-rotation RoPE, written independently)."""
    P, l, Dm, Hq, Hkv, d, C = 2, 5, 24, 2, 1, 8, 7
    rng = np.random.default_rng(3)
    x = bf16((P, l, Dm), 100)
    sel = rng.integers(0, Dm, size=(Hq + 2 * Hkv) * d)
    w = torch.zeros(((Hq + 2 * Hkv) * d, Dm), dtype=torch.float32)
    w[np.arange(len(sel)), torch.from_numpy(sel)] = 1.0
    w = w.to(torch.bfloat16)
    q, k, v = proj.qkv_rope(x, w, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, cached=C)
    xf = f64(x)
    picked = xf[:, :, sel]  # [P][l][(Hq + 2Hkv) d]
    for p in range(P):
        pos = C + np.arange(l)
        for h in range(Hq):
            want = rope_complex(picked[p, :, h * d:(h + 1) * d], pos)
            assert np.abs(q[p, :, h] - want).max() < 1e-12
        want_k = rope_complex(picked[p, :, Hq * d:(Hq + 1) * d], pos)
        assert np.abs(k[p, :, 0] - want_k).max() < 1e-12
        assert np.array_equal(v[p, :, 0], picked[p, :, (Hq + Hkv) * d:])
    # given positions move the rotation
    pos_off = np.array([100, 0])
    q2, _, _ = proj.qkv_rope(x, w, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, cached=C,
                             pos_offset=pos_off)
    assert np.abs(q2[0, :, 0] - rope_complex(picked[0, :, :d], 100 + np.arange(l))).max() < 1e-12


def test_prerotated_attention_equals_in_attention_rope():
    """The attention given Q and K_new already rotated at their positions equals
    the attention that rotates them itself."""
    q, kn, vn, pool, table, pos0, D = small_case(17)
    P, l = D["num_pairs"], D["n_new"]
    qr = np.stack([np.stack([rope_complex(f64(q[p, :, h]), pos0[p] + np.arange(l))
                             for h in range(q.shape[2])], axis=1) for p in range(P)])
    kr = np.stack([np.stack([rope_complex(f64(kn[p, :, g]), pos0[p] + np.arange(l))
                             for g in range(kn.shape[2])], axis=1) for p in range(P)])
    a = oracle.gist_attn(f64(q), f64(kn), f64(vn), f64(pool), block_table=table, pos_offset=pos0,
                         dims=D, f64_inputs=True)
    b = oracle.gist_attn(qr, kr, f64(vn), f64(pool), block_table=table, pos_offset=pos0,
                         dims=dict(D, flags=1), f64_inputs=True)
    assert np.abs(a - b).max() < 1e-12
    # without the flag the rotation would be applied twice
    c = oracle.gist_attn(qr, kr, f64(vn), f64(pool), block_table=table, pos_offset=pos0, dims=D,
                         f64_inputs=True)
    assert np.abs(a - c).max() > 1e-3


def test_out_proj_closed_form():
    """A one-hot W_o picks attention columns; the projection is linear."""
    M, K, N = 6, 32, 5
    a = bf16((M, K), 110)
    cols = np.array([3, 0, 31, 7, 7])
    w = torch.zeros((N, K), dtype=torch.float32)
    w[np.arange(N), torch.from_numpy(cols)] = 1.0
    y = proj.out_proj(a, w.to(torch.bfloat16))
    assert np.array_equal(y, f64(a)[:, cols])
    w2 = bf16((N, K), 111)
    y1, y2 = proj.out_proj(a, w2), proj.out_proj(f64(a) * 2.0, w2)
    assert np.abs(y2 - 2.0 * y1).max() < 1e-12
