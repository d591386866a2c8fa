"""The linear layers on either side of the attention, in float64 -- TEST
INFRASTRUCTURE ONLY.

[Gist page, "在线的一次 attention"] ("把 item 压成 KV：gist 能不能用在相关性任务上"):
per layer the new tokens' hidden states X are projected to Q, K, V, the
attention runs, and its output goes through the output projection before the
MLP.  Here the projections are plain matrix products of the bf16 inputs,
widened exactly to float64; the query and key heads are then rotated at their
positions (rotate-half RoPE, the same reading the attention oracle takes), so
that the attention can be given pre-rotated inputs.  Weights are synthetic:
nothing here claims model quality.

Layouts (row-major):
  x      [P][l][D_model]
  w_qkv  [(Hq + 2 Hkv) d][D_model]   rows: q heads, then k heads, then v heads
  w_o    [D_model][Hq d]
"""
from __future__ import annotations

import numpy as np

from . import bf16_bits


def _f64(t) -> np.ndarray:
    """bf16 tensor or bit array -> float64, exactly."""
    bits = bf16_bits(t).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def rope_rows(x: np.ndarray, pos: np.ndarray, theta: float = 1e4) -> np.ndarray:
    """Rotate-half RoPE of x[..., n, d] at positions pos[n]: the pair (j, j + d/2)
    turns by the angle pos * theta^(-2j/d)."""
    d = x.shape[-1]
    h = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta ** (-2.0 * np.arange(h) / d)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def qkv_rope(x, w_qkv, *, num_q_heads: int, num_kv_heads: int, head_dim: int, cached: int,
             pos_offset=None, theta: float = 1e4):
    """Q, K_new, V_new of the new tokens ([P][l][H][d] each, float64), Q and K
    rotated at positions pos_offset[p] + t (default: cached + t)."""
    xf = _f64(x)
    P, l, _ = xf.shape
    W = _f64(w_qkv)
    y = xf.reshape(P * l, -1) @ W.T  # [P*l][(Hq + 2Hkv) d]
    Hq, Hkv, d = num_q_heads, num_kv_heads, head_dim
    q = y[:, : Hq * d].reshape(P, l, Hq, d)
    k = y[:, Hq * d:(Hq + Hkv) * d].reshape(P, l, Hkv, d)
    v = y[:, (Hq + Hkv) * d:].reshape(P, l, Hkv, d)
    base = np.full(P, cached) if pos_offset is None else np.asarray(pos_offset).reshape(P)
    qr, kr = np.empty_like(q), np.empty_like(k)
    for p in range(P):
        pos = base[p] + np.arange(l)
        qr[p] = rope_rows(q[p].transpose(1, 0, 2), pos, theta).transpose(1, 0, 2)
        kr[p] = rope_rows(k[p].transpose(1, 0, 2), pos, theta).transpose(1, 0, 2)
    return qr, kr, v


def out_proj(attn, w_o) -> np.ndarray:
    """Y = attn W_o^T: attn [..., Hq d] (bf16 or float64), w_o [D_model][Hq d] bf16."""
    a = attn if isinstance(attn, np.ndarray) and attn.dtype == np.float64 else _f64(attn)
    return a @ _f64(w_o).T
