"""Training-side view of gisting, for brute-force pins -- TEST INFRASTRUCTURE ONLY.

[Gist page, "论文做了什么"] ("把 item 压成 KV：gist 能不能用在相关性任务上"):
training changes only the attention mask.  Over the sequence
[prompt (j tokens); gist (k tokens); rest (l tokens)] it is the ordinary causal
mask with the lower-left block removed: tokens after the gist may not see
tokens before it, so the prompt reaches them only through the k gist
positions.  [Gist page, "在线的一次 attention"]: at inference the prompt is gone
and its gist K/V sit in a cache; the new tokens are numbered after them.

These functions are the plain definitions (float64 numpy, explicit loops over
rows), used to show that the cached form the oracle and the CUDA library
compute equals full-sequence attention under the gist mask.
"""
from __future__ import annotations

import numpy as np


def gist_mask(j: int, k: int, l: int) -> np.ndarray:
    """allowed[r, c] over n = j + k + l positions: causal, minus the block
    (rows after the gist) x (columns before the gist)."""
    n = j + k + l
    allowed = np.zeros((n, n), dtype=bool)
    for r in range(n):
        for c in range(r + 1):
            post_gist_row = r >= j + k
            pre_gist_col = c < j
            allowed[r, c] = not (post_gist_row and pre_gist_col)
    return allowed


def rope_rotate_half(x: np.ndarray, pos: np.ndarray, theta: float = 1e4) -> np.ndarray:
    """Rotate-half RoPE of rows x[n, d] at positions pos[n] (float64)."""
    n, d = x.shape
    half = d // 2
    y = np.empty_like(x, dtype=np.float64)
    for r in range(n):
        for jj in range(half):
            a = float(pos[r]) * theta ** (-2.0 * jj / d)
            c, s = np.cos(a), np.sin(a)
            y[r, jj] = x[r, jj] * c - x[r, jj + half] * s
            y[r, jj + half] = x[r, jj + half] * c + x[r, jj] * s
    return y


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, allowed: np.ndarray,
                     scale: float) -> np.ndarray:
    """Softmax attention of rows q[n, d] over keys k[m, d], values v[m, dv],
    restricted to allowed[n, m] (every row must allow at least one key)."""
    n = q.shape[0]
    out = np.zeros((n, v.shape[1]), dtype=np.float64)
    for r in range(n):
        cols = np.nonzero(allowed[r])[0]
        s = np.array([scale * float(np.dot(q[r], k[c])) for c in cols])
        w = np.exp(s - s.max())
        w /= w.sum()
        out[r] = (w[:, None] * v[cols]).sum(axis=0)
    return out
