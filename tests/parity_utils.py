"""Helpers for the GPU parity tests: run the library, run the oracle on the
same inputs (optionally a sample of pairs), compare with the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from attention_cached_kv_gb300 import binding

# bf16 inputs and output, fp32 accumulation: |got - ref| <= ATOL + RTOL * |ref|
ATOL = 1e-2
RTOL = 1e-2


def run_gpu(wl, layer=0, status=None, out=None):
    dims = dict(wl.dims, layer=layer)
    return binding.gist_attn_fwd(wl.q, wl.k_new, wl.v_new, wl.kv_pool, wl.item_ids,
                                 wl.block_table, wl.pos_offset, out, dims=dims, status=status)


def oracle_ref(wl, layer=0, pairs=None):
    """Oracle output (float64 numpy) for the given pairs (all if None).

    Only the selected pairs' rows and the pool blocks they name are copied to
    the host; block ids are renumbered into that compact pool."""
    P = wl.dims["num_pairs"]
    sel = np.arange(P) if pairs is None else np.asarray(pairs)
    idx = torch.from_numpy(sel).to(wl.q.device)
    q = wl.q.index_select(0, idx)
    kn = wl.k_new.index_select(0, idx)
    vn = wl.v_new.index_select(0, idx)
    dims = dict(wl.dims, num_pairs=len(sel), num_layers=1, layer=0)
    C = wl.dims["block_len"] * wl.dims["blocks_per_pair"]
    pool = ids = table = None
    if C > 0:
        src = wl.block_table if wl.block_table is not None else wl.item_ids.view(-1, 1)
        blocks = src.index_select(0, idx).cpu().numpy()
        uniq, inv = np.unique(blocks, return_inverse=True)
        inv = inv.reshape(blocks.shape).astype(np.int32)
        pool = wl.kv_pool[:, layer].index_select(0, torch.from_numpy(uniq).to(wl.q.device).long())
        pool = pool.unsqueeze(1).contiguous()
        dims["num_blocks"] = len(uniq)
        if wl.block_table is not None:
            table = inv
        else:
            ids = inv[:, 0].copy()
    pos = None if wl.pos_offset is None else wl.pos_offset.index_select(0, idx)
    return oracle.gist_attn(q, kn, vn, pool, item_ids=ids, block_table=table, pos_offset=pos,
                            dims=dims)


def compare(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    """Element-wise |got - ref| <= ATOL + RTOL |ref|; returns the worst excess ratio."""
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = float((err / bound).max()) if err.size else 0.0
    if worst > 1.0:
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: |d|={err[i]:.3e} > bound {bound[i]:.3e} at {i} "
                             f"(got {g[i]:.5f}, ref {ref[i]:.5f}); max|d|={err.max():.3e}")
    return worst


def oracle_ref_fp8(wl, pool8, scale, layer=0, pairs=None):
    """Oracle output for an E4M3 pool, copying only the selected pairs' blocks."""
    P = wl.dims["num_pairs"]
    sel = np.arange(P) if pairs is None else np.asarray(pairs)
    idx = torch.from_numpy(sel).to(wl.q.device)
    src = wl.block_table if wl.block_table is not None else wl.item_ids.view(-1, 1)
    blocks = src.index_select(0, idx).cpu().numpy()
    uniq, inv = np.unique(blocks, return_inverse=True)
    inv = inv.reshape(blocks.shape).astype(np.int32)
    u = torch.from_numpy(uniq).to(wl.q.device).long()
    p8 = pool8.view(torch.uint8)[:, layer].index_select(0, u).unsqueeze(1).contiguous()
    sc = scale[:, layer].index_select(0, u).unsqueeze(1).contiguous()
    dims = dict(wl.dims, num_pairs=len(sel), num_layers=1, layer=0, num_blocks=len(uniq))
    table = inv if wl.block_table is not None else None
    ids = None if wl.block_table is not None else inv[:, 0].copy()
    pos = None if wl.pos_offset is None else wl.pos_offset.index_select(0, idx)
    return oracle.gist_attn_fp8kv(wl.q.index_select(0, idx), wl.k_new.index_select(0, idx),
                                  wl.v_new.index_select(0, idx), p8, sc, item_ids=ids,
                                  block_table=table, pos_offset=pos, dims=dims)
