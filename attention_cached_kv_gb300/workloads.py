"""Seeded synthetic workloads shaped like the pages' settings.

This module draws random inputs and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the oracle can be fed from it.

Recipe (all tensors bf16 ~ N(0, 1); one torch.Generator per tensor, seeded
``16 * seed + stream`` with stream q=0, k_new=1, v_new=2, pool=3, ids=4; the
pool is treated as already-rotated K and plain V):

  tiny   1 layer, Hq=14, Hkv=2, d=64, k=8 gist positions, l=64; pool of 16 items;
         32 pairs with uniform item ids.
  gist   24 layers, Hq=14, Hkv=2, d=64, k=8, l=64; pool of 100k items; 256
         queries x 50 distinct candidates with Zipf(1.1) item ids (rank r has
         weight r^-1.1; ranks map to ids through a seeded permutation).
  qgist  same model, l=1 (the EOS token) against k=8 item-gist + k'=8 query-gist
         positions; 500 queries x 50 candidates; block_table[p] =
         (item, 100000 + query), so a query's gist block is shared by its 50
         adjacent candidates.
  wide   28 layers, Hq=32, Hkv=8, d=128, k=8, l=64; pool of 20k items; 128
         queries x 50 distinct uniform item ids.
  paged  32 layers, Hq=Hkv=32, d=128, l=1; 32 sequences of 4096 cached tokens in
         16 blocks of 256, block ids drawn from a seeded permutation of a
         512-block pool; the new token sits at position 4096.

Sizes come from the gist relevance page ("把 item 压成 KV：gist 能不能用在相关性任务上",
sections "收益有多大：存储" for the 24/2/64 and 28/8/128 models and "能不能再进一步"
for the query-gisted form) and from the suffix-cache page (icman.com.cn news
64898, §5: 256-token blocks behind a block table).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

STREAM_Q, STREAM_K, STREAM_V, STREAM_POOL, STREAM_IDS, STREAM_SCALE = 0, 1, 2, 3, 4, 5


@dataclass
class Spec:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    n_new: int
    block_len: int
    blocks_per_pair: int
    queries: int = 0          # gist settings: queries x candidates pairs
    candidates: int = 0
    pool_items: int = 0       # item blocks in the pool
    ids: str = "uniform"      # uniform | zipf
    query_gist: bool = False  # second cached block per pair = the query's gist
    paged_seqs: int = 0       # paged setting: sequences
    paged_pool_blocks: int = 0
    num_pairs_override: int = 0

    @property
    def num_pairs(self) -> int:
        if self.num_pairs_override:
            return self.num_pairs_override
        if self.paged_seqs:
            return self.paged_seqs
        return self.queries * self.candidates

    @property
    def num_blocks(self) -> int:
        if self.paged_seqs:
            return self.paged_pool_blocks
        return self.pool_items + (self.queries if self.query_gist else 0)


SPECS = {
    "tiny": Spec("tiny", 1, 14, 2, 64, 64, 8, 1, pool_items=16, num_pairs_override=32),
    "gist": Spec("gist", 24, 14, 2, 64, 64, 8, 1, queries=256, candidates=50,
                 pool_items=100_000, ids="zipf"),
    "qgist": Spec("qgist", 24, 14, 2, 64, 1, 8, 2, queries=500, candidates=50,
                  pool_items=100_000, ids="zipf", query_gist=True),
    "wide": Spec("wide", 28, 32, 8, 128, 64, 8, 1, queries=128, candidates=50,
                 pool_items=20_000, ids="uniform"),
    "paged": Spec("paged", 32, 32, 32, 128, 1, 256, 16, paged_seqs=32, paged_pool_blocks=512),
    # the same paged decode with the wide model's GQA heads (28 layers, 32 / 8, d 128)
    "paged_gqa": Spec("paged_gqa", 28, 32, 8, 128, 1, 256, 16, paged_seqs=32, paged_pool_blocks=512),
}


def sweep_spec(k: int, l: int) -> Spec:
    """The gist setting with k cached positions and l new tokens."""
    s = SPECS["gist"]
    return Spec(f"gist_k{k}_l{l}", s.num_layers, s.num_q_heads, s.num_kv_heads, s.head_dim,
                l, k, 1, queries=s.queries, candidates=s.candidates, pool_items=s.pool_items,
                ids="zipf")


@dataclass
class Workload:
    spec: Spec
    dims: dict                       # gist_attn_dims fields except status
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    kv_pool: torch.Tensor
    item_ids: torch.Tensor | None
    block_table: torch.Tensor | None
    pos_offset: torch.Tensor | None
    meta: dict = field(default_factory=dict)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(16 * seed + stream)
    return g


def _randn(shape, device, seed, stream) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(device, seed, stream), device=device,
                       dtype=torch.bfloat16)


def zipf_distinct(num_items: int, queries: int, per_query: int, s: float,
                  rng: np.random.Generator) -> np.ndarray:
    """[queries, per_query] ids: Zipf(s) over ranks 1..N, distinct within a query
    (duplicates are redrawn), ranks mapped to ids by a seeded permutation."""
    ranks = np.arange(1, num_items + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** -s)
    cdf /= cdf[-1]
    perm = rng.permutation(num_items)
    out = np.empty((queries, per_query), dtype=np.int64)
    for qi in range(queries):
        chosen: list[int] = []
        seen: set[int] = set()
        while len(chosen) < per_query:
            draw = np.searchsorted(cdf, rng.random(per_query), side="right")
            for r in draw:
                r = int(min(r, num_items - 1))
                if r not in seen:
                    seen.add(r)
                    chosen.append(r)
                    if len(chosen) == per_query:
                        break
        out[qi] = perm[np.array(chosen)]
    return out


def uniform_distinct(num_items: int, queries: int, per_query: int,
                     rng: np.random.Generator) -> np.ndarray:
    out = np.empty((queries, per_query), dtype=np.int64)
    for qi in range(queries):
        out[qi] = rng.choice(num_items, size=per_query, replace=False)
    return out


def dims_of(spec: Spec, layer: int = 0) -> dict:
    return dict(num_pairs=spec.num_pairs, n_new=spec.n_new, num_q_heads=spec.num_q_heads,
                num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                block_len=spec.block_len, blocks_per_pair=spec.blocks_per_pair,
                num_blocks=spec.num_blocks, num_layers=spec.num_layers, layer=layer,
                rope_theta=1e4, softmax_scale=0.0)


def make(spec: Spec | str, device="cpu", seed: int = 0, **overrides) -> Workload:
    """Draw a workload.  ``overrides`` replace Spec fields (e.g. smaller pools,
    fewer queries or layers for tests)."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    if overrides:
        spec = Spec(**{**spec.__dict__, **overrides})
    P, l, Hq, Hkv, d = spec.num_pairs, spec.n_new, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    q = _randn((P, l, Hq, d), device, seed, STREAM_Q)
    k_new = _randn((P, l, Hkv, d), device, seed, STREAM_K)
    v_new = _randn((P, l, Hkv, d), device, seed, STREAM_V)
    nb = spec.num_blocks
    kv_pool = _randn((nb, spec.num_layers, 2, Hkv, spec.block_len, d), device, seed, STREAM_POOL)

    rng = np.random.default_rng(16 * seed + STREAM_IDS)
    item_ids = block_table = None
    meta: dict = {}
    if spec.paged_seqs:
        perm = rng.permutation(nb)[: P * spec.blocks_per_pair]
        table = perm.reshape(P, spec.blocks_per_pair)
        block_table = torch.from_numpy(table.astype(np.int32)).to(device)
    else:
        if spec.queries:
            if spec.ids == "zipf":
                ids = zipf_distinct(spec.pool_items, spec.queries, spec.candidates, 1.1, rng)
            else:
                ids = uniform_distinct(spec.pool_items, spec.queries, spec.candidates, rng)
            ids = ids.reshape(-1)[:P]
        else:
            ids = rng.integers(0, spec.pool_items, size=P)
        if spec.query_gist:
            qidx = np.repeat(np.arange(spec.queries), spec.candidates)[:P]
            table = np.stack([ids, spec.pool_items + qidx], axis=1)
            block_table = torch.from_numpy(table.astype(np.int32)).to(device)
        elif spec.blocks_per_pair == 1:
            item_ids = torch.from_numpy(ids.astype(np.int32)).to(device)
        else:
            raise ValueError("gist settings use one item block per pair")
    blocks = (block_table if block_table is not None else item_ids).reshape(-1).cpu().numpy()
    meta["unique_blocks"] = int(np.unique(blocks).shape[0])
    return Workload(spec, dims_of(spec), q, k_new, v_new, kv_pool, item_ids, block_table, None, meta)


def make_custom(P: int, l: int, Hq: int, Hkv: int, d: int, block_len: int, blocks_per_pair: int,
                num_blocks: int, num_layers: int = 1, layer: int = 0, device="cpu", seed: int = 0,
                random_pos: bool = False, use_table: bool | None = None) -> Workload:
    """Any shape, for edge cases: N(0,1) tensors, uniform block ids (a block
    table unless there is exactly one block per pair and use_table is not set),
    and optionally per-pair random positions in [0, 5000)."""
    spec = Spec(f"custom_P{P}_l{l}_G{Hq // Hkv}_d{d}_C{block_len * blocks_per_pair}", num_layers,
                Hq, Hkv, d, l, block_len, blocks_per_pair, pool_items=num_blocks,
                num_pairs_override=P)
    q = _randn((P, l, Hq, d), device, seed, STREAM_Q)
    k_new = _randn((P, l, Hkv, d), device, seed, STREAM_K)
    v_new = _randn((P, l, Hkv, d), device, seed, STREAM_V)
    kv_pool = _randn((max(num_blocks, 1), num_layers, 2, Hkv, max(block_len, 1), d), device, seed,
                     STREAM_POOL)
    rng = np.random.default_rng(16 * seed + STREAM_IDS)
    ids = rng.integers(0, max(num_blocks, 1), size=(P, blocks_per_pair)).astype(np.int32)
    if use_table is None:
        use_table = blocks_per_pair != 1
    item_ids = block_table = None
    if blocks_per_pair * block_len > 0:
        if use_table:
            block_table = torch.from_numpy(ids).to(device)
        else:
            item_ids = torch.from_numpy(ids[:, 0].copy()).to(device)
    pos = None
    if random_pos:
        pos = torch.from_numpy(rng.integers(0, 5000, size=P).astype(np.int32)).to(device)
    dims = dict(num_pairs=P, n_new=l, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                block_len=block_len, blocks_per_pair=blocks_per_pair, num_blocks=num_blocks,
                num_layers=num_layers, layer=layer, rope_theta=1e4, softmax_scale=0.0)
    return Workload(spec, dims, q, k_new, v_new, kv_pool, item_ids, block_table, pos,
                    {"unique_blocks": int(np.unique(ids).shape[0])})


def make_fp8_pool(wl: Workload, seed: int = 0, chunk_blocks: int = 64):
    """An E4M3 pool of the workload's shape (float8_e4m3fn, N(0,1) draws cast to
    E4M3, generated a few blocks at a time) and fp32 scales uniform in
    [0.25, 1.75) per (block, layer, K|V, KV head).  Replaces wl.kv_pool; returns
    (pool8, scales)."""
    shape = wl.kv_pool.shape
    dev = wl.kv_pool.device
    wl.kv_pool = None
    pool8 = torch.empty(shape, dtype=torch.float8_e4m3fn, device=dev)
    g = _gen(dev, seed, STREAM_POOL)
    for b0 in range(0, shape[0], chunk_blocks):
        b1 = min(shape[0], b0 + chunk_blocks)
        part = torch.randn((b1 - b0,) + tuple(shape[1:]), generator=g, device=dev, dtype=torch.bfloat16)
        pool8[b0:b1] = part.to(torch.float8_e4m3fn)
        del part
    scale = torch.rand(tuple(shape[:4]), generator=_gen(dev, seed, STREAM_SCALE), device=dev,
                       dtype=torch.float32) * 1.5 + 0.25
    return pool8, scale
