"""Host-side logic without a GPU: the seeded workload recipes and the
benchmark's byte accounting."""
from __future__ import annotations

import numpy as np
import pytest

import bench
from attention_cached_kv_gb300 import workloads


def test_zipf_ids_are_distinct_per_query_and_skewed():
    rng = np.random.default_rng(0)
    ids = workloads.zipf_distinct(1000, 40, 50, 1.1, rng)
    assert ids.shape == (40, 50)
    for row in ids:
        assert len(set(row.tolist())) == 50
    assert ids.min() >= 0 and ids.max() < 1000
    # skewed: far fewer distinct ids than draws, hot ids repeat across queries
    counts = np.bincount(ids.reshape(-1), minlength=1000)
    assert counts.max() == 40 and (counts > 0).sum() < 0.8 * 1000


def test_qgist_block_table_shares_the_query_gist():
    wl = workloads.make("qgist", queries=6, pool_items=200, num_layers=1)
    t = wl.block_table.numpy()
    assert t.shape == (300, 2)
    assert (t[:, 0] < 200).all()
    assert (t[:, 1] == 200 + np.repeat(np.arange(6), 50)).all()


def test_paged_tables_are_a_permutation():
    wl = workloads.make("paged", paged_seqs=4, paged_pool_blocks=80, num_layers=1)
    t = wl.block_table.numpy()
    assert t.shape == (4, 16) and len(set(t.reshape(-1).tolist())) == 64
    assert wl.dims["blocks_per_pair"] * wl.dims["block_len"] == 4096


def test_workloads_are_reproducible():
    a = workloads.make("tiny")
    b = workloads.make("tiny")
    assert a.q.equal(b.q) and a.kv_pool.equal(b.kv_pool) and a.item_ids.equal(b.item_ids)
    c = workloads.make("tiny", seed=1)
    assert not a.q.equal(c.q)


def test_gist_bytes_per_pair():
    """Q + O: 64 tokens x 14 heads x 64 x 2 B each; K_new + V_new: 64 x 2 x 64 x 2 B
    each; one int32 id; one 4 KiB gist block (2 x 2 heads x 8 x 64 x 2 B)."""
    wl = workloads.make("gist", queries=2, pool_items=100, num_layers=1)
    b = bench.algorithmic_bytes_per_launch(wl)
    assert b["per_pair"] == 2 * 114688 + 2 * 16384 + 4
    assert b["per_block"] == 4096
    assert b["total"] == 100 * b["per_pair"] + b["unique_blocks"] * 4096


@pytest.mark.parametrize("name", sorted(workloads.SPECS))
def test_spec_dims_are_consistent(name):
    s = workloads.SPECS[name]
    d = workloads.dims_of(s)
    assert d["num_q_heads"] % d["num_kv_heads"] == 0
    assert d["num_blocks"] >= 1 and d["num_pairs"] >= 1
