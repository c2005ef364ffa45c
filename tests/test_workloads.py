"""The seeded input generators: deterministic, and shaped as the workload recipes say."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import workloads as W


@pytest.mark.parametrize("name", ["tiny", "8b", "70b", "sw"])
def test_deterministic(name):
    a, b = W.make(name, "small"), W.make(name, "small")
    assert np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(a.context_lens, b.context_lens)
    assert torch.equal(a.query(), b.query())
    ka, va = a.segment_kv(0, 5)
    kb, vb = b.segment_kv(0, 5)
    assert torch.equal(ka, kb) and torch.equal(va, vb) and not torch.equal(ka, va)


def test_tiny_recipe():
    w = W.make("tiny")
    assert w.context_lens.tolist() == [5, 16, 33, 70]
    assert w.num_blocks == 64 and (w.n_q_heads, w.n_kv_heads, w.head_dim) == (2, 1, 64)
    ids = w.block_tables[w.block_tables >= 0]
    assert len(ids) == 1 + 1 + 3 + 5 == len(np.unique(ids))
    setup, (k, v, slots) = w.fill_plan()
    # the four new tokens sit at positions 4, 15, 32, 69
    assert w.new_pos.tolist() == [4, 15, 32, 69]
    assert slots.tolist() == [int(w.slot(b, [p])[0]) for b, p in enumerate([4, 15, 32, 69])]


@pytest.mark.parametrize("size", ["small", "full"])
def test_8b_recipe(size):
    w = W.make("8b", size)
    assert w.batch == (64 if size == "full" else 8)
    assert w.context_lens.min() >= 128 and w.context_lens.max() <= 4096
    need = sum(-(-int(c) // 16) for c in w.context_lens)
    assert w.num_blocks == int(np.ceil(1.2 * need))
    ids = w.block_tables[w.block_tables >= 0]
    assert len(ids) == need == len(np.unique(ids)) and ids.max() < w.num_blocks


def test_70b_shared_prefix():
    w = W.make("70b", "full")
    assert w.batch == 128 and w.context_lens.min() >= 256 and w.context_lens.max() <= 8192
    pre = w.prefix_blocks
    for b in range(w.batch):
        n = -(-int(w.context_lens[b]) // 16)
        assert np.array_equal(w.block_tables[b, :min(n, 64)], pre[:min(n, 64)])
        assert (w.block_tables[b, n:] == -1).all()
    assert w.kv_bytes_unique() < w.kv_bytes_attended()


def test_sw_only_window_blocks_mapped():
    w = W.make("sw", "full")
    for b in range(w.batch):
        c = int(w.context_lens[b])
        first, last = (c - 4096) // 16, (c - 1) // 16
        row = w.block_tables[b]
        assert (row[first:last + 1] >= 0).all()
        assert (row[:first] == -1).all() and (row[last + 1:] == -1).all()
    assert w.attended_tokens() == 32 * 4096


def test_fp8_churn_deterministic():
    a = W.make("fp8", "small", make_allocator=oracle.Allocator)
    b = W.make("fp8", "small", make_allocator=oracle.Allocator)
    assert np.array_equal(a.block_tables, b.block_tables) and a.num_blocks == b.num_blocks
    assert a.k_scale.shape == (8,) and (a.k_scale > 0).all()
