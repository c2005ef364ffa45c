"""paged_decode_attention_noalloc: the decode entry point for callers that
cannot allocate device memory at call time (its split-K scratch is a static
device array inside the library).  It must give the workspace entry point's
results, call after call, and refuse sizes whose scratch would not fit.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""

import numpy as np
import pytest
import torch

from paged_kv_cache_33_gb300 import pagedkv
from paged_kv_cache_33_gb300 import workloads as W

from _parity import BF16_MAX_ABS, BF16_REL_L2, errors, fill_both, make_gpu_pool

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 * 1024 * 1024   # PAGED_DECODE_STATIC_SCRATCH_BYTES in pagedkv.h


@pytest.mark.parametrize("name,part_blocks", [("8b", 8), ("sw", 4), ("70b", 12)])
def test_matches_workspace_entry_point_on_two_calls_in_a_row(name, part_blocks):
    w = W.make(name, "small")
    pool = make_gpu_pool(w)
    pool.set_partition_blocks(part_blocks)   # several partitions: the scratch is really used
    fill_both(w, pool, None)
    need = pagedkv.paged_decode_workspace_bytes(pool, w.batch, w.n_q_heads, w.max_context_len,
                                                w.window)
    assert 0 < need <= STATIC_SCRATCH_BYTES
    tables = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.context_lens).cuda()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for call in range(2):
        g = torch.Generator().manual_seed(100 + call)   # a different query each call
        q = torch.randn(w.batch, w.n_q_heads, w.head_dim, generator=g).bfloat16().cuda()
        ref = pagedkv.paged_decode_attention(pool, q, tables, lens, w.scale, w.window,
                                             max_context_len=w.max_context_len, workspace=ws)
        out = torch.full_like(ref, float("nan"))
        pagedkv.paged_decode_attention_noalloc(pool, q, tables, lens, w.scale, w.window,
                                               w.max_context_len, out)
        torch.cuda.synchronize()
        assert pool.check_status() == pagedkv.KV_OK
        got, want = out.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(got).all()
        max_abs, rel = errors(got, want)
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, (name, call, max_abs, rel)
    pool.destroy()


def test_refuses_sizes_beyond_the_static_scratch():
    pool = pagedkv.KVPool(64, 16, 8, 128)
    pool.set_partition_blocks(4)
    B, Hq, ctx = 1024, 64, 8192
    assert pagedkv.paged_decode_workspace_bytes(pool, B, Hq, ctx) > STATIC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros(B, ctx // 16, dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.zeros(B, Hq, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(pagedkv.KVError) as e:
        pagedkv.paged_decode_attention_noalloc(pool, q, tables, lens, 0.1, 0, ctx, out)
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert not out.any()   # nothing was launched
    pool.destroy()


def test_pinned_host_output_and_undersized_output():
    w = W.make("8b", "small")
    pool = make_gpu_pool(w)
    pool.set_partition_blocks(8)
    fill_both(w, pool, None)
    tables = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.context_lens).cuda()
    q = torch.randn(w.batch, w.n_q_heads, w.head_dim,
                    generator=torch.Generator().manual_seed(7)).bfloat16().cuda()
    ref = pagedkv.paged_decode_attention(pool, q, tables, lens, w.scale, w.window,
                                         max_context_len=w.max_context_len)
    host = torch.full(tuple(ref.shape), float("nan")).pin_memory()
    pagedkv.paged_decode_attention_noalloc(pool, q, tables, lens, w.scale, w.window,
                                           w.max_context_len, host)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    max_abs, rel = errors(host.numpy(), ref.cpu().numpy())
    assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2
    small = torch.zeros(w.batch, w.n_q_heads - 1, w.head_dim, device="cuda")
    with pytest.raises(ValueError):
        pagedkv.paged_decode_attention_noalloc(pool, q, tables, lens, w.scale, w.window,
                                               w.max_context_len, small)
    pool.destroy()
