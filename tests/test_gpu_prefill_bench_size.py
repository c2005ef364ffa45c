"""Prefill parity at the sizes bench.py times: full causal prefills of 4 x 2,048
and 4 x 8,192 tokens with 32 query / 8 KV heads, head_dim 128, 16-token
blocks in shuffled tables, over bf16, FP8 and FP4 pools, launched as the bench
launches them (one call for the whole batch).

The oracle computes sampled output rows one by one: token i of sequence b is
the last (only) new token of a prefill whose context ends at its position, so
a one-token oracle prefill over the same pool and table gives its row.  The
samples cover the first and last tokens, block edges and 128-key tile edges.
Bars: bf16 and FP4 the decode's bf16 bar (max |err| 2e-3, relative L2 1e-3);
FP8 the FP8 bar (3e-2) and the relative L2 bound of its tests (1e-2).
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv

from _parity import BF16_MAX_ABS, BF16_REL_L2, FP8_MAX_ABS, errors

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS = 32, 8, 128, 16


@pytest.mark.parametrize("ctx", [2048, 8192])
@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp4"])
def test_prefill_bench_size_sampled_rows(dtype, ctx):
    B = 4
    nblk = ctx // BS
    tables = np.random.default_rng(3).permutation(B * nblk).astype(np.int32).reshape(B, nblk)
    g = torch.Generator().manual_seed(5 + ctx)
    k = torch.randn(B * ctx, HKV, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B * ctx, HKV, D, generator=g).to(torch.bfloat16)
    q = torch.randn(B * ctx, HQ, D, generator=g).to(torch.bfloat16)
    pos = np.arange(ctx)
    slots = (tables[:, pos // BS].astype(np.int64) * BS + pos % BS).reshape(-1)
    pool = pagedkv.KVPool(B * nblk, BS, HKV, D, dtype)
    opool = oracle.Pool(B * nblk, BS, HKV, D, dtype)
    if dtype in ("fp8", "fp4"):   # randn bf16: |x| < 4.5 at these sizes
        sc = np.full(HKV, 4.5 / (448 if dtype == "fp8" else 6 * 448), np.float32)
        pool.set_scales(torch.from_numpy(sc).cuda(), torch.from_numpy(sc).cuda())
        opool.set_scales(sc, sc)
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda())
    opool.write(k, v, slots)
    cu = np.arange(0, B * ctx + 1, ctx, dtype=np.int32)
    lens = np.full(B, ctx, np.int32)
    scale = 128 ** -0.5
    out = pagedkv.paged_prefill_attention(
        pool, q.cuda(), torch.from_numpy(cu).cuda(), torch.from_numpy(tables).cuda(),
        torch.from_numpy(lens).cuda(), scale, 0, max_q_len=ctx, max_context_len=ctx)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    got_all = out.cpu().numpy()
    samples = [(0, 0), (0, 1), (1, 15), (1, 16), (2, 127), (2, 128), (3, 129), (3, 255),
               (0, 1000), (1, ctx // 2 + 7), (2, ctx - 129), (3, ctx - 1)]
    got, ref = [], []
    for b, i in samples:
        row = b * ctx + i
        ref.append(opool.prefill(q[row:row + 1], np.array([0, 1], np.int32), tables[b:b + 1],
                                 np.array([i + 1], np.int32), scale)[0])
        got.append(got_all[row])
    got, ref = np.stack(got), np.stack(ref)
    assert np.isfinite(got).all()
    max_abs, rel = errors(got, ref)
    print(f"PARITY prefill bench-size {dtype} 4x{ctx} ({len(samples)} rows) "
          f"max_abs={max_abs:.3e} rel_l2={rel:.3e}")
    if dtype == "fp8":
        assert max_abs <= FP8_MAX_ABS and rel <= 1e-2
    else:   # bf16, and FP4 (values exact in f16)
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2
    pool.destroy()
