"""GPU tests of a bf16 pool's V exponent map: one byte per (block, KV head,
token), the largest exponent field of the token's V row, which
paged_kv_write records, paged_kv_copy_blocks moves, kv_pool_refresh_exponent_map
recomputes and the prefill reads to scale its f16 copy of V.

The expected bytes are computed here from the bf16 bits of the rows (the
exponent field is the format's definition: bits 14..7, at least 1); a row
never recorded holds 0, and a prefill attending to it reports the stale map.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv

from _parity import BF16_MAX_ABS, BF16_REL_L2, errors, poison

pytestmark = pytest.mark.gpu


def _row_exponents(v: torch.Tensor) -> torch.Tensor:
    """[T, Hkv, D] bf16 -> [T, Hkv] the largest exponent field, at least 1."""
    bits = v.contiguous().view(torch.int16).to(torch.int32) & 0x7F80
    return torch.clamp((bits >> 7).amax(dim=2), min=1).to(torch.uint8)


@pytest.mark.parametrize("bs,d", [(16, 128), (32, 128), (16, 64)])
def test_write_records_row_exponents(bs, d):
    nb, hkv = 12, 4
    pool = pagedkv.KVPool(nb, bs, hkv, d)
    emap = pool.exponent_map()
    assert emap is not None and tuple(emap.shape) == (nb, hkv, bs)
    assert int(emap.max()) == 0                              # nothing recorded yet
    g = torch.Generator().manual_seed(3)
    T = 40
    k = torch.randn(T, hkv, d, generator=g).bfloat16()
    v = (torch.randn(T, hkv, d, generator=g) * torch.logspace(-30, 30, T).view(T, 1, 1)).bfloat16()
    v[0] = 0.0                                               # an all-zero row: stored as 1
    v[1, 0, 5] = float("inf")                                # exponent field 255
    v[2, 1, :] = 2.0 ** -130                                 # subnormal bf16: field 0 -> 1
    slots = torch.from_numpy(np.random.default_rng(4).permutation(nb * bs)[:T].astype(np.int64))
    slots[::9] = -1                                          # padded tokens: no entry
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), slots.cuda())
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    got = emap.cpu()
    want = torch.zeros(nb, hkv, bs, dtype=torch.uint8)
    ex = _row_exponents(v)
    for t in range(T):
        s = int(slots[t])
        if s >= 0:
            want[s // bs, :, s % bs] = ex[t]
    assert torch.equal(got, want)
    assert int(ex[0].max()) == 1 and int(ex[1, 0]) == 255 and int(ex[2, 1]) == 1
    pool.destroy()


def test_decode_step_records_the_new_rows():
    """The fused decode step writes through the same kernel: its new tokens'
    rows get their entries too."""
    nb, hkv, hq, d, B = 8, 2, 8, 128, 3
    pool = pagedkv.KVPool(nb, 16, hkv, d)
    g = torch.Generator().manual_seed(9)
    lens = torch.tensor([5, 17, 30], dtype=torch.int32)
    tables = torch.tensor([[0, -1], [1, 2], [3, 4]], dtype=torch.int32)
    T = int(lens.sum())
    kv = (torch.randn(T, hkv, d, generator=g) * 3).bfloat16()
    slots = torch.cat([tables[b, torch.arange(int(lens[b]) - 1) // 16].long() * 16
                       + torch.arange(int(lens[b]) - 1) % 16 for b in range(B)])
    pagedkv.paged_kv_write(pool, kv[:slots.numel()].cuda(), kv[:slots.numel()].cuda(), slots.cuda())
    k_new = torch.randn(B, hkv, d, generator=g).bfloat16()
    v_new = (torch.randn(B, hkv, d, generator=g) * 2.0 ** 12).bfloat16()
    pos = lens.long() - 1
    new_slots = tables[torch.arange(B), pos // 16].long() * 16 + pos % 16
    q = torch.randn(B, hq, d, generator=g).bfloat16()
    pagedkv.paged_decode_step(pool, k_new.cuda(), v_new.cuda(), new_slots.cuda(), q.cuda(),
                              tables.cuda(), lens.cuda(), d ** -0.5, 0)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    emap = pool.exponent_map().cpu()
    ex = _row_exponents(v_new)
    for b in range(B):
        s_ = int(new_slots[b])
        assert torch.equal(emap[s_ // 16, :, s_ % 16], ex[b])
    pool.destroy()


def test_copy_moves_the_map_and_refresh_recomputes_it():
    nb, hkv, d = 10, 2, 128
    pool = pagedkv.KVPool(nb, 16, hkv, d)
    g = torch.Generator().manual_seed(5)
    T = nb * 16
    v = (torch.randn(T, hkv, d, generator=g) * torch.logspace(-8, 8, T).view(T, 1, 1)).bfloat16()
    pagedkv.paged_kv_write(pool, v.cuda(), v.cuda(), torch.arange(T, dtype=torch.int64).cuda())
    emap = pool.exponent_map()
    before = emap.clone()
    pairs = np.array([[1, 7], [7, 2], [3, 3], [9, 0]], np.int32)   # a chain, a self-copy
    pagedkv.paged_kv_copy_blocks(pool, pairs)
    torch.cuda.synchronize()
    want = before.clone()
    for s, dst in pairs:                                     # applied one after another
        want[dst] = want[s]
    assert torch.equal(emap, want)
    # V changed through the pool's memory: the refresh recomputes every entry
    raw = pool.view()
    raw[4, :, 1] = (torch.randn(hkv, 16, d, generator=g) * 2.0 ** 40).bfloat16().cuda()
    raw[5, :, 1] = 0.0
    emap.zero_()
    pool.refresh_exponent_map()
    torch.cuda.synchronize()
    rows = raw[:, :, 1].reshape(nb * hkv * 16, d).cpu()
    assert torch.equal(emap.reshape(-1).cpu(), _row_exponents(rows.view(-1, 1, d)).view(-1))
    pool.destroy()


def _pools_with_v_written_directly(seed, scale_late):
    """One sequence whose K/V go into the GPU pool through view(), so the
    exponent map holds nothing for them; V of key tiles 2.. is scaled by
    `scale_late`."""
    hkv, hq, ctx, bs = 2, 8, 600, 16
    nblk = -(-ctx // bs)
    tables = np.random.default_rng(seed).permutation(nblk + 2)[:nblk].astype(np.int32).reshape(1, nblk)
    pool = pagedkv.KVPool(nblk + 2, bs, hkv, 128)
    poison(pool)
    opool = oracle.Pool(nblk + 2, bs, hkv, 128, "bf16")
    g = torch.Generator().manual_seed(seed + 1)
    k = torch.randn(ctx, hkv, 128, generator=g).bfloat16()
    f = torch.tensor([1.0 if i < 256 else scale_late for i in range(ctx)]).view(ctx, 1, 1)
    v = (torch.randn(ctx, hkv, 128, generator=g) * f).bfloat16()
    pos = np.arange(ctx)
    blk, off = tables[0, pos // bs], pos % bs
    raw = pool.view()
    bi, oi = torch.from_numpy(blk).long().cuda(), torch.from_numpy(off).long().cuda()
    raw[bi, :, 0, oi] = k.cuda()
    raw[bi, :, 1, oi] = v.cuda()
    opool.write(k, v, (blk.astype(np.int64) * bs + off))
    q = torch.randn(200, hq, 128, generator=g).bfloat16()
    return pool, opool, q, tables, np.array([0, 200], np.int32), np.array([ctx], np.int32)


def _prefill(pool, q, tables, cu, lens):
    out = pagedkv.paged_prefill_attention(
        pool, q.cuda(), torch.from_numpy(cu).cuda(), torch.from_numpy(tables).cuda(),
        torch.from_numpy(lens).cuda(), 128 ** -0.5, 0, max_q_len=200, max_context_len=int(lens[0]))
    torch.cuda.synchronize()
    return out


def _check(out, opool, q, tables, cu, lens, label):
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5)
    got = out.cpu().numpy()
    assert np.isfinite(got).all(), label
    unit = float(np.abs(ref).max())
    max_abs, rel = errors(got / unit, ref / unit)
    print(f"PARITY prefill {label} max_abs/unit={max_abs:.3e} rel_l2={rel:.3e}")
    assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, (label, max_abs, rel)


def test_prefill_without_map_entries_reports_then_refresh():
    """V written through the pool's memory leaves the map without entries:
    the prefill says so; after the refresh it is right (later tiles 2^20
    larger, so the power of two is raised along the way)."""
    pool, opool, q, tables, cu, lens = _pools_with_v_written_directly(41, 2.0 ** 20)
    assert int(pool.exponent_map().max()) == 0
    _prefill(pool, q, tables, cu, lens)
    assert pool.check_status() == 10                        # KV_ERR_STALE_EXPONENT_MAP
    pool.refresh_exponent_map()
    out = _prefill(pool, q, tables, cu, lens)
    assert pool.check_status() == pagedkv.KV_OK
    _check(out, opool, q, tables, cu, lens, "V written directly, map refreshed")
    pool.destroy()


def test_prefill_after_overwrite_and_refresh():
    """Rows first written through paged_kv_write with small values, then
    overwritten through the pool's memory with values 2^30 larger: after the
    refresh the prefill is right again."""
    pool, opool, q, tables, cu, lens = _pools_with_v_written_directly(43, 2.0 ** 30)
    ctx, bs = int(lens[0]), pool.block_size
    pos = np.arange(ctx)
    slots = torch.from_numpy(tables[0, pos // bs].astype(np.int64) * bs + pos % bs)
    small = torch.full((ctx, pool.n_kv_heads, 128), 2.0 ** -10).bfloat16()
    raw = pool.view()
    keep = raw.clone()
    pagedkv.paged_kv_write(pool, small.cuda(), small.cuda(), slots.cuda())   # map: small exponents
    torch.cuda.synchronize()
    raw.copy_(keep)                                          # the large values again, map unchanged
    pool.refresh_exponent_map()
    out = _prefill(pool, q, tables, cu, lens)
    assert pool.check_status() == pagedkv.KV_OK
    _check(out, opool, q, tables, cu, lens, "V overwritten, map refreshed")
    pool.destroy()
