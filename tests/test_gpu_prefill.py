"""GPU parity of paged prefill (extend) attention on tcgen05 against the fp64
oracle.

Tolerance: the bf16 KV bar of the decode (max |err| <= 2e-3, relative L2
<= 1e-3).  The kernel hands P to the P V product as one f16 per weight
(relative rounding <= 2^-11) and V as f16 values scaled by a power of two
that keeps them exact, and accumulates in fp32: errors of 2^-11 per weight
give a few 1e-4 on the output, below the bar (one bf16 P, 2^-8 per weight,
would not be).
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv

from _parity import BF16_MAX_ABS as MAX_ABS
from _parity import BF16_REL_L2 as REL_L2
from _parity import compare_pools, errors, poison

pytestmark = pytest.mark.gpu


def _build(ctx_lens, q_lens, hq, hkv, bs=16, seed=0, extra_blocks=5):
    """Pools (GPU poisoned, oracle) holding every context token; the queries
    of the last q_len positions; shuffled tables."""
    rng = np.random.default_rng(seed)
    ctx_lens = np.asarray(ctx_lens, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    B = len(ctx_lens)
    nblk = [max(1, -(-int(c) // bs)) for c in ctx_lens]
    nb = sum(nblk) + extra_blocks
    ids = rng.permutation(nb).astype(np.int32)
    tables = np.full((B, max(nblk)), -1, np.int32)
    at = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = ids[at:at + n]
        at += n
    g = torch.Generator().manual_seed(seed + 1)
    pool = pagedkv.KVPool(nb, bs, hkv, 128, "bf16")
    poison(pool)
    opool = oracle.Pool(nb, bs, hkv, 128, "bf16")
    for b, c in enumerate(ctx_lens):
        if c == 0:
            continue
        k = torch.randn(int(c), hkv, 128, generator=g).to(torch.bfloat16)
        v = torch.randn(int(c), hkv, 128, generator=g).to(torch.bfloat16)
        pos = np.arange(int(c))
        slots = (tables[b, pos // bs].astype(np.int64) * bs + pos % bs)
        pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda())
        opool.write(k, v, slots)
    T = int(q_lens.sum())
    q = torch.randn(T, hq, 128, generator=g).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return pool, opool, q, cu, tables, ctx_lens


def _run(pool, q, cu, tables, lens, scale, window=0):
    return pagedkv.paged_prefill_attention(
        pool, q.cuda(), torch.from_numpy(cu).cuda(), torch.from_numpy(tables).cuda(),
        torch.from_numpy(lens).cuda(), scale, window,
        max_q_len=int((cu[1:] - cu[:-1]).max()), max_context_len=int(lens.max()))


def _check(out, ref, label):
    got = out.cpu().numpy()
    assert np.isfinite(got).all(), label
    max_abs, rel = errors(got, ref)
    print(f"PARITY prefill {label} max_abs={max_abs:.3e} rel_l2={rel:.3e}")
    assert max_abs <= MAX_ABS and rel <= REL_L2, (label, max_abs, rel)


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (16, 2), (3, 1), (12, 2)])
def test_prefill_matches_oracle(hq, hkv, bs):
    # full prompts, cached prefixes with short and long tails, q_len 1 and 0
    ctx = [1, 16, 17, 63, 64, 65, 200, 300, 129, 90]
    ql = [1, 16, 5, 63, 1, 30, 200, 77, 0, 90]
    pool, opool, q, cu, tables, lens = _build(ctx, ql, hq, hkv, bs=bs, seed=hq * 10 + hkv + bs)
    out = _run(pool, q, cu, tables, lens, 128 ** -0.5)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5)
    _check(out, ref, f"hq={hq} hkv={hkv} bs={bs}")
    pool.destroy()


@pytest.mark.parametrize("window", [1, 7, 64, 100, 5000])
def test_prefill_sliding_window(window):
    ctx = [50, 300, 700]
    ql = [50, 120, 300]
    pool, opool, q, cu, tables, lens = _build(ctx, ql, 16, 4, seed=window)
    # blocks wholly before every window of the sequence are unmapped
    for b, c in enumerate(lens):
        first_pos = int(c) - int(ql[b])
        lo = max(0, first_pos + 1 - window)
        tables[b, : lo // 16] = -1
    out = _run(pool, q, cu, tables, lens, 0.1, window)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 0.1, window)
    _check(out, ref, f"window={window}")
    pool.destroy()


def test_prefill_long_prompt_many_tiles():
    # several query tiles and many key tiles per (sequence, KV head)
    pool, opool, q, cu, tables, lens = _build([2048, 1500], [300, 1500], 8, 2, seed=3)
    out = _run(pool, q, cu, tables, lens, 128 ** -0.5)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5)
    _check(out, ref, "long")
    pool.destroy()


def test_prefill_last_token_matches_decode():
    pool, opool, q, cu, tables, lens = _build([77, 300], [20, 33], 8, 2, seed=11)
    out = _run(pool, q, cu, tables, lens, 0.09)
    last = q[torch.from_numpy(cu[1:] - 1).long()]
    dec = pagedkv.paged_decode_attention(pool, last.cuda(), torch.from_numpy(tables).cuda(),
                                         torch.from_numpy(lens).cuda(), 0.09,
                                         max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    got = out.cpu().numpy()[cu[1:] - 1]
    max_abs, _ = errors(got, dec.cpu().numpy())
    assert max_abs <= MAX_ABS
    pool.destroy()


def test_prefill_bad_block_and_bad_context():
    pool, opool, q, cu, tables, lens = _build([100, 100], [40, 40], 8, 2, seed=13)
    bad = tables.copy()
    bad[0, 2] = pool.num_blocks + 3
    out = _run(pool, q, cu, bad, lens, 0.1)
    torch.cuda.synchronize()
    assert pool.check_status() == 5                        # KV_ERR_BAD_BLOCK_ID
    ref = opool.prefill(q, cu, tables, lens, 0.1)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    r1 = slice(cu[1], cu[2])                                # the other sequence is unaffected
    max_abs, _ = errors(got[r1], ref[r1])
    assert max_abs <= MAX_ABS
    # q_len above the context: reported, skipped
    lens2 = lens.copy()
    lens2[1] = 30
    _run(pool, q, cu, tables, lens2, 0.1)
    torch.cuda.synchronize()
    assert pool.check_status() == 8                        # KV_ERR_BAD_CONTEXT
    pool.destroy()


def test_prefill_host_checks():
    pool = pagedkv.KVPool(8, 16, 2, 128)
    q = torch.zeros(4, 4, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    t = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
    c = torch.tensor([4], dtype=torch.int32, device="cuda")
    with pytest.raises(pagedkv.KVError):
        pagedkv.paged_prefill_attention(pool, q, cu, t, c, 0.1, max_q_len=4, max_context_len=64)
    d64 = pagedkv.KVPool(8, 16, 2, 64)                      # head_dim 64: no prefill
    q64 = torch.zeros(4, 4, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pagedkv.KVError):
        pagedkv.paged_prefill_attention(d64, q64, cu, t, c, 0.1, max_q_len=4, max_context_len=4)
    pool.destroy()
    d64.destroy()


@pytest.mark.parametrize("bs", [16, 32])
def test_prefill_rescales_on_every_key_tile(bs):
    """Keys aligned with the queries and growing along the sequence push each
    row's maximum up by more than the lazy-rescale threshold on nearly every
    key tile, so O in tensor memory is rescaled again and again (and the
    product that feeds it must have finished first)."""
    hkv, hq, ctx, ql = 2, 8, 900, 700
    nblk = -(-ctx // bs)
    rng = np.random.default_rng(7)
    tables = rng.permutation(nblk + 3)[:nblk].astype(np.int32).reshape(1, nblk)
    pool = pagedkv.KVPool(nblk + 3, bs, hkv, 128, "bf16")
    poison(pool)
    opool = oracle.Pool(nblk + 3, bs, hkv, 128, "bf16")
    g = torch.Generator().manual_seed(8)
    direction = torch.randn(hkv, 128, generator=g)
    direction = direction / direction.norm(dim=1, keepdim=True)
    growth = torch.arange(ctx, dtype=torch.float32).view(ctx, 1, 1) * 0.02
    k = (growth * direction.view(1, hkv, 128) + 0.1 * torch.randn(ctx, hkv, 128, generator=g)).bfloat16()
    v = torch.randn(ctx, hkv, 128, generator=g).bfloat16()
    pos = np.arange(ctx)
    slots = tables[0, pos // bs].astype(np.int64) * bs + pos % bs
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda())
    opool.write(k, v, slots)
    q = (direction.repeat_interleave(hq // hkv, dim=0).view(1, hq, 128) * 3
         + 0.1 * torch.randn(ql, hq, 128, generator=g)).bfloat16()
    cu = np.array([0, ql], np.int32)
    lens = np.array([ctx], np.int32)
    out = _run(pool, q, cu, tables, lens, 1.0)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 1.0)
    _check(out, ref, f"rescale bs={bs}")
    pool.destroy()


@pytest.mark.parametrize("scale", [-0.09, 0.0])
def test_prefill_negative_and_zero_scale(scale):
    """A negative softmax scale favours the keys least aligned with the
    query; scale 0 weighs every attended key alike (masked keys still out)."""
    pool, opool, q, cu, tables, lens = _build([77, 300], [20, 150], 8, 2, seed=17)
    out = _run(pool, q, cu, tables, lens, scale, 100)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, scale, 100)
    _check(out, ref, f"scale={scale}")
    pool.destroy()


def test_prefill_query_rows_of_any_magnitude():
    """Rows of q scaled by 2^-30 .. 2^30 (and an all-zero row): scores up to
    ~2^32 in log2 units, where the exponent of the maximum key must still
    come out exact (the row is then its maximum key's value)."""
    pool, opool, q, cu, tables, lens = _build([300], [64], 8, 2, seed=21)
    f = torch.tensor([2.0 ** e for e in range(-30, 31, 4)] + [0.0])
    rows = q.float().view(64 * 8, 128)
    rows[: f.numel()] *= f.view(-1, 1)
    q = rows.view(64, 8, 128).bfloat16()
    out = _run(pool, q, cu, tables, lens, 0.05)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 0.05)
    _check(out, ref, "query magnitudes")
    pool.destroy()


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("profile", ["mixed", "tiny", "huge", "zero_first"])
def test_prefill_values_of_any_magnitude(profile, bs):
    """V rows scaled per 128-key tile (mixed: 2^-12 .. 2^8 in one sequence,
    the largest arriving late), all by 2^-40 or 2^60, or zero over the first
    key tile and N(0,1) after it: the output matches the oracle in units of
    its own largest magnitude (relative L2 and max |err| / max |ref| within
    the bar)."""
    hkv, hq, ctx, ql = 2, 8, 700, 300
    nblk = -(-ctx // bs)
    rng = np.random.default_rng(31)
    tables = rng.permutation(nblk + 3)[:nblk].astype(np.int32).reshape(1, nblk)
    pool = pagedkv.KVPool(nblk + 3, bs, hkv, 128, "bf16")
    poison(pool)
    opool = oracle.Pool(nblk + 3, bs, hkv, 128, "bf16")
    g = torch.Generator().manual_seed(32)
    k = torch.randn(ctx, hkv, 128, generator=g).bfloat16()
    powers = {"mixed": [-12, 8, 0, -4, 3, 6], "tiny": [-40] * 6, "huge": [60] * 6,
              "zero_first": [None, 0, 0, 0, 0, 0]}[profile]
    tile_scale = torch.tensor([0.0 if powers[i // 128] is None else 2.0 ** powers[i // 128]
                               for i in range(ctx)]).view(ctx, 1, 1)
    v = (torch.randn(ctx, hkv, 128, generator=g) * tile_scale).bfloat16()
    pos = np.arange(ctx)
    slots = tables[0, pos // bs].astype(np.int64) * bs + pos % bs
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda())
    opool.write(k, v, slots)
    q = torch.randn(ql, hq, 128, generator=g).bfloat16()
    cu = np.array([0, ql], np.int32)
    lens = np.array([ctx], np.int32)
    out = _run(pool, q, cu, tables, lens, 128 ** -0.5)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5)
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    unit = float(np.abs(ref).max())
    max_abs, rel = errors(got / unit, ref / unit)
    print(f"PARITY prefill V {profile} bs={bs} max_abs/unit={max_abs:.3e} rel_l2={rel:.3e}")
    assert max_abs <= MAX_ABS and rel <= REL_L2, (profile, max_abs, rel)
    pool.destroy()


@pytest.mark.parametrize("hq,hkv", [(16, 1), (48, 2), (128, 1)])
def test_prefill_large_groups(hq, hkv):
    """Groups of 16, 24 (padded to 32) and 128 query heads per KV head: a
    query tile then holds 8, 4 or 1 tokens."""
    pool, opool, q, cu, tables, lens = _build([150, 300], [150, 77], hq, hkv, seed=hq + hkv)
    out = _run(pool, q, cu, tables, lens, 128 ** -0.5, 200)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5, 200)
    _check(out, ref, f"group hq={hq} hkv={hkv}")
    pool.destroy()
