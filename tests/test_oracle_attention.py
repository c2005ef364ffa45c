"""Pins of the oracle's paged KV write and fp64 paged decode attention.

Nothing here re-types the oracle's formula.  The attention is pinned by
  * dense attention from torch's scaled_dot_product_attention (fp64, CPU) on a
    pool filled through an identity block table, with GQA, several head
    dimensions and a sliding window expressed as an explicit mask;
  * invariance under any permutation of the physical blocks (bit-identical);
  * equal results for sequences sharing prefix blocks;
  * closed forms: one token returns its V, equal keys or scale 0 give the
    mean of V, a window of one returns the newest V, a window at least the
    context length changes nothing, an empty context gives zeros;
the KV write by an identity-slot copy, padded slots, and the FP8 path by
torch's own float8_e4m3fn conversion.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

BS = 16


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def _fill_identity(pool, k, v, lens, mbs):
    """Sequence b's logical block i -> physical block b*mbs + i; write every token."""
    B = len(lens)
    tables = np.full((B, mbs), -1, dtype=np.int32)
    for b, c in enumerate(lens):
        nblk = -(-c // BS)
        tables[b, :nblk] = b * mbs + np.arange(nblk)
        slots = (b * mbs * BS + np.arange(c)).astype(np.int64)
        pool.write(k[b, :c], v[b, :c], slots)
    return tables


def _dense(q, k, v, lens, scale, window=0, fp8=None):
    """Reference via torch SDPA in fp64 on contiguous K/V (GQA by repeat)."""
    B, Hq, D = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b, c in enumerate(lens):
        if c == 0:
            continue
        kk = k[b, :c].double()
        vv = v[b, :c].double()
        if fp8 is not None:
            kk = fp8["k"][b, :c].double() * fp8["ks"].view(1, -1, 1)
            vv = fp8["v"][b, :c].double() * fp8["vs"].view(1, -1, 1)
        kk = kk.permute(1, 0, 2).repeat_interleave(g, dim=0)   # [Hq, c, D]
        vv = vv.permute(1, 0, 2).repeat_interleave(g, dim=0)
        qq = q[b].double().unsqueeze(1)                         # [Hq, 1, D]
        mask = None
        if window > 0:
            pos = torch.arange(c)
            mask = (pos >= c - window).view(1, 1, c).expand(Hq, 1, c)
        o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        out[b] = o[:, 0].numpy()
    return out


@pytest.mark.parametrize("D,Hq,Hkv,window", [(64, 2, 1, 0), (128, 32, 8, 0), (128, 64, 8, 0),
                                             (128, 32, 8, 40), (64, 4, 4, 17), (128, 8, 1, 0)])
def test_identity_table_equals_dense_sdpa(D, Hq, Hkv, window):
    torch.manual_seed(D + Hq + Hkv + window)
    lens = [1, 15, 16, 17, 33, 70, 100]
    B, mbs = len(lens), -(-max(lens) // BS)
    q = torch.randn(B, Hq, D).bfloat16()
    k = torch.randn(B, max(lens), Hkv, D).bfloat16()
    v = torch.randn(B, max(lens), Hkv, D).bfloat16()
    pool = oracle.Pool(B * mbs, BS, Hkv, D)
    tables = _fill_identity(pool, k, v, lens, mbs)
    scale = 1.0 / np.sqrt(D)
    got = pool.decode(q, tables, np.array(lens), scale, window)
    ref = _dense(q, k, v, lens, scale, window)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-6)


def test_fp8_identity_table_equals_dense_on_dequantized_codes():
    torch.manual_seed(5)
    D, Hq, Hkv = 128, 16, 4
    lens = [3, 16, 29, 64]
    B, mbs = len(lens), -(-max(lens) // BS)
    q = torch.randn(B, Hq, D).bfloat16()
    k = (3 * torch.randn(B, max(lens), Hkv, D)).bfloat16()
    v = torch.randn(B, max(lens), Hkv, D).bfloat16()
    ks = torch.tensor([0.011, 0.013, 0.02, 0.05], dtype=torch.float32)
    vs = torch.tensor([0.012, 0.009, 0.03, 0.004], dtype=torch.float32)
    pool = oracle.Pool(B * mbs, BS, Hkv, D, dtype="fp8")
    pool.set_scales(ks.numpy(), vs.numpy())
    tables = _fill_identity(pool, k, v, lens, mbs)
    # torch's own e4m3 conversion of x/scale (values beyond 448 saturate)
    kq = (k.float() / ks.view(1, 1, -1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn)
    vq = (v.float() / vs.view(1, 1, -1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn)
    arr = pool.array()
    for b, c in enumerate(lens):
        for t in range(c):
            blk, off = tables[b, t // BS], t % BS
            assert np.array_equal(arr[blk, 0, off], kq[b, t].view(torch.uint8).numpy())
            assert np.array_equal(arr[blk, 1, off], vq[b, t].view(torch.uint8).numpy())
    scale = 1.0 / np.sqrt(D)
    got = pool.decode(q, tables, np.array(lens), scale)
    ref = _dense(q, k, v, lens, scale,
                 fp8={"k": kq.double(), "v": vq.double(), "ks": ks.double(), "vs": vs.double()})
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-6)


def test_permuting_physical_blocks_is_bit_identical():
    torch.manual_seed(9)
    D, Hq, Hkv = 64, 8, 2
    lens = [7, 16, 40, 97]
    B, mbs = len(lens), -(-max(lens) // BS)
    q = torch.randn(B, Hq, D).bfloat16()
    k = torch.randn(B, max(lens), Hkv, D).bfloat16()
    v = torch.randn(B, max(lens), Hkv, D).bfloat16()
    nb = B * mbs
    outs = []
    for seed in (0, 1, 2):
        perm = np.random.default_rng(seed).permutation(nb + 5)[:nb]
        pool = oracle.Pool(nb + 5, BS, Hkv, D)
        tables = np.full((B, mbs), -1, dtype=np.int32)
        for b, c in enumerate(lens):
            nblk = -(-c // BS)
            tables[b, :nblk] = perm[b * mbs: b * mbs + nblk]
            pos = np.arange(c)
            slots = tables[b][pos // BS].astype(np.int64) * BS + pos % BS
            pool.write(k[b, :c], v[b, :c], slots)
        outs.append(pool.decode(q, tables, np.array(lens), 0.125))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_shared_prefix_blocks_give_identical_results():
    torch.manual_seed(13)
    D, Hq, Hkv = 64, 4, 2
    ctx = 53
    nblk = -(-ctx // BS)
    pool = oracle.Pool(16, BS, Hkv, D)
    k = torch.randn(ctx, Hkv, D).bfloat16()
    v = torch.randn(ctx, Hkv, D).bfloat16()
    table = np.array([9, 2, 14, 5], dtype=np.int32)
    pos = np.arange(ctx)
    pool.write(k, v, table[pos // BS].astype(np.int64) * BS + pos % BS)
    q1 = torch.randn(1, Hq, D).bfloat16()
    q = torch.cat([q1, q1, q1])
    tables = np.stack([table, table, table])
    out = pool.decode(q, tables, np.array([ctx, ctx, ctx]), 0.125)
    assert np.array_equal(out[0], out[1]) and np.array_equal(out[0], out[2])
    assert nblk == 4


def _single(D=64, Hq=2, Hkv=1, ctx=37, seed=0, k=None, v=None):
    torch.manual_seed(seed)
    q = torch.randn(1, Hq, D).bfloat16()
    if k is None:
        k = torch.randn(ctx, Hkv, D).bfloat16()
    if v is None:
        v = torch.randn(ctx, Hkv, D).bfloat16()
    mbs = -(-max(ctx, 1) // BS)
    pool = oracle.Pool(mbs + 3, BS, Hkv, D)
    table = np.full((1, mbs), -1, dtype=np.int32)
    table[0, : -(-ctx // BS)] = np.random.default_rng(seed).permutation(mbs + 3)[: -(-ctx // BS)]
    pos = np.arange(ctx)
    if ctx:
        pool.write(k, v, table[0][pos // BS].astype(np.int64) * BS + pos % BS)
    return pool, q, k, v, table


def test_single_token_returns_its_value():
    pool, q, k, v, table = _single(ctx=1)
    out = pool.decode(q, table, np.array([1]), 0.3)
    assert np.array_equal(out[0, 0], v[0, 0].float().numpy())
    assert np.array_equal(out[0, 1], v[0, 0].float().numpy())


def test_equal_keys_give_mean_of_values():
    ctx = 45
    k = torch.randn(1, 1, 64).bfloat16().expand(ctx, 1, 64).contiguous()
    pool, q, k, v, table = _single(ctx=ctx, k=k)
    out = pool.decode(q, table, np.array([ctx]), 0.125)
    mean = v[:, 0].double().mean(0).numpy()
    np.testing.assert_allclose(out[0, 0], mean, rtol=0, atol=1e-7)


def test_zero_scale_gives_mean_of_values():
    pool, q, k, v, table = _single(ctx=61, seed=4)
    out = pool.decode(q, table, np.array([61]), 0.0)
    np.testing.assert_allclose(out[0, 1], v[:, 0].double().mean(0).numpy(), rtol=0, atol=1e-7)


def test_window_of_one_returns_newest_value():
    pool, q, k, v, table = _single(ctx=50, seed=5)
    out = pool.decode(q, table, np.array([50]), 0.125, window=1)
    assert np.array_equal(out[0, 0], v[49, 0].float().numpy())


def test_window_at_least_context_is_no_window():
    pool, q, k, v, table = _single(ctx=50, seed=6)
    a = pool.decode(q, table, np.array([50]), 0.125, window=0)
    for w in (50, 51, 1000):
        assert np.array_equal(a, pool.decode(q, table, np.array([50]), 0.125, window=w))


def test_window_ignores_unmapped_blocks_before_it():
    pool, q, k, v, table = _single(ctx=80, seed=8)
    ref = pool.decode(q, table, np.array([80]), 0.125, window=20)
    t2 = table.copy()
    t2[0, :3] = -1   # blocks wholly before position 60 are not needed
    assert np.array_equal(ref, pool.decode(q, t2, np.array([80]), 0.125, window=20))
    with pytest.raises(ValueError):
        t3 = table.copy()
        t3[0, 3] = -1  # block 3 holds position 60..63, inside the window
        pool.decode(q, t3, np.array([80]), 0.125, window=20)


def test_empty_context_gives_zeros():
    pool, q, k, v, table = _single(ctx=20, seed=2)
    out = pool.decode(q, table, np.array([0]), 0.125)
    assert not out.any()


def test_subset_of_sequences_matches_full_call():
    torch.manual_seed(21)
    D, Hq, Hkv = 64, 4, 2
    lens = [9, 31, 64, 3]
    B, mbs = len(lens), 4
    q = torch.randn(B, Hq, D).bfloat16()
    k = torch.randn(B, 64, Hkv, D).bfloat16()
    v = torch.randn(B, 64, Hkv, D).bfloat16()
    pool = oracle.Pool(B * mbs, BS, Hkv, D)
    tables = _fill_identity(pool, k, v, lens, mbs)
    full = pool.decode(q, tables, np.array(lens), 0.2)
    part = pool.decode(q, tables, np.array(lens), 0.2, seqs=[2, 0])
    assert np.array_equal(full[[0, 2]], part[[0, 2]])
    assert not part[[1, 3]].any()


def test_write_identity_slots_is_a_contiguous_copy():
    torch.manual_seed(1)
    T, Hkv, D = 48, 3, 64
    k = torch.randn(T, Hkv, D).bfloat16()
    v = torch.randn(T, Hkv, D).bfloat16()
    pool = oracle.Pool(3, BS, Hkv, D)
    pool.write(k, v, np.arange(T))
    arr = pool.array()   # [NB, 2, BS, Hkv, D]
    assert np.array_equal(arr[:, 0].reshape(T, Hkv, D), _bits(k))
    assert np.array_equal(arr[:, 1].reshape(T, Hkv, D), _bits(v))


def test_write_skips_padded_slots_and_rejects_out_of_range():
    torch.manual_seed(2)
    k = torch.randn(3, 1, 64).bfloat16()
    pool = oracle.Pool(2, BS, 1, 64)
    pool.write(k, k, np.array([-1, 17, -5]))
    arr = pool.array()
    assert np.array_equal(arr[1, 0, 1, 0], _bits(k[1, 0]))
    assert arr.sum(dtype=np.int64) == 2 * int(_bits(k[1, 0]).sum(dtype=np.int64))
    with pytest.raises(ValueError):
        pool.write(k, k, np.array([0, 1, 32]))


def test_block_copy_moves_whole_blocks_in_order():
    import torch
    p = oracle.Pool(6, 16, 2, 64, "bf16")
    g = torch.Generator().manual_seed(3)
    k = torch.randn(6 * 16, 2, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(6 * 16, 2, 64, generator=g).to(torch.bfloat16)
    p.write(k, v, np.arange(6 * 16))
    before = p.array().copy()
    p.copy_blocks([(1, 4), (4, 5)])         # in order: block 5 receives block 1's rows
    after = p.array()
    assert np.array_equal(after[4], before[1]) and np.array_equal(after[5], before[1])
    for b in (0, 1, 2, 3):
        assert np.array_equal(after[b], before[b])
    with pytest.raises(ValueError):
        p.copy_blocks([(0, 6)])
    assert np.array_equal(p.array(), after)
