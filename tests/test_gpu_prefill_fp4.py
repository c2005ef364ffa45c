"""GPU parity of paged prefill (extend) attention over FP4 pools (E2M1 codes,
an E4M3 scale per 16 elements, per-KV-head scales), on the tensor cores,
against the fp64 oracle on the same codes and scales.

Tolerance: the bf16 bar, as for the FP4 decode: every key and value is
dequantised exactly into f16 (an E2M1 value times an E4M3 scale has at most
5 significant bits), each query row enters as f16 after a power-of-two
scaling that keeps its bf16 values exact, each weight as one f16 (relative
rounding <= 2^-11), accumulation in fp32.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv

from _parity import FP4_MAX_ABS, FP4_REL_L2, errors, poison

pytestmark = pytest.mark.gpu



def _build(ctx_lens, q_lens, hq, hkv, bs=16, seed=0, extra_blocks=5, kv=None):
    """FP4 pools (GPU poisoned, oracle) holding every context token with
    per-KV-head scales amax / (6 x 448); queries of the last q_len positions;
    shuffled tables.  `kv(c, g)` may supply a sequence's K and V."""
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
    data = []
    for c in ctx_lens:
        if kv is not None:
            data.append(kv(int(c), g))
        else:
            data.append((torch.randn(int(c), hkv, 128, generator=g).to(torch.bfloat16),
                         torch.randn(int(c), hkv, 128, generator=g).to(torch.bfloat16)))
    kmax = torch.stack([k.float().abs().amax(dim=(0, 2)) for k, _ in data if k.shape[0]]).amax(0)
    vmax = torch.stack([v.float().abs().amax(dim=(0, 2)) for _, v in data if v.shape[0]]).amax(0)
    ks = (kmax / 2688).numpy().astype(np.float32)
    vs = (vmax / 2688).numpy().astype(np.float32)
    pool = pagedkv.KVPool(nb, bs, hkv, 128, "fp4")
    poison(pool)
    pool.set_scales(torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())
    opool = oracle.Pool(nb, bs, hkv, 128, "fp4")
    opool.set_scales(ks, vs)
    for b, (k, v) in enumerate(data):
        c = k.shape[0]
        if c == 0:
            continue
        pos = np.arange(c)
        slots = tables[b, pos // bs].astype(np.int64) * bs + pos % bs
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
    print(f"PARITY prefill fp4 {label} max_abs={max_abs:.3e} rel_l2={rel:.3e}")
    assert max_abs <= FP4_MAX_ABS and rel <= FP4_REL_L2, (label, max_abs, rel)


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (3, 1), (12, 2)])
def test_prefill_fp4_matches_oracle(hq, hkv, bs):
    # ragged contexts: sequence ends inside a 16-token record, on its edge,
    # and inside a 32-token block; cached prefixes; q_len 1 and 0
    ctx = [1, 16, 17, 63, 64, 65, 200, 300, 129, 90]
    ql = [1, 16, 5, 63, 1, 30, 200, 77, 0, 90]
    pool, opool, q, cu, tables, lens = _build(ctx, ql, hq, hkv, bs=bs, seed=hq * 10 + hkv + bs)
    out = _run(pool, q, cu, tables, lens, 128 ** -0.5)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5)
    _check(out, ref, f"hq={hq} hkv={hkv} bs={bs}")
    pool.destroy()


@pytest.mark.parametrize("window", [1, 7, 100, 5000])
def test_prefill_fp4_sliding_window(window):
    ctx = [50, 300, 700]
    ql = [50, 120, 300]
    pool, opool, q, cu, tables, lens = _build(ctx, ql, 16, 4, seed=window)
    for b, c in enumerate(lens):                  # blocks before every window: unmapped
        lo = max(0, int(c) - int(ql[b]) + 1 - window)
        tables[b, : lo // 16] = -1
    out = _run(pool, q, cu, tables, lens, 0.1, window)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 0.1, window)
    _check(out, ref, f"window={window}")
    pool.destroy()


def test_prefill_fp4_long_prompt_many_tiles():
    pool, opool, q, cu, tables, lens = _build([2048, 1500], [300, 1500], 8, 2, seed=3)
    out = _run(pool, q, cu, tables, lens, 128 ** -0.5)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5)
    _check(out, ref, "long")
    pool.destroy()


@pytest.mark.parametrize("bs", [16, 32])
def test_prefill_fp4_rescales_often(bs):
    """Keys aligned with the queries and growing along the sequence raise each
    row's maximum on nearly every key tile, past the lazy-rescale threshold,
    so O in tensor memory is rescaled again and again."""
    hkv, hq, ctx, ql = 2, 8, 900, 700
    g0 = torch.Generator().manual_seed(8)
    direction = torch.randn(hkv, 128, generator=g0)
    direction = direction / direction.norm(dim=1, keepdim=True)

    def kv(c, g):
        growth = torch.arange(c, dtype=torch.float32).view(c, 1, 1) * 0.02
        k = (growth * direction.view(1, hkv, 128) + 0.1 * torch.randn(c, hkv, 128, generator=g)).bfloat16()
        return k, torch.randn(c, hkv, 128, generator=g).bfloat16()

    pool, opool, _, cu, tables, lens = _build([ctx], [ql], hq, hkv, bs=bs, seed=9, kv=kv)
    g = torch.Generator().manual_seed(10)
    q = (direction.repeat_interleave(hq // hkv, dim=0).view(1, hq, 128) * 3
         + 0.1 * torch.randn(ql, hq, 128, generator=g)).bfloat16()
    out = _run(pool, q, cu, tables, lens, 1.0)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 1.0)
    _check(out, ref, f"rescale bs={bs}")
    pool.destroy()


def test_prefill_fp4_query_rows_of_any_magnitude():
    """Each query row takes its own power of two: rows scaled by 2^-30 .. 2^30
    (and an all-zero row) give the oracle's result for those rows."""
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


def test_prefill_fp4_last_token_matches_decode():
    pool, opool, q, cu, tables, lens = _build([77, 300], [20, 33], 8, 2, seed=11)
    out = _run(pool, q, cu, tables, lens, 0.09)
    last = q[torch.from_numpy(cu[1:] - 1).long()]
    dec = pagedkv.paged_decode_attention(pool, last.cuda(), torch.from_numpy(tables).cuda(),
                                         torch.from_numpy(lens).cuda(), 0.09,
                                         max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    got = out.cpu().numpy()[cu[1:] - 1]
    max_abs, _ = errors(got, dec.cpu().numpy())
    assert max_abs <= FP4_MAX_ABS
    pool.destroy()


def test_prefill_fp4_bad_block():
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
    assert max_abs <= FP4_MAX_ABS
    pool.destroy()


@pytest.mark.parametrize("scale", [-0.09, 0.0])
def test_prefill_fp4_negative_and_zero_scale(scale):
    pool, opool, q, cu, tables, lens = _build([77, 300], [20, 150], 8, 2, seed=17)
    out = _run(pool, q, cu, tables, lens, scale, 100)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, scale, 100)
    _check(out, ref, f"scale={scale}")
    pool.destroy()


@pytest.mark.parametrize("hq,hkv", [(32, 2), (96, 1)])
def test_prefill_fp4_large_groups(hq, hkv):
    """Groups of 16 and 96 (padded to 128) query heads per KV head."""
    pool, opool, q, cu, tables, lens = _build([150, 300], [150, 77], hq, hkv, seed=hq + hkv)
    out = _run(pool, q, cu, tables, lens, 128 ** -0.5)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.prefill(q, cu, tables, lens, 128 ** -0.5)
    _check(out, ref, f"group hq={hq} hkv={hkv}")
    pool.destroy()
