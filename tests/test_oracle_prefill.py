"""Pins of the oracle's paged prefill (extend) attention.

* With an identity block table over a contiguous pool, every sequence's
  result equals dense causal attention computed by PyTorch's
  scaled_dot_product_attention in fp64 on the CPU (a library routine, with
  an explicit boolean mask: query i at position pos sees keys [lo, pos]).
* Shuffling the physical blocks and relabelling the table changes nothing.
* The last new token of a sequence gets exactly the decode result.
* A window of 1 returns the token's own V; a window covering the whole
  context equals no window.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _case(lens, qlens, hq, hkv, d, bs=16, seed=0, shuffle=False):
    g = torch.Generator().manual_seed(seed)
    lens = np.asarray(lens, np.int32)
    qlens = np.asarray(qlens, np.int32)
    nblk = [-(-int(c) // bs) for c in lens]
    nb = sum(nblk) + 3
    ids = np.random.default_rng(seed).permutation(nb) if shuffle else np.arange(nb)
    tables = np.full((len(lens), max(nblk)), -1, np.int32)
    at = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = ids[at:at + n]
        at += n
    K = [torch.randn(int(c), hkv, d, generator=g, dtype=torch.float64).to(torch.bfloat16) for c in lens]
    V = [torch.randn(int(c), hkv, d, generator=g, dtype=torch.float64).to(torch.bfloat16) for c in lens]
    T = int(qlens.sum())
    q = torch.randn(T, hq, d, generator=g, dtype=torch.float64).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    pool = oracle.Pool(nb, bs, hkv, d, "bf16")
    for b, c in enumerate(lens):
        pos = np.arange(int(c))
        slots = tables[b, pos // bs].astype(np.int64) * bs + pos % bs
        pool.write(K[b], V[b], slots)
    return pool, q, cu, tables, lens, K, V


def _dense(q, cu, lens, K, V, scale, window, hq, hkv):
    outs = []
    for b, c in enumerate(lens):
        qb = q[cu[b]:cu[b + 1]].double().transpose(0, 1)              # [Hq, n, D]
        kb = K[b].double().repeat_interleave(hq // hkv, dim=1).transpose(0, 1)
        vb = V[b].double().repeat_interleave(hq // hkv, dim=1).transpose(0, 1)
        n = qb.shape[1]
        pos = torch.arange(c - n, c)[:, None]
        key = torch.arange(c)[None, :]
        mask = key <= pos
        if window > 0:
            mask &= key >= pos + 1 - window
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=scale)
        outs.append(o.transpose(0, 1))
    return torch.cat(outs).numpy()


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("window", [0, 1, 7, 40])
def test_identity_table_is_dense_causal_attention(bs, window):
    lens, qlens = [5, 33, 64, 100], [5, 1, 20, 37]
    pool, q, cu, tables, lens, K, V = _case(lens, qlens, 8, 2, 64, bs=bs, seed=bs + window)
    got = pool.prefill(q, cu, tables, lens, 0.125, window)
    want = _dense(q, cu, lens, K, V, 0.125, window, 8, 2)
    assert np.abs(got - want).max() < 1e-6


def test_block_shuffle_changes_nothing():
    args = ([40, 77], [40, 13], 4, 4, 64)
    a = _case(*args, seed=3)
    b = _case(*args, seed=3, shuffle=True)
    ra = a[0].prefill(a[1], a[2], a[3], a[4], 0.2)
    rb = b[0].prefill(b[1], b[2], b[3], b[4], 0.2)
    assert np.array_equal(ra, rb)


def test_last_new_token_is_the_decode_result():
    pool, q, cu, tables, lens, K, V = _case([30, 50], [7, 50], 8, 2, 64, seed=5)
    pre = pool.prefill(q, cu, tables, lens, 0.1, 0)
    last = q[torch.from_numpy(cu[1:] - 1).long()]
    dec = pool.decode(last, tables, lens, 0.1, 0)
    assert np.array_equal(pre[cu[1:] - 1], dec)


def test_window_edges():
    pool, q, cu, tables, lens, K, V = _case([20, 45], [20, 10], 2, 1, 64, seed=9)
    one = pool.prefill(q, cu, tables, lens, 0.3, 1)
    for b, c in enumerate(lens):
        n = cu[b + 1] - cu[b]
        own = V[b][c - n:c, 0].float().numpy()            # each token's own V (Hkv = 1)
        for j in range(2):
            assert np.allclose(one[cu[b]:cu[b + 1], j], own, atol=0, rtol=0)
    wide = pool.prefill(q, cu, tables, lens, 0.3, 1000)
    none = pool.prefill(q, cu, tables, lens, 0.3, 0)
    assert np.array_equal(wide, none)
