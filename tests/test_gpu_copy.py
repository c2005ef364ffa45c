"""GPU tests of paged_kv_copy_blocks (copy-on-write block copies) and of the
fork / copy-on-write / decode loop driven by the product block manager.

Block copies must be bit-exact against the oracle applying the same pairs
one after another (chains, repeated destinations and self-copies included).
The decode loop runs the product manager + CUDA path on one side and the
oracle allocator + oracle pool on the other, from the same seeded inputs.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv
from paged_kv_cache_33_gb300 import workloads as W

from _parity import assert_close, compare_pools, poison

pytestmark = pytest.mark.gpu


def _filled_pair(nb, hkv, d, dtype, seed):
    """A GPU pool and an oracle pool holding the same random contents in every slot."""
    pool = pagedkv.KVPool(nb, 16, hkv, d, dtype)
    opool = oracle.Pool(nb, 16, hkv, d, dtype)
    if dtype in ("fp8", "fp4"):
        ks = (0.5 + np.arange(hkv)).astype(np.float32) / 448.0 * 4
        vs = (0.75 + np.arange(hkv)).astype(np.float32) / 448.0 * 4
        pool.set_scales(torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())
        opool.set_scales(ks, vs)
    g = torch.Generator().manual_seed(seed)
    T = nb * 16
    k = torch.randn(T, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(T, hkv, d, generator=g).to(torch.bfloat16)
    slots = torch.arange(T, dtype=torch.int64)
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), slots.cuda())
    opool.write(k, v, slots.numpy())
    return pool, opool


@pytest.mark.parametrize("dtype,hkv,d", [("bf16", 8, 128), ("bf16", 2, 64), ("fp8", 4, 128),
                                         ("fp4", 4, 128)])
def test_copies_match_in_order_application(dtype, hkv, d):
    nb = 48
    pool, opool = _filled_pair(nb, hkv, d, dtype, seed=5)
    rng = np.random.default_rng(1)
    pairs = rng.integers(0, nb, size=(300, 2)).astype(np.int32)
    pairs[::17, 1] = pairs[::17, 0]                          # self-copies
    pairs[5:40:3, 0] = pairs[4:39:3, 1]                      # chains: read what was just written
    pagedkv.paged_kv_copy_blocks(pool, pairs)
    opool.copy_blocks(pairs)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    compare_pools(pool, opool, np.arange(nb * 16))
    pool.destroy()


def test_many_disjoint_copies_span_several_launches():
    nb = 10_000
    pool, opool = _filled_pair(nb, 1, 64, "bf16", seed=6)
    perm = np.random.default_rng(2).permutation(nb).astype(np.int32)
    pairs = np.stack([perm[:4500], perm[4500:9000]], axis=1)   # > 2 waves of 2048
    pagedkv.paged_kv_copy_blocks(pool, pairs)
    opool.copy_blocks(pairs)
    torch.cuda.synchronize()
    compare_pools(pool, opool, np.arange(nb * 16))
    pool.destroy()


def test_bad_ids_are_rejected_before_any_copy():
    pool, opool = _filled_pair(8, 2, 64, "bf16", seed=7)
    before = pool.view().clone()
    for bad in ([[0, 8]], [[-1, 2]], [[1, 2], [3, 9]]):
        with pytest.raises(pagedkv.KVError):
            pagedkv.paged_kv_copy_blocks(pool, bad)
    torch.cuda.synchronize()
    assert torch.equal(pool.view(), before)
    pagedkv.paged_kv_copy_blocks(pool, np.zeros((0, 2), np.int32))   # nothing to do
    pool.destroy()


def test_fork_copy_on_write_decode_loop():
    """Parallel sampling: one prompt forked into three sequences that then
    decode different tokens.  Every step: append one token per sequence in
    the block manager, run its copy-on-write copies, write the new K/V and
    attend; the oracle side mirrors it with its own allocator and pool."""
    nb, hkv, hq, d, bs = 40, 2, 8, 128, 16
    scale = d ** -0.5
    pm, om = pagedkv.BlockManager(nb, bs), oracle.Allocator(nb, bs)
    pool = pagedkv.KVPool(nb, bs, hkv, d, "bf16")
    poison(pool)
    opool = oracle.Pool(nb, bs, hkv, d, "bf16")
    g = torch.Generator().manual_seed(21)

    def kv(n):
        return (torch.randn(n, hkv, d, generator=g).to(torch.bfloat16),
                torch.randn(n, hkv, d, generator=g).to(torch.bfloat16))

    prompt = 37                                    # last block partly filled: forks share it
    assert pm.admit(0, num_tokens=prompt)[0] == 0 and om.admit(0, num_tokens=prompt)[0] == 0
    k, v = kv(prompt)
    slots = pm.slot_mapping(0, 0, prompt)
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda())
    opool.write(k, v, slots)
    for child in (1, 2):
        assert pm.fork(0, child) == 0 and om.fork(0, child) == 0
    seqs = [0, 1, 2]
    total_copies = 0
    w = W.make("tiny")                             # bf16 tolerances
    for step in range(24):
        for s in seqs:
            assert pm.append(s, n=1) == 0 and om.append(s, n=1) == 0
        pc, oc = pm.copies(), om.copies()
        assert pc == oc
        total_copies += len(pc)
        pagedkv.paged_kv_copy_blocks(pool, pc)
        if oc:
            opool.copy_blocks(oc)
        mbs = max(len(pm.table(s)) for s in seqs)
        tables, lens, new_slots = pm.decode_inputs(seqs, mbs)
        ot = np.full_like(tables, -1)
        for i, s in enumerate(seqs):
            t = om.table(s)
            ot[i, :len(t)] = t
        assert np.array_equal(tables, ot)
        k, v = kv(len(seqs))
        q = torch.randn(len(seqs), hq, d, generator=g).to(torch.bfloat16)
        out = pagedkv.paged_decode_step(pool, k.cuda(), v.cuda(),
                                        torch.from_numpy(new_slots).cuda(), q.cuda(),
                                        torch.from_numpy(tables).cuda(),
                                        torch.from_numpy(lens).cuda(), scale,
                                        max_context_len=int(lens.max()))
        opool.write(k, v, new_slots)
        ref = opool.decode(q, tables, lens, scale, 0)
        torch.cuda.synchronize()
        assert pool.check_status() == pagedkv.KV_OK
        assert_close(w, out.cpu().numpy(), ref, f"step {step}")
    assert total_copies == 2                       # the first writes of two of the three sharers
    live = np.concatenate([pm.slot_mapping(s, 0, pm.num_tokens(s)) for s in seqs])
    compare_pools(pool, opool, np.unique(live))
    pool.destroy()
