"""GPU parity: the sm_103a kernels through the C ABI against the fp64 oracle.

The KV write must be bit-exact (bf16 bit copy, FP8 codes, FP4 codes and block
scales); attention must be within max |err| <= 2e-3 and relative L2 <= 1e-3
for bf16 and FP4 KV (against the oracle on the stored codes), max |err| <=
3e-2 for FP8 KV.  The pool is poisoned with NaN codes before any write, so a
read of a slot that was never written would surface as a non-finite output.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv
from paged_kv_cache_33_gb300 import workloads as W

from _parity import (assert_close, compare_pools, decode_gpu, fill_both, make_gpu_pool, poison,
                     make_oracle_pool, run_parity, written_slots)

pytestmark = pytest.mark.gpu


def _workload(name, size, block_size=16):
    return W.make(name, size, make_allocator=oracle.Allocator if name in ("fp8", "fp4") else None,
                  block_size=block_size)


@pytest.mark.parametrize("block_size", [16, 32])
def test_tiny_workload_exact_path(block_size):
    w = W.make("tiny", block_size=block_size)
    r = run_parity(w)
    assert r["max_abs"] < 1e-4


@pytest.mark.parametrize("block_size", [16, 32])
@pytest.mark.parametrize("name", ["8b", "70b", "sw", "fp8", "fp4", "long"])
@pytest.mark.parametrize("part_blocks", [None, 4, 12])
def test_small_workloads(name, part_blocks, block_size):
    # several partitions per sequence (forced small partitions exercise the reduce)
    run_parity(_workload(name, "small", block_size), part_blocks=part_blocks)


@pytest.mark.parametrize("block_size", [16, 32])
@pytest.mark.parametrize("name", ["8b", "70b", "sw", "fp8", "fp4", "long"])
def test_full_workloads_sampled(name, block_size):
    """Full-size workloads in the bench's launch configuration; the oracle
    computes a sample of sequences (the longest, the shortest, and random)."""
    w = _workload(name, "full", block_size)
    lens = w.context_lens
    rng = np.random.default_rng(5)
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    pick |= set(int(x) for x in rng.choice(w.batch, 4, replace=False))
    run_parity(w, seqs=sorted(pick), device_fill_rest=True)


def _custom(lens, hq=8, hkv=2, d=128, window=0, dtype="bf16", extra_blocks=7, seed=0, bs=16):
    """A workload with chosen context lengths and shuffled physical blocks."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nblk = [max(1, -(-int(c) // bs)) for c in lens]
    nb = sum(nblk) + extra_blocks
    perm = rng.permutation(nb).astype(np.int32)
    mbs = max(nblk)
    tables = np.full((len(lens), mbs), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[off:off + n]
        off += n
    w = W.Workload("custom", "small", len(lens), hq, hkv, d, bs, nb, window, dtype,
                   1.0 / np.sqrt(d), lens, tables, np.where(lens > 0, lens - 1, -1).astype(np.int64),
                   data_seed=seed + 77)
    if dtype == "fp8":
        w.k_scale = np.linspace(0.009, 0.013, hkv).astype(np.float32)
        w.v_scale = np.linspace(0.011, 0.015, hkv).astype(np.float32)
    if dtype == "fp4":
        w.k_scale = np.linspace(0.0015, 0.0022, hkv).astype(np.float32)
        w.v_scale = np.linspace(0.0019, 0.0025, hkv).astype(np.float32)
    return w


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (4, 2, 128), (16, 4, 128), (16, 2, 128),
                                      (2, 1, 64), (8, 1, 64), (7, 7, 64), (24, 3, 128),
                                      (32, 2, 128), (24, 2, 128), (18, 2, 64), (64, 1, 128)])
def test_head_grouping_and_head_dim(hq, hkv, d, bs):
    lens = [1, 15, 16, 17, 31, 32, 33, 47, 48, 49, 200, 513]
    run_parity(_custom(lens, hq, hkv, d, seed=hq + hkv + d, bs=bs))


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp4"])
@pytest.mark.parametrize("window", [1, 15, 16, 17, 31, 33, 100, 512, 10_000])
def test_sliding_window_edges(window, dtype, bs):
    lens = [1, 16, 17, 32, 33, 100, 101, 600, 1111]
    w = _custom(lens, 16, 4, 128, window=window, dtype=dtype, seed=window, bs=bs)
    # blocks wholly before the window are unmapped: the kernel must not read them
    for b, c in enumerate(w.context_lens):
        lo = max(0, int(c) - window)
        w.block_tables[b, : lo // bs] = -1
    run_parity(w, part_blocks=4)


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("dtype", ["fp8", "fp4"])
def test_quantised_head_groups_and_partitions(bs, dtype):
    # 16-token blocks: FP8 units hold two blocks and FP4 units three, so block
    # counts leave partial units; 32-token blocks: one block, two sub-tiles
    lens = [1, 5, 16, 17, 31, 32, 33, 47, 48, 49, 300, 2000]
    for hq, hkv in [(8, 8), (16, 2), (32, 8), (3, 1), (24, 3)]:
        run_parity(_custom(lens, hq, hkv, 128, dtype=dtype, seed=hq, bs=bs), part_blocks=8)


def test_empty_and_single_token_contexts():
    w = _custom([0, 1, 0, 2, 16], 8, 2, 128, seed=3)
    pool = make_gpu_pool(w)
    opool = make_oracle_pool(w)
    fill_both(w, pool, opool)
    q = w.query()
    out = decode_gpu(w, pool, q).cpu().numpy()
    assert pool.check_status() == pagedkv.KV_OK
    assert not out[0].any() and not out[2].any()
    ref = opool.decode(q, w.block_tables, w.context_lens, w.scale)
    assert_close(w, out, ref)


def test_block_permutation_gives_bit_identical_output():
    lens = [40, 300, 77]
    outs = []
    for seed in (1, 2):
        w = _custom(lens, 8, 2, 128, seed=seed, extra_blocks=11)
        w.data_seed = 5   # same content, different physical placement
        pool = make_gpu_pool(w)
        fill_both(w, pool, None)
        outs.append(decode_gpu(w, pool, w.query()).cpu())
    assert torch.equal(outs[0], outs[1])


def test_sequences_sharing_blocks_agree():
    w = _custom([300, 300, 300], 8, 2, 128, seed=4)
    w.block_tables[1] = w.block_tables[0]
    w.block_tables[2] = w.block_tables[0]
    w.new_pos[:] = -1
    w.new_pos[0] = 299
    pool = make_gpu_pool(w)
    fill_both(w, pool, None, seqs=[0])
    q = w.query()
    q[1] = q[0]
    q[2] = q[0]
    out = decode_gpu(w, pool, q).cpu()
    assert torch.equal(out[0], out[1]) and torch.equal(out[0], out[2])


def test_non_default_stream():
    w = _custom([50, 400], 8, 2, 128, seed=9)
    pool = make_gpu_pool(w)
    opool = make_oracle_pool(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fill_both(w, pool, opool)
        q = w.query()
        out = decode_gpu(w, pool, q)
    s.synchronize()
    ref = opool.decode(q, w.block_tables, w.context_lens, w.scale)
    assert_close(w, out.cpu().numpy(), ref)


# ----------------------------------------------------------------- KV write --

@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("fp8", 128), ("fp4", 128)])
def test_write_bit_exact_with_padding_and_repeats(dtype, d, bs):
    torch.manual_seed(0)
    nb, hkv, T = 40, 4, 300
    pool = pagedkv.KVPool(nb, bs, hkv, d, dtype)
    opool = oracle.Pool(nb, bs, hkv, d, dtype)
    if dtype in ("fp8", "fp4"):
        ks = torch.tensor([0.01, 0.02, 0.003, 1.0])
        vs = torch.tensor([0.05, 0.001, 0.02, 0.5])
        pool.set_scales(ks.cuda(), vs.cuda())
        opool.set_scales(ks.numpy(), vs.numpy())
    pool.view().zero_()
    k = (torch.randn(T, hkv, d) * 4).bfloat16()
    v = torch.randn(T, hkv, d).bfloat16()
    k[0, 0, :4] = torch.tensor([1e6, -1e6, 1e-9, -0.0])    # saturation, underflow, signed zero
    slots = torch.from_numpy(np.random.default_rng(1).permutation(nb * bs)[:T].astype(np.int64))
    slots[::7] = -1
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), slots.cuda())
    opool.write(k, v, slots.numpy())
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    s = slots.numpy()
    compare_pools(pool, opool, s[s >= 0])
    # a padded token's slot stays untouched (zero)
    skipped = np.setdiff1d(np.arange(nb * bs), s[s >= 0])
    vv = pool.rows()[torch.from_numpy(skipped // bs).cuda(), :, :, torch.from_numpy(skipped % bs).cuda()]
    raw = vv.view(torch.int16) if dtype == "bf16" else vv
    assert int((raw != 0).sum()) == 0


def test_fp4_write_special_values_and_one_token_calls():
    """FP4: NaN, infinities, zero and tiny rows, and tokens written one call
    at a time at every offset (the V bytes pair two tokens, so each call
    merges its nibble next to the other token's), bit-exact against the oracle."""
    torch.manual_seed(3)
    nb, hkv, bs = 12, 2, 16
    pool = pagedkv.KVPool(nb, bs, hkv, 128, "fp4")
    poison(pool)
    opool = oracle.Pool(nb, bs, hkv, 128, "fp4")
    ks, vs = torch.tensor([0.004, 0.9]), torch.tensor([0.002, 0.03])
    pool.set_scales(ks.cuda(), vs.cuda())
    opool.set_scales(ks.numpy(), vs.numpy())
    T = nb * bs
    k = (torch.randn(T, hkv, 128) * 3).bfloat16()
    v = torch.randn(T, hkv, 128).bfloat16()
    k[0, 0, :5] = torch.tensor([float("nan"), float("inf"), -float("inf"), 0.0, -0.0])
    v[1, 1, 16:32] = 0.0                                     # an all-zero group
    v[2, 0, 32:48] = 1e-30                                   # a group whose scale underflows
    k[3, 1, :] = 1e5                                         # saturated block scales
    perm = np.random.default_rng(4).permutation(T)
    # one call per token, in shuffled order (partners land before or after)
    for t in perm[: T // 2]:
        s1 = torch.tensor([int(t)], dtype=torch.int64)
        pagedkv.paged_kv_write(pool, k[t:t + 1].cuda(), v[t:t + 1].cuda(), s1.cuda())
        opool.write(k[t:t + 1], v[t:t + 1], s1.numpy())
    # the rest in one call
    rest = torch.from_numpy(perm[T // 2:].astype(np.int64))
    pagedkv.paged_kv_write(pool, k[rest].cuda(), v[rest].cuda(), rest.cuda())
    opool.write(k[rest], v[rest], rest.numpy())
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    compare_pools(pool, opool, np.arange(T))


def test_write_reports_a_slot_outside_the_pool():
    pool = pagedkv.KVPool(4, 16, 2, 128)
    k = torch.randn(3, 2, 128, device="cuda").bfloat16()
    slots = torch.tensor([0, 64, 5], device="cuda")
    pagedkv.paged_kv_write(pool, k, k, slots)
    assert pool.check_status() == 7              # KV_ERR_BAD_SLOT
    assert pool.check_status() == pagedkv.KV_OK   # cleared by the read
    v = pool.view()
    assert torch.equal(v[0, :, 0, 0], k[0])
    assert torch.equal(v[0, :, 0, 5], k[2])


def test_write_of_zero_tokens_is_a_no_op():
    pool = pagedkv.KVPool(4, 16, 2, 128)
    e = torch.empty(0, 2, 128, device="cuda", dtype=torch.bfloat16)
    pagedkv.paged_kv_write(pool, e, e, torch.empty(0, dtype=torch.int64, device="cuda"))
    assert pool.check_status() == pagedkv.KV_OK


# ------------------------------------------------------------ error reporting --

def test_bad_block_id_is_reported_and_contained():
    w = _custom([100, 200, 300], 8, 2, 128, seed=12)
    pool = make_gpu_pool(w)
    opool = make_oracle_pool(w)
    fill_both(w, pool, opool)
    q = w.query()
    tables = w.block_tables.copy()
    tables[1, 3] = w.num_blocks + 5       # outside the pool
    out = decode_gpu(w, pool, q, tables=tables).cpu().numpy()
    assert pool.check_status() == 5
    ref = opool.decode(q, w.block_tables, w.context_lens, w.scale, seqs=[0, 2])
    assert_close(w, out[[0, 2]], ref[[0, 2]])
    assert np.isfinite(out[1]).all()


def test_context_above_the_bound_is_reported():
    w = _custom([100, 200], 8, 2, 128, seed=13)
    pool = make_gpu_pool(w)
    fill_both(w, pool, None)
    out = decode_gpu(w, pool, w.query(), max_context_len=150).cpu().numpy()
    assert pool.check_status() == 8
    assert not out[1].any()


def test_host_argument_checks():
    pool = pagedkv.KVPool(8, 16, 2, 128)
    q = torch.zeros(2, 6, 128, device="cuda", dtype=torch.bfloat16)   # 6 % 2 == 0, g = 3
    t = torch.zeros(2, 4, device="cuda", dtype=torch.int32)
    c = torch.ones(2, device="cuda", dtype=torch.int32)
    pagedkv.paged_decode_attention(pool, q, t, c, 0.1, max_context_len=64)
    with pytest.raises(pagedkv.KVError) as e:
        pagedkv.paged_decode_attention(pool, q, t, c, 0.1, max_context_len=65)
    assert e.value.status == 1
    with pytest.raises(pagedkv.KVError) as e:
        pagedkv.paged_decode_attention(pool, torch.zeros(2, 5, 128, device="cuda",
                                                         dtype=torch.bfloat16), t, c, 0.1,
                                       max_context_len=64)
    assert e.value.status == 1
    with pytest.raises(pagedkv.KVError) as e:                          # group 65 > 64
        pagedkv.paged_decode_attention(pool, torch.zeros(2, 130, 128, device="cuda",
                                                         dtype=torch.bfloat16), t, c, 0.1,
                                       max_context_len=64)
    assert e.value.status == 4
    # an output that is not 16-byte aligned (the reduce stores float4) is refused
    unaligned = torch.empty(2 * 6 * 128 + 1, device="cuda")[1:].view(2, 6, 128)
    with pytest.raises(pagedkv.KVError) as e:
        pagedkv.paged_decode_attention(pool, q, t, c, 0.1, max_context_len=64, out=unaligned)
    assert e.value.status == 1


@pytest.mark.parametrize("dtype", ["fp8", "fp4"])
@pytest.mark.parametrize("window", [0, 40])
def test_groups_above_eight_quantised_and_windowed(dtype, window):
    # 16 query heads per KV head (two passes of 8) on the quantised pools,
    # with and without a window, and a forced small partition so pairs are cut
    w = _custom([1, 16, 17, 100, 333, 700], 32, 2, 128, seed=5, bs=16, dtype=dtype, window=window)
    run_parity(w, part_blocks=4)
