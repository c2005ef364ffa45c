"""The product host block manager (libpagedkv, include/kv_block_manager.h)
against the oracle allocator: both are driven with the same seeded sequences
of admits (with and without token ids, salts, extra keys), appends, forks
with copy-on-write, frees and preemptions, and must agree exactly on every
return code, cached-token count, block table, free-queue order, reference
count, block hash, hash-map entry, statistic and pending copy.  The product's
SHA-256 is also checked against Python's hashlib.  No GPU is needed.
"""

import hashlib

import numpy as np
import pytest

import oracle
from paged_kv_cache_33_gb300 import pagedkv
from paged_kv_cache_33_gb300 import workloads as W


def _state(a, live):
    tables = {r: a.table(r) for r in sorted(live)}
    blocks = [a.block(b) for b in range(a.num_blocks)]
    st = a.stats()
    return (tables, a.free_queue(), a.num_free(), blocks, a.map_entries(),
            [st[k] for k in ("queries", "hits", "evictions", "preemptions", "running")],
            {r: a.num_tokens(r) for r in sorted(live)})


def _compare(p, o, live, where):
    sp, so = _state(p, live), _state(o, live)
    names = ("tables", "free queue", "num_free", "blocks", "map", "stats", "num_tokens")
    for name, x, y in zip(names, sp, so):
        assert x == y, (where, name)


@pytest.mark.parametrize("seed,bs,nb,vocab", [(1, 4, 40, 3), (2, 16, 64, 2), (3, 1, 30, 4),
                                              (4, 8, 200, 50)])
def test_random_operations_match_the_oracle(seed, bs, nb, vocab):
    rng = np.random.default_rng(seed)
    p, o = pagedkv.BlockManager(nb, bs), oracle.Allocator(nb, bs)
    live: set[int] = set()
    next_id = 0
    counts = {"admit": 0, "oom": 0, "fork": 0, "cow": 0, "preempt": 0}
    for step in range(1200):
        op = int(rng.integers(0, 12))
        lv = sorted(live)
        if op <= 2 or not lv:
            n = int(rng.integers(0, 5 * bs + 3))
            salt = bytes(rng.integers(0, 256, int(rng.integers(0, 3)), dtype=np.uint8))
            extra = bytes(rng.integers(0, 256, int(rng.integers(0, 2)), dtype=np.uint8))
            if rng.random() < 0.85:
                toks = rng.integers(0, vocab, n).astype(np.int32)
                rp = p.admit(next_id, tokens=toks, salt=salt, extra=extra)
                ro = o.admit(next_id, tokens=toks, salt=salt, extra=extra)
            else:
                rp = p.admit(next_id, num_tokens=n)
                ro = o.admit(next_id, num_tokens=n)
            assert rp == ro, (step, rp, ro)
            if rp[0] == 0:
                live.add(next_id)
                counts["admit"] += 1
            else:
                counts["oom"] += 1
            next_id += 1
        elif op <= 4:
            parent = lv[int(rng.integers(0, len(lv)))]
            assert p.fork(parent, next_id) == o.fork(parent, next_id) == 0
            live.add(next_id)
            next_id += 1
            counts["fork"] += 1
        elif op <= 8:
            rid = lv[int(rng.integers(0, len(lv)))]
            n = int(rng.integers(0, 2 * bs + 2))
            if rng.random() < 0.9:
                toks = rng.integers(0, vocab, n).astype(np.int32)
                assert p.append(rid, tokens=toks) == o.append(rid, tokens=toks), step
            else:
                assert p.append(rid, n=n) == o.append(rid, n=n), step
            cp, co = p.copies(), o.copies()
            assert cp == co, step
            counts["cow"] += len(cp)
        elif op <= 10:
            rid = lv[int(rng.integers(0, len(lv)))]
            assert p.free(rid) == o.free(rid) == 0
            live.discard(rid)
        else:
            rp, ro = p.preempt_newest(), o.preempt_newest()
            assert rp == ro, step
            if rp[0] == 0:
                live.discard(rp[1])
                counts["preempt"] += 1
        if step % 20 == 0:
            _compare(p, o, live, step)
    _compare(p, o, live, "end")
    assert p.stats()["cow_copies"] == counts["cow"]
    if bs == 1:
        counts.pop("cow")                  # one-token blocks are never partly filled
    assert min(counts.values()) > 0, counts


def test_errors_match_the_oracle():
    p, o = pagedkv.BlockManager(4, 4), oracle.Allocator(4, 4)
    for a in (p, o):
        assert a.admit(1, num_tokens=5)[0] == 0
        assert a.admit(1, num_tokens=1)[0] == 1        # duplicate id
        assert a.admit(2, num_tokens=13)[0] == 2       # 4 blocks > 2 free
        assert a.append(9, n=1) == 1                   # unknown
        assert a.fork(9, 3) == 1 and a.fork(1, 1) == 1
        assert a.free(9) == 1
        assert a.append(1, n=-1) == 1
    assert _state(p, {1}) == _state(o, {1})
    assert p.preempt_newest() == o.preempt_newest() == (0, 1)
    assert p.preempt_newest()[0] == o.preempt_newest()[0] == 2   # nothing running


@pytest.mark.parametrize("extra_len", [0, 1, 7, 8, 9, 23, 24, 25, 31, 55, 56, 64, 100])
def test_block_hash_is_sha256_of_the_documented_bytes(extra_len):
    # parent (32 zero bytes) || token ids as int32 LE || extra || salt, padded
    # across the 55/56/64-byte boundaries of SHA-256's last block
    bs = 4
    p = pagedkv.BlockManager(8, bs)
    toks = np.array([5, -1, 70000, 2**31 - 1, 3], np.int32)
    extra = bytes(range(extra_len))
    salt = b"salt!"
    assert p.admit(7, tokens=toks, salt=salt, extra=extra)[0] == 0
    msg = bytes(32) + toks[:bs].astype("<i4").tobytes() + extra + salt
    b0 = p.table(7)[0]
    assert p.block(b0)[1] == hashlib.sha256(msg).digest()
    # block 1: chained, no salt
    assert p.append(7, tokens=np.array([8, 9, 10], np.int32)) == 0
    msg1 = hashlib.sha256(msg).digest() + np.array([3, 8, 9, 10], "<i4").tobytes() + extra
    assert p.block(p.table(7)[1])[1] == hashlib.sha256(msg1).digest()


def test_decode_inputs_and_slot_mapping():
    p = pagedkv.BlockManager(16, 4)
    assert p.admit(1, num_tokens=6)[0] == 0        # blocks 0, 1
    assert p.admit(2, num_tokens=4)[0] == 0        # block 2
    assert p.append(2, n=1) == 0                   # block 3 for position 4
    tables, lens, slots = p.decode_inputs([2, 1], 3)
    assert tables.tolist() == [[2, 3, -1], [0, 1, -1]]
    assert lens.tolist() == [5, 6]
    assert slots.tolist() == [3 * 4 + 0, 1 * 4 + 1]
    assert p.slot_mapping(1, 0, 6).tolist() == [0, 1, 2, 3, 4, 5]
    assert p.slot_mapping(2, 3, 2).tolist() == [2 * 4 + 3, 3 * 4 + 0]
    with pytest.raises(pagedkv.KVError):
        p.decode_inputs([1], 1)                    # needs 2 blocks
    with pytest.raises(pagedkv.KVError):
        p.decode_inputs([9], 3)                    # unknown
    with pytest.raises(pagedkv.KVError):
        p.slot_mapping(1, 5, 2)                    # past the end


@pytest.mark.parametrize("size", ["small", "full"])
def test_churned_workload_tables_are_identical(size):
    a = W.make("fp8", size, make_allocator=oracle.Allocator)
    b = W.make("fp8", size, make_allocator=pagedkv.BlockManager)
    assert a.num_blocks == b.num_blocks
    assert np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(a.context_lens, b.context_lens)
