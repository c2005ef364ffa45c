"""Pins of the oracle's block-pool bookkeeping against the pages' worked
examples and stated answers, and against invariants under seeded churn.

Sources: "PagedAttention" (zhangchitc.github.io/posts/paged-attention), the
4-request walk-through; "Why the KV cache is a pool of 16-token blocks",
follow-ups (25 shared tokens -> 16 cached; salts; preempting the newest);
"The memory behind the next token", sections "Sharing requires explicit
ownership" and "How vLLM recognizes a reusable prefix" (10 shared tokens with
4-token blocks -> 8 reused; full-hit cap; append-only duplicates; salt)."""

import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_33_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _toks(s: str) -> list[int]:
    return [ord(c) for c in s]


def _chain(tokens, bs, salt=b"", extra=b""):
    """Expected chain hashes from the documented hash input (hashlib is the library here)."""
    import hashlib
    out, parent = [], bytes(32)
    for i in range(len(tokens) // bs):
        blk = np.asarray(tokens[i * bs:(i + 1) * bs], dtype="<i4").tobytes()
        h = hashlib.sha256(parent + blk + extra + (salt if i == 0 else b"")).digest()
        out.append(h)
        parent = h
    return out


def test_worked_example_from_the_pages():
    ex = json.load(open(os.path.join(GOLDEN, "p4_worked_example.json")))
    bs = ex["block_size"]
    a = oracle.Allocator(ex["pool_blocks"], bs)
    ids = {"R1": 1, "R2": 2, "R3": 3}
    for ev in ex["events"]:
        r = ev["req"]
        if ev["op"] == "admit":
            rc, cached = a.admit(ids[r], tokens=_toks(ex["requests"][r]))
            assert rc == 0
            assert cached == ev["cached_tokens"], ev
            want = ev.get("table", ev.get("table_rules"))
            assert a.table(ids[r]) == want, ev
        else:
            assert a.free(ids[r]) == 0
        for blk, ref in ev["ref_cnt"].items():
            assert a.block(int(blk))[0] == ref, (ev["t"], blk)
        for blk in ev.get("hashed_blocks", []):
            assert a.block(blk)[1] is not None
        for blk in ev.get("unhashed_blocks", []):
            assert a.block(blk)[1] is None
        for blk in ev.get("free_blocks", []):
            assert blk in a.free_queue()
        if "free_count" in ev:
            assert a.num_free() == ev["free_count"]
        assert len(a.map_entries()) == ev["map_size"], ev["t"]
        if "evicted_prefix" in ev:
            gone = _chain(_toks(ev["evicted_prefix"]), bs)[-1]
            assert a.lookup(gone) == -1
    # rule-derived R3 table differs from the page's simplified diagram
    assert ex["events"][-1]["table_page"] != ex["events"][-1]["table_rules"]


def test_hash_is_the_documented_sha256_chain():
    a = oracle.Allocator(8, 4)
    toks = _toks("ABCDEFGHIJ")
    a.admit(1, tokens=toks, salt=b"s1", extra=b"lora:x")
    want = _chain(toks, 4, salt=b"s1", extra=b"lora:x")
    t = a.table(1)
    assert [a.block(t[i])[1] for i in range(2)] == want
    assert a.block(t[2])[1] is None  # partial block is not hashed


def test_25_shared_tokens_reuse_one_block():
    a = oracle.Allocator(32, 16)
    p = list(range(100, 125))
    assert a.admit(1, tokens=p) == (0, 0)
    rc, cached = a.admit(2, tokens=p)
    assert rc == 0 and cached == 16 and 25 - cached == 9


def test_10_shared_tokens_with_4_token_blocks_reuse_8():
    a = oracle.Allocator(32, 4)
    a.admit(1, tokens=list(range(10)) + [500, 501, 502])
    rc, cached = a.admit(2, tokens=list(range(10)) + [900, 901])
    assert cached == 8


def test_full_hit_still_computes_the_last_token():
    a = oracle.Allocator(32, 16)
    p = list(range(32))
    a.admit(1, tokens=p)
    rc, cached = a.admit(2, tokens=p)
    assert cached == 16   # floor((32-1)/16) blocks, never all 32 tokens
    rc, cached = a.admit(3, tokens=list(range(33)))
    assert cached == 32


def test_different_salts_never_share_blocks():
    a = oracle.Allocator(32, 16)
    p = list(range(48))
    a.admit(1, tokens=p, salt=b"tenant-a-secret")
    assert a.admit(2, tokens=p, salt=b"tenant-b-secret")[1] == 0
    assert a.admit(3, tokens=p, salt=b"tenant-a-secret")[1] == 32
    assert not set(a.table(1)) & set(a.table(2))


def test_extra_keys_separate_adapters():
    a = oracle.Allocator(32, 16)
    p = list(range(40))
    a.admit(1, tokens=p, extra=b"lora-1")
    assert a.admit(2, tokens=p, extra=b"lora-2")[1] == 0
    assert a.admit(3, tokens=p, extra=b"lora-1")[1] == 32


def test_position_is_part_of_identity():
    a = oracle.Allocator(32, 4)
    a.admit(1, tokens=_toks("XXXXABCDEFGH"))
    # the same block ABCD after a different first block does not hit
    assert a.admit(2, tokens=_toks("YYYYABCDZZ"))[1] == 0


def test_touch_pulls_free_block_out_of_queue_before_counting():
    a = oracle.Allocator(6, 4)
    a.admit(1, tokens=_toks("ABCDEFGH"))
    a.free(1)
    assert a.num_free() == 6
    rc, cached = a.admit(2, tokens=_toks("ABCDEFGHI"))
    assert cached == 8
    t = a.table(2)
    assert t[:2] == [0, 1]
    assert 0 not in a.free_queue() and 1 not in a.free_queue()
    assert a.block(0)[0] == 1 and a.num_free() == 3


def test_reverse_order_free_and_lru_reuse():
    a = oracle.Allocator(8, 4)
    a.admit(1, num_tokens=12)          # blocks 0,1,2
    a.admit(2, num_tokens=4)           # block 3
    assert a.free_queue() == [4, 5, 6, 7]
    a.free(1)
    assert a.free_queue() == [4, 5, 6, 7, 2, 1, 0]   # tail block released first
    a.admit(3, num_tokens=20)          # takes the five longest unused
    assert a.table(3) == [4, 5, 6, 7, 2]


def test_lazy_eviction_keeps_hash_until_reuse():
    a = oracle.Allocator(3, 4)
    a.admit(1, tokens=_toks("ABCDEFGH"))
    h = _chain(_toks("ABCDEFGH"), 4)
    a.free(1)
    assert a.lookup(h[0]) == 0 and a.lookup(h[1]) == 1   # still cached while free
    assert a.stats()["evictions"] == 0
    a.admit(2, num_tokens=4)           # queue head is block 2 (never hashed)
    assert a.lookup(h[1]) == 1 and a.stats()["evictions"] == 0
    a.admit(3, num_tokens=4)           # next head: block 1 (freed first) -> evicted now
    assert a.table(3) == [1]
    assert a.lookup(h[1]) == -1 and a.lookup(h[0]) == 0
    assert a.stats()["evictions"] == 1


def test_append_only_tables_may_duplicate_a_cached_hash():
    a = oracle.Allocator(8, 4)
    a.admit(1, tokens=_toks("ABCDEF"))
    a.append(1, tokens=_toks("GHI"))          # block "EFGH" fills and is cached
    h = _chain(_toks("ABCDEFGH"), 4)
    first = a.table(1)
    assert a.lookup(h[1]) == first[1]
    rc, cached = a.admit(2, tokens=_toks("ABCDEF"))
    assert cached == 4
    a.append(2, tokens=_toks("GH"))           # its own "EFGH" block fills too
    second = a.table(2)
    assert second[0] == first[0] and second[1] != first[1]   # table not rewritten
    assert a.block(second[1])[1] == h[1]                     # same hash, two blocks
    assert a.lookup(h[1]) == first[1]                        # map keeps the first
    a.free(2)
    assert a.lookup(h[1]) == first[1]


def test_decode_growth_takes_a_block_every_block_size_tokens():
    a = oracle.Allocator(8, 16)
    a.admit(1, num_tokens=16)
    assert len(a.table(1)) == 1
    a.append(1, n=1)                   # 16 -> 17 crosses a boundary
    assert len(a.table(1)) == 2
    a.append(1, n=15)
    assert len(a.table(1)) == 2
    a.append(1, n=1)
    assert len(a.table(1)) == 3


def test_out_of_blocks_preempts_the_newest():
    a = oracle.Allocator(6, 16)
    a.admit(1, num_tokens=32)
    a.admit(2, num_tokens=32)
    a.admit(3, num_tokens=16)
    assert a.admit(4, num_tokens=32)[0] == oracle.OOM      # all-or-nothing
    assert a.num_free() == 1
    rc, victim = a.preempt_newest()
    assert rc == 0 and victim == 3 and a.num_free() == 2
    assert a.admit(4, num_tokens=32)[0] == 0
    assert a.append(4, n=1) == oracle.OOM
    for expect in (4, 2, 1):
        assert a.preempt_newest() == (0, expect)
    assert a.preempt_newest()[0] == oracle.OOM
    assert a.stats()["preemptions"] == 4 and a.num_free() == 6


def _check_invariants(a: oracle.Allocator, live: dict[int, int], bs: int):
    refs = np.zeros(a.num_blocks, dtype=np.int64)
    for rid, ntok in live.items():
        t = a.table(rid)
        assert len(t) == -(-ntok // bs)                       # waste <= bs-1 tokens
        assert len(t) * bs - ntok <= bs - 1
        for blk in t:
            refs[blk] += 1
    for blk in range(a.num_blocks):
        assert a.block(blk)[0] == refs[blk]
    fq = a.free_queue()
    assert len(fq) == len(set(fq)) == a.num_free()
    assert set(fq) == {b for b in range(a.num_blocks) if refs[b] == 0}
    for h, blk in a.map_entries().items():
        assert a.block(blk)[1] == h


def test_invariants_hold_under_seeded_churn():
    rng = np.random.default_rng(123)
    bs = 4
    a = oracle.Allocator(64, bs)
    live: dict[int, int] = {}
    vocab = 3
    for step in range(1500):
        op = rng.integers(0, 4)
        if op <= 1:
            rid = step
            n = int(rng.integers(1, 30))
            toks = rng.integers(0, vocab, n)      # small vocabulary: many prefix hits
            rc, _ = a.admit(rid, tokens=toks, salt=bytes([int(rng.integers(0, 2))]))
            if rc == 0:
                live[rid] = n
            else:
                assert rc == oracle.OOM
        elif op == 2 and live:
            rid = list(live)[int(rng.integers(0, len(live)))]
            n = int(rng.integers(1, 9))
            if a.append(rid, tokens=rng.integers(0, vocab, n)) == 0:
                live[rid] += n
        elif live:
            rid = list(live)[int(rng.integers(0, len(live)))]
            assert a.free(rid) == 0
            del live[rid]
        if step % 50 == 0:
            _check_invariants(a, live, bs)
    _check_invariants(a, live, bs)
    st = a.stats()
    assert st["hits"] > 0 and st["evictions"] > 0


def test_churned_tables_reach_the_requested_occupancy():
    w = workloads.make("fp8", "small", make_allocator=oracle.Allocator)
    used = sum(-(-int(c) // 16) for c in w.context_lens)
    ids = w.block_tables[w.block_tables >= 0]
    assert len(ids) == used and len(np.unique(ids)) == used
    assert ids.min() >= 0 and ids.max() < w.num_blocks
    assert abs(used / w.num_blocks - 0.95) < 0.01
    # the churn scatters the ids: far from the identity layout
    assert np.mean(np.diff(w.block_tables[0][: -(-int(w.context_lens[0]) // 16)]) == 1) < 0.9


# ------------------------------------------------------ fork / copy-on-write --

def test_cow_walkthrough_from_the_pages():
    ex = json.load(open(os.path.join(GOLDEN, "cow_walkthrough.json")))
    a = oracle.Allocator(ex["pool_blocks"], ex["block_size"])
    for ev in ex["events"]:
        if ev["op"] == "admit":
            assert a.admit(ev["seq"], num_tokens=ev["tokens"])[0] == 0
        elif ev["op"] == "fork":
            assert a.fork(ev["parent"], ev["child"]) == 0
        else:
            assert a.append(ev["seq"], n=ev["n"]) == 0
        for seq, table in ev["table"].items():
            assert a.table(int(seq)) == table, ev
        assert a.num_free() == ev["free"], ev
        for blk, ref in ev["ref_cnt"].items():
            assert a.block(int(blk))[0] == ref, ev
        assert [list(p) for p in a.copies()] == ev["copies"], ev
        for seq, n in ev.get("num_tokens", {}).items():
            assert a.num_tokens(int(seq)) == n


def test_fork_of_a_full_last_block_needs_no_copy():
    a = oracle.Allocator(8, 4)
    assert a.admit(1, num_tokens=8)[0] == 0
    assert a.fork(1, 2) == 0
    assert a.append(2, n=1) == 0            # position 8 opens a new block
    assert a.table(2) == [0, 1, 2] and a.table(1) == [0, 1]
    assert a.copies() == []
    assert a.fork(1, 2) == 1 and a.fork(9, 3) == 1   # child exists / unknown parent


def test_copy_on_write_counts_its_block_against_capacity():
    a = oracle.Allocator(3, 4)
    assert a.admit(1, num_tokens=6)[0] == 0             # blocks 0, 1 (1 partly full)
    assert a.fork(1, 2) == 0
    assert a.append(2, n=3) == oracle.OOM               # copy + new block: 2 needed, 1 free
    assert a.table(2) == [0, 1] and a.copies() == []    # all-or-nothing
    assert a.append(2, n=2) == 0                        # copy only
    assert a.table(2) == [0, 2] and a.copies() == [(1, 2)]


def test_every_request_reads_back_only_its_own_tokens():
    """Brute force over a token-per-slot store: admitted tokens are written
    from the first uncached position, pending copies are applied before each
    append's writes, and after every step each live request's table must
    yield exactly its own token history.  A missed copy-on-write lets one
    sharer overwrite another's block; a wrong or reversed copy pair brings in
    the wrong contents; a wrong prefix hit maps foreign tokens."""
    rng = np.random.default_rng(7)
    bs = 4
    a = oracle.Allocator(48, bs)
    store = np.full(48 * bs, -1, dtype=np.int64)
    hist: dict[int, list[int]] = {}

    def write(rid, first):
        t = a.table(rid)
        for p in range(first, len(hist[rid])):
            store[t[p // bs] * bs + p % bs] = hist[rid][p]

    def apply_copies():
        for src, dst in a.copies():
            store[dst * bs:(dst + 1) * bs] = store[src * bs:(src + 1) * bs]

    next_id = 0
    forks = cows = 0
    for step in range(3000):
        op = int(rng.integers(0, 10))
        live = list(hist)
        if op <= 2 or not live:
            toks = rng.integers(0, 3, int(rng.integers(1, 14))).tolist()
            rc, cached = a.admit(next_id, tokens=toks)
            if rc == 0:
                hist[next_id] = list(toks)
                write(next_id, cached)
            next_id += 1
        elif op <= 4:
            parent = live[int(rng.integers(0, len(live)))]
            assert a.fork(parent, next_id) == 0
            hist[next_id] = list(hist[parent])
            next_id += 1
            forks += 1
        elif op <= 7:
            rid = live[int(rng.integers(0, len(live)))]
            toks = rng.integers(0, 3, int(rng.integers(1, 6))).tolist()
            before = len(hist[rid])
            if a.append(rid, tokens=toks) == 0:
                pend = a.copies(take=False)
                cows += len(pend)
                apply_copies()
                hist[rid] += toks
                write(rid, before)
            else:
                assert a.copies(take=False) == []
        elif op == 8:
            rid = live[int(rng.integers(0, len(live)))]
            assert a.free(rid) == 0
            del hist[rid]
        else:
            rc, rid = a.preempt_newest()
            if rc == 0:
                del hist[rid]
        for rid, h in hist.items():
            t = a.table(rid)
            got = [int(store[t[p // bs] * bs + p % bs]) for p in range(len(h))]
            assert got == h, (step, rid)
        if step % 100 == 0:
            _check_invariants(a, {r: len(h) for r, h in hist.items()}, bs)
    assert forks > 100 and cows > 15
