"""Seeded synthetic workloads for the paged decode path.

This module only draws inputs: context lengths, block tables, slot positions,
query and K/V tensors.  It holds none of the method's arithmetic (no attention,
no quantisation) and imports neither the CUDA binding nor the oracle, so the
tests, the bench and the oracle can all take their inputs from it.

The five workloads mirror the shapes the pages talk about (Llama-3-8B / 70B
style GQA layers, 16-token blocks; "Optimizing KV Cache Memory Management in
vLLM...", section "The Math of the KV Cache Bottleneck"):

  tiny  4 seqs, ctx {5,16,33,70}, 64-block pool from a seeded permutation,
        2 query heads / 1 KV head, head_dim 64, plus a 4-token write
  8b    batch 64, 32/8 heads, head_dim 128, ctx ~ U{128..4096},
        pool 1.2x the needed blocks with shuffled ids, 1 new token per seq
  70b   batch 128, 64/8 heads, ctx ~ log-uniform [256, 8192]; every sequence
        maps its first 64 logical blocks to the same 64 physical blocks
  sw    batch 32, 32/8 heads, window 4096, ctx ~ U{4096..32768}; only blocks
        that hold a token of the last window have a table entry (others -1)
  fp8   batch 256, 32/8 heads, e4m3 KV with per-KV-head scales,
        ctx ~ U{1..16384}; tables come from a block allocator after a seeded
        churn of 10,000 alloc/free steps at 95% occupancy
  fp4   the fp8 workload's shape and table recipe (its own seeds) with an
        FP4 pool: E2M1 codes, E4M3 scales per 16 elements, per-KV-head scales

All numbers are N(0,1) draws from seeded torch generators; every sequence's
K/V comes from its own seed so that a subset can be regenerated alone.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16        # default tokens per block
GROWTH_TOKENS = 16     # tokens a churn step appends to a running request
CONFIGS = ("tiny", "8b", "70b", "sw", "fp8", "fp4")

DATA_SEED = {"tiny": 1000, "8b": 1001, "70b": 1002, "sw": 1003, "fp8": 1004, "long": 1005,
             "fp4": 1006}
TABLE_SEED = {"tiny": 2000, "8b": 2001, "70b": 2002, "sw": 2003, "fp8": 2004, "long": 2005,
              "fp4": 2006}


@dataclass
class Workload:
    name: str
    size: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    window: int                 # <= 0: no sliding window
    dtype: str                  # "bf16", "fp8" or "fp4"
    scale: float                # softmax scale
    context_lens: np.ndarray    # int32 [B]: tokens per sequence after this step's write
    block_tables: np.ndarray    # int32 [B, MBS]; -1 = no block mapped
    new_pos: np.ndarray         # int64 [B]: position written this step, -1 = none
    shared_prefix_tokens: int = 0
    prefix_blocks: np.ndarray | None = None   # int32: physical ids of the shared prefix
    k_scale: np.ndarray | None = None   # fp32 [Hkv] (fp8 and fp4 only)
    v_scale: np.ndarray | None = None
    data_seed: int = 0
    notes: dict = field(default_factory=dict)

    # ------------------------------------------------------------ geometry --
    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.batch else 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def attended_range(self, b: int) -> tuple[int, int]:
        """Positions [lo, ctx) the query of sequence b attends to."""
        ctx = int(self.context_lens[b])
        lo = max(0, ctx - self.window) if self.window > 0 else 0
        return lo, ctx

    def slot(self, b: int, pos: np.ndarray) -> np.ndarray:
        """Slots of positions `pos` of sequence b (b = -1: the shared prefix)."""
        pos = np.asarray(pos, dtype=np.int64)
        row = self.prefix_blocks if b < 0 else self.block_tables[b]
        blk = row[pos // self.block_size].astype(np.int64)
        return blk * self.block_size + pos % self.block_size

    def attended_tokens(self) -> int:
        return int(sum(self.attended_range(b)[1] - self.attended_range(b)[0]
                       for b in range(self.batch)))

    def kv_bytes_per_token_head(self) -> int:
        """Stored K+V bytes of one token of one KV head: 2 bytes an element
        (bf16), 1 (FP8), or half a byte plus one scale byte per 16 (FP4)."""
        if self.dtype == "bf16":
            return 2 * self.head_dim * 2
        if self.dtype == "fp8":
            return 2 * self.head_dim
        return 2 * (self.head_dim // 2 + self.head_dim // 16)

    def kv_bytes_attended(self) -> int:
        """K+V bytes of the attended tokens (per layer), the roofline's unit of work."""
        return self.attended_tokens() * self.n_kv_heads * self.kv_bytes_per_token_head()

    def kv_bytes_unique(self) -> int:
        """K+V bytes of distinct attended tokens: the shared prefix counts once."""
        P = self.shared_prefix_tokens
        n = 0
        prefix_read = 0
        for b in range(self.batch):
            lo, ctx = self.attended_range(b)
            if P:
                if lo < min(ctx, P):
                    prefix_read = max(prefix_read, min(ctx, P))
                n += max(0, ctx - max(lo, P))
            else:
                n += ctx - lo
        return (n + prefix_read) * self.n_kv_heads * self.kv_bytes_per_token_head()

    # ---------------------------------------------------------------- data --
    def _gen(self, key: int, device) -> torch.Generator:
        seed = int(np.random.SeedSequence([self.data_seed, key + 1]).generate_state(1)[0])
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        return g

    def query(self, device="cpu") -> torch.Tensor:
        g = self._gen(1_000_000_007, device)
        return torch.randn(self.batch, self.n_q_heads, self.head_dim, generator=g,
                           device=device, dtype=torch.float32).to(torch.bfloat16)

    def segments(self):
        """Token ranges whose K/V must be in the pool, each with its own seed.

        Yields (key, b, positions): b is the sequence whose table maps the
        positions, or -1 for the shared prefix (key -1)."""
        if self.shared_prefix_tokens:
            yield (-1, -1, np.arange(self.shared_prefix_tokens, dtype=np.int64))
        for b in range(self.batch):
            lo, ctx = self.attended_range(b)
            if self.shared_prefix_tokens:
                lo = max(lo, self.shared_prefix_tokens)
            if ctx > lo:
                yield (b, b, np.arange(lo, ctx, dtype=np.int64))

    def segment_kv(self, key: int, n: int, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
        g = self._gen(key, device)
        shape = (n, self.n_kv_heads, self.head_dim)
        k = torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        v = torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        return k, v

    def fill_plan(self, seqs=None, device="cpu"):
        """(setup, step) writes: each a list of (k, v, slots) with slots int64.

        `setup` holds every cached token except this step's new ones; `step`
        holds one token per sequence (slot -1 where nothing is written).  With
        `seqs`, only those sequences' segments (and the shared prefix) are made."""
        want = None if seqs is None else set(int(s) for s in seqs)
        setup, step_k, step_v = [], {}, {}
        for key, b, pos in self.segments():
            if want is not None and key >= 0 and key not in want:
                continue
            k, v = self.segment_kv(key, len(pos), device)
            slots = self.slot(b, pos)
            new = int(self.new_pos[b]) if b >= 0 else -1
            if key >= 0 and new >= 0 and pos[-1] == new:
                step_k[b], step_v[b] = k[-1:], v[-1:]
                k, v, slots = k[:-1], v[:-1], slots[:-1]
            if len(slots):
                setup.append((k, v, torch.from_numpy(np.ascontiguousarray(slots))))
        B = self.batch
        kz = torch.zeros(B, self.n_kv_heads, self.head_dim, dtype=torch.bfloat16, device=device)
        vz = torch.zeros_like(kz)
        slots = np.full(B, -1, dtype=np.int64)
        for b in step_k:
            kz[b] = step_k[b][0]
            vz[b] = step_v[b][0]
            slots[b] = self.slot(b, np.array([self.new_pos[b]]))[0]
        return setup, (kz, vz, torch.from_numpy(slots))


# ------------------------------------------------------------------ tables --

def _tables_from_ids(lens_blocks: list[int], ids: np.ndarray, mbs: int) -> np.ndarray:
    t = np.full((len(lens_blocks), max(mbs, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(lens_blocks):
        t[b, :n] = ids[off:off + n]
        off += n
    return t


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _tiny(size: str, bs: int = BLOCK_SIZE) -> Workload:
    rng = np.random.default_rng(TABLE_SEED["tiny"])
    lens = np.array([5, 16, 33, 70], dtype=np.int32)
    nb = 64
    perm = rng.permutation(nb).astype(np.int32)
    nblk = [_cdiv(int(c), bs) for c in lens]
    tables = _tables_from_ids(nblk, perm, max(nblk))
    return Workload("tiny", size, 4, 2, 1, 64, bs, nb, 0, "bf16", 1.0 / math.sqrt(64),
                    lens, tables, (lens - 1).astype(np.int64), data_seed=DATA_SEED["tiny"])


def _8b(size: str, bs: int = BLOCK_SIZE) -> Workload:
    rng = np.random.default_rng(TABLE_SEED["8b"])
    B = 64 if size == "full" else 8
    lens = rng.integers(128, 4096, size=B, endpoint=True).astype(np.int32)
    nblk = [_cdiv(int(c), bs) for c in lens]
    needed = sum(nblk)
    nb = math.ceil(1.2 * needed)
    perm = rng.permutation(nb).astype(np.int32)
    tables = _tables_from_ids(nblk, perm, max(nblk))
    return Workload("8b", size, B, 32, 8, 128, bs, nb, 0, "bf16", 1.0 / math.sqrt(128),
                    lens, tables, (lens - 1).astype(np.int64), data_seed=DATA_SEED["8b"])


def _70b(size: str, bs: int = BLOCK_SIZE) -> Workload:
    rng = np.random.default_rng(TABLE_SEED["70b"])
    B = 128 if size == "full" else 12
    u = rng.uniform(math.log(256), math.log(8192), size=B)
    lens = np.clip(np.round(np.exp(u)), 256, 8192).astype(np.int32)
    prefix_blocks = 1024 // bs
    private = [max(0, _cdiv(int(c), bs) - prefix_blocks) for c in lens]
    needed = prefix_blocks + sum(private)
    nb = math.ceil(1.2 * needed)
    perm = rng.permutation(nb).astype(np.int32)
    shared = perm[:prefix_blocks]
    mbs = max(_cdiv(int(c), bs) for c in lens)
    tables = np.full((B, mbs), -1, dtype=np.int32)
    off = prefix_blocks
    for b, c in enumerate(lens):
        n = _cdiv(int(c), bs)
        tables[b, :min(n, prefix_blocks)] = shared[:min(n, prefix_blocks)]
        if n > prefix_blocks:
            tables[b, prefix_blocks:n] = perm[off:off + n - prefix_blocks]
            off += n - prefix_blocks
    # Sequences that live inside the shared prefix write nothing this step:
    # their newest token is already part of the shared blocks.
    new_pos = np.where(lens > prefix_blocks * bs, lens - 1, -1).astype(np.int64)
    return Workload("70b", size, B, 64, 8, 128, bs, nb, 0, "bf16", 1.0 / math.sqrt(128),
                    lens, tables, new_pos, shared_prefix_tokens=prefix_blocks * bs,
                    prefix_blocks=shared.copy(), data_seed=DATA_SEED["70b"])


def _sw(size: str, bs: int = BLOCK_SIZE) -> Workload:
    rng = np.random.default_rng(TABLE_SEED["sw"])
    B = 32 if size == "full" else 4
    W = 4096
    lens = rng.integers(4096, 32768, size=B, endpoint=True).astype(np.int32)
    mbs = _cdiv(32768, bs)
    first = [(int(c) - W) // bs for c in lens]
    last = [(int(c) - 1) // bs for c in lens]
    needed = sum(l - f + 1 for f, l in zip(first, last))
    nb = math.ceil(1.2 * needed)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((B, mbs), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = last[b] - first[b] + 1
        tables[b, first[b]:last[b] + 1] = perm[off:off + n]
        off += n
    return Workload("sw", size, B, 32, 8, 128, bs, nb, W, "bf16", 1.0 / math.sqrt(128),
                    lens, tables, (lens - 1).astype(np.int64), data_seed=DATA_SEED["sw"])


def churn_tables(make_allocator, final_lens: np.ndarray, steps: int, occupancy: float,
                 seed: int, max_len: int, bs: int = BLOCK_SIZE) -> tuple[int, np.ndarray, dict]:
    """Block tables for `final_lens` taken from an allocator after a seeded churn.

    The pool holds ceil(needed / occupancy) blocks.  Each churn step admits a
    request of U{1..max_len} tokens while fewer than occupancy * NB blocks are
    in use (a preempted request waits at the head of the queue and is admitted
    again first), and otherwise frees a uniformly chosen running request;
    every 4th step also grows a random running request by one block of
    tokens.  Then every running request is freed in a seeded order and the
    final requests are admitted one after another.  `make_allocator(NB, BS)`
    returns an object with admit/append/free/preempt_newest/table/num_free.
    """
    rng = np.random.default_rng(seed)
    needed = int(sum(_cdiv(int(c), bs) for c in final_lens))
    nb = math.ceil(needed / occupancy)
    alloc = make_allocator(nb, bs)
    running: list[int] = []
    waiting: list[tuple[int, int]] = []   # (req_id, tokens), head first
    next_id = 0
    stats = {"admitted": 0, "freed": 0, "grown": 0, "preempted": 0}
    sizes: dict[int, int] = {}

    def admit(rid: int, n: int) -> bool:
        while True:
            rc, _ = alloc.admit(rid, num_tokens=n)
            if rc == 0:
                running.append(rid)
                return True
            if not running:
                return False
            rc2, victim = alloc.preempt_newest()
            if rc2 != 0:
                return False
            running.remove(victim)
            waiting.insert(0, (victim, sizes[victim]))
            stats["preempted"] += 1

    for step in range(steps):
        used = nb - alloc.num_free()
        if used < occupancy * nb:
            if waiting:
                rid, n = waiting.pop(0)
            else:
                rid, n = next_id, int(rng.integers(1, max_len, endpoint=True))
                next_id += 1
                sizes[rid] = n
            if admit(rid, n):
                stats["admitted"] += 1
        elif running:
            rid = running.pop(int(rng.integers(0, len(running))))
            alloc.free(rid)
            stats["freed"] += 1
        if step % 4 == 3 and running:
            rid = running[int(rng.integers(0, len(running)))]
            if alloc.append(rid, n=GROWTH_TOKENS) == 0:
                sizes[rid] += GROWTH_TOKENS
                stats["grown"] += 1
    for i in rng.permutation(len(running)):
        alloc.free(running[i])
    base = 1 << 40
    mbs = max(_cdiv(int(c), bs) for c in final_lens)
    tables = np.full((len(final_lens), mbs), -1, dtype=np.int32)
    for b, c in enumerate(final_lens):
        rc, _ = alloc.admit(base + b, num_tokens=int(c))
        if rc != 0:
            raise RuntimeError("final admission failed")
        t = alloc.table(base + b)
        tables[b, :len(t)] = t
    stats["occupancy"] = (nb - alloc.num_free()) / nb
    return nb, tables, stats


FP8_K_SCALE_BASE = 5.0   # per-KV-head scale = (base + step * h) / 448
FP8_V_SCALE_BASE = 5.5


def _fp8(size: str, make_allocator=None, bs: int = BLOCK_SIZE, fmt: str = "fp8") -> Workload:
    rng = np.random.default_rng(TABLE_SEED[fmt])
    B = 256 if size == "full" else 16
    max_len = 16384 if size == "full" else 4096
    steps = 10_000 if size == "full" else 2_000
    lens = rng.integers(1, max_len, size=B, endpoint=True).astype(np.int32)
    if make_allocator is None:
        raise ValueError(f"the {fmt} workload needs a block allocator (make_allocator)")
    nb, tables, stats = churn_tables(make_allocator, lens, steps, 0.95,
                                     int(rng.integers(0, 2**31)), max_len, bs)
    hkv = 8
    # Fixed per-KV-head scales: N(0,1) data saturates only beyond ~5 sigma.
    # FP4: the head scale spans the E4M3 block scales' range once more (6 is
    # the largest E2M1 magnitude), so a 16-element group's scale stays <= 448.
    div = 448.0 if fmt == "fp8" else 6.0 * 448.0
    k_scale = ((FP8_K_SCALE_BASE + 0.25 * np.arange(hkv)) / div).astype(np.float32)
    v_scale = ((FP8_V_SCALE_BASE + 0.125 * np.arange(hkv)) / div).astype(np.float32)
    return Workload(fmt, size, B, 32, hkv, 128, bs, nb, 0, fmt, 1.0 / math.sqrt(128),
                    lens, tables, (lens - 1).astype(np.int64), k_scale=k_scale,
                    v_scale=v_scale, data_seed=DATA_SEED[fmt], notes={"churn": stats})


def _long(size: str, bs: int = BLOCK_SIZE) -> Workload:
    """8B-shaped decode over long contexts (the regime where the pages expect
    32-token blocks to pay): batch 16, ctx U{32768..65536}."""
    rng = np.random.default_rng(TABLE_SEED["long"])
    B = 16 if size == "full" else 3
    lo_len, hi_len = (32768, 65536) if size == "full" else (2048, 4096)
    lens = rng.integers(lo_len, hi_len, size=B, endpoint=True).astype(np.int32)
    nblk = [_cdiv(int(c), bs) for c in lens]
    nb = math.ceil(1.2 * sum(nblk))
    perm = rng.permutation(nb).astype(np.int32)
    tables = _tables_from_ids(nblk, perm, max(nblk))
    return Workload("long", size, B, 32, 8, 128, bs, nb, 0, "bf16", 1.0 / math.sqrt(128),
                    lens, tables, (lens - 1).astype(np.int64), data_seed=DATA_SEED["long"])


def make(name: str, size: str = "full", make_allocator=None, block_size: int = BLOCK_SIZE) -> Workload:
    """Build workload `name` ("tiny", "8b", "70b", "sw", "fp8", "fp4", "long") at size
    "full" or "small", with pool blocks of `block_size` tokens (16 or 32)."""
    if size not in ("full", "small"):
        raise ValueError(size)
    if block_size not in (16, 32):
        raise ValueError(block_size)
    if name == "tiny":
        return _tiny(size, block_size)
    if name == "8b":
        return _8b(size, block_size)
    if name == "70b":
        return _70b(size, block_size)
    if name == "sw":
        return _sw(size, block_size)
    if name in ("fp8", "fp4"):
        return _fp8(size, make_allocator, block_size, name)
    if name == "long":
        return _long(size, block_size)
    raise ValueError(f"unknown workload {name!r}")
