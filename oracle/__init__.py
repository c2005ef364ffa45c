"""Oracle for the paged KV cache decode path -- TEST INFRASTRUCTURE ONLY.

A plain single-threaded C++ restatement (fp64 for the attention) of what the
pages compute: the bf16 / FP8-E4M3 / FP4-E2M1 formats, the paged KV write, paged decode
attention walking the block table, and the host block pool (LRU free queue,
ref_cnt, touch, reverse-order free, chained SHA-256 hashes, lazy eviction,
preemption).  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  It shares no code with the CUDA
library ``paged_kv_cache_33_gb300`` and neither imports the other.

Every function of the C library cites the page section it restates; this
module only marshals numpy arrays into it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SOURCES = ["attention.cpp", "allocator.cpp", "sha256.cpp"]
LIB_PATH = os.path.join(_HERE, "liboracle.so")

OK, INVALID_ARG, OOM, BAD_BLOCK_ID = 0, 1, 2, 5


def build_command(out_path: str = LIB_PATH) -> list[str]:
    """The g++ command that builds the oracle (no -ffast-math, no contraction)."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    return ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
            "-o", out_path] + srcs


def build(out_path: str = LIB_PATH) -> subprocess.Popen:
    """Start compiling liboracle.so; the caller waits on the returned process."""
    return subprocess.Popen(build_command(out_path), stdout=subprocess.PIPE,
                            stderr=subprocess.STDOUT)


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(os.path.join(_HERE, s)) > t
               for s in _SOURCES + ["oracle.h"])


_lib = None


def lib() -> ctypes.CDLL:
    """Load liboracle.so, compiling it first when missing or older than its sources."""
    global _lib
    if _lib is not None:
        return _lib
    if _stale():
        proc = build()
        out, _ = proc.communicate()
        if proc.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + out.decode(errors="replace"))
    L = ctypes.CDLL(LIB_PATH)
    c = ctypes
    P = c.c_void_p
    sig = {
        "oracle_bf16_to_double": (c.c_double, [c.c_uint16]),
        "oracle_e4m3_to_double": (c.c_double, [c.c_uint8]),
        "oracle_e4m3_from_float": (c.c_uint8, [c.c_float]),
        "oracle_e4m3_quantize": (c.c_uint8, [c.c_uint16, c.c_float]),
        "oracle_e2m1_to_double": (c.c_double, [c.c_uint8]),
        "oracle_e2m1_from_float": (c.c_uint8, [c.c_float]),
        "oracle_fp4_quantize_row": (None, [P, c.c_int32, c.c_float, P, P]),
        "oracle_pool_block_scales": (P, [P]),
        "oracle_pool_create": (P, [c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int32]),
        "oracle_pool_destroy": (None, [P]),
        "oracle_pool_data": (P, [P]),
        "oracle_pool_bytes": (c.c_uint64, [P]),
        "oracle_pool_set_scales": (c.c_int, [P, P, P]),
        "oracle_kv_write": (c.c_int, [P, P, P, P, c.c_int64]),
        "oracle_pool_copy_blocks": (c.c_int, [P, P, c.c_int64]),
        "oracle_paged_decode": (c.c_int, [P, P, c.c_int32, P, c.c_int32, P, c.c_int32,
                                          c.c_double, c.c_int32, P, c.c_int32, P]),
        "oracle_paged_prefill": (c.c_int, [P, P, c.c_int32, P, P, c.c_int32, P, c.c_int32,
                                           c.c_double, c.c_int32, P]),
        "oracle_sha256": (None, [P, c.c_uint64, P]),
        "oracle_alloc_create": (P, [c.c_int32, c.c_int32]),
        "oracle_alloc_destroy": (None, [P]),
        "oracle_alloc_admit": (c.c_int, [P, c.c_int64, P, c.c_int64, P, c.c_int32, P,
                                         c.c_int32, P]),
        "oracle_alloc_append": (c.c_int, [P, c.c_int64, P, c.c_int64]),
        "oracle_alloc_free": (c.c_int, [P, c.c_int64]),
        "oracle_alloc_fork": (c.c_int, [P, c.c_int64, c.c_int64]),
        "oracle_alloc_copies": (c.c_int64, [P, P, c.c_int64, c.c_int32]),
        "oracle_alloc_preempt_newest": (c.c_int, [P, P]),
        "oracle_alloc_table": (c.c_int, [P, c.c_int64, P, c.c_int64, P]),
        "oracle_alloc_num_tokens": (c.c_int64, [P, c.c_int64]),
        "oracle_alloc_num_free": (c.c_int32, [P]),
        "oracle_alloc_free_queue": (c.c_int32, [P, P, c.c_int32]),
        "oracle_alloc_block_info": (c.c_int, [P, c.c_int32, P, P, P]),
        "oracle_alloc_lookup": (c.c_int32, [P, P]),
        "oracle_alloc_map_size": (c.c_int32, [P]),
        "oracle_alloc_map_entries": (c.c_int32, [P, P, P, c.c_int32]),
        "oracle_alloc_stats": (None, [P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(x) -> np.ndarray:
    """bf16 data as its uint16 bit patterns (accepts a torch bf16 tensor or uint16 array)."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)
    a = np.ascontiguousarray(x)
    assert a.dtype == np.uint16, a.dtype
    return a


# ------------------------------------------------------------------ formats --

def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code))


def e4m3_from_float(x: float) -> int:
    return int(lib().oracle_e4m3_from_float(float(x)))


def e4m3_quantize(bf16_bits: int, scale: float) -> int:
    return int(lib().oracle_e4m3_quantize(int(bf16_bits), float(scale)))


def e2m1_to_double(code: int) -> float:
    return lib().oracle_e2m1_to_double(int(code))


def e2m1_from_float(x: float) -> int:
    return int(lib().oracle_e2m1_from_float(float(x)))


def fp4_quantize_row(x, head_scale: float) -> tuple[np.ndarray, np.ndarray]:
    """One row of bf16 values (length a multiple of 16) -> (E2M1 codes, E4M3 block scales)."""
    x = _u16(x).reshape(-1)
    n = x.shape[0]
    codes = np.zeros(n, np.uint8)
    scales = np.zeros(n // 16, np.uint8)
    lib().oracle_fp4_quantize_row(_ptr(x), n, float(head_scale), _ptr(codes), _ptr(scales))
    return codes, scales


# --------------------------------------------------------------------- pool --

class Pool:
    """Host KV pool in the pages' block shape: [num_blocks, 2, BS, Hkv, D]."""

    def __init__(self, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                 dtype: str = "bf16"):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.n_kv_heads, self.head_dim = int(n_kv_heads), int(head_dim)
        self.dtype = dtype
        code = {"bf16": 0, "fp8": 1, "fp4": 2}[dtype]
        self._h = lib().oracle_pool_create(self.num_blocks, self.block_size, self.n_kv_heads,
                                           self.head_dim, code)
        if not self._h:
            raise ValueError("oracle_pool_create rejected its arguments")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.oracle_pool_destroy(h)

    def array(self) -> np.ndarray:
        """A numpy view of the pool: [NB, 2, BS, Hkv, D] of uint16 (bf16) or uint8
        (an E4M3 code, or an E2M1 code in the low four bits, per element)."""
        n = lib().oracle_pool_bytes(self._h)
        buf = (ctypes.c_uint8 * n).from_address(lib().oracle_pool_data(self._h))
        a = np.frombuffer(buf, dtype=np.uint8)
        if self.dtype == "bf16":
            a = a.view(np.uint16)
        return a.reshape(self.num_blocks, 2, self.block_size, self.n_kv_heads, self.head_dim)

    def block_scales(self) -> np.ndarray:
        """FP4 pools: the E4M3 block scales, [NB, 2, BS, Hkv, D / 16] of uint8."""
        assert self.dtype == "fp4"
        n = self.num_blocks * 2 * self.block_size * self.n_kv_heads * (self.head_dim // 16)
        buf = (ctypes.c_uint8 * n).from_address(lib().oracle_pool_block_scales(self._h))
        return np.frombuffer(buf, dtype=np.uint8).reshape(
            self.num_blocks, 2, self.block_size, self.n_kv_heads, self.head_dim // 16)

    def set_scales(self, k_scale, v_scale) -> None:
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        rc = lib().oracle_pool_set_scales(self._h, _ptr(ks), _ptr(vs))
        if rc != OK:
            raise ValueError(f"oracle_pool_set_scales: {rc}")

    def write(self, k, v, slot_mapping) -> None:
        """Paged KV write: k, v are [T, Hkv, D] bf16; slot < 0 skips the token."""
        k, v = _u16(k), _u16(v)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        T = slots.shape[0]
        assert k.shape == (T, self.n_kv_heads, self.head_dim) and v.shape == k.shape
        rc = lib().oracle_kv_write(self._h, _ptr(k), _ptr(v), _ptr(slots), T)
        if rc != OK:
            raise ValueError(f"oracle_kv_write: {rc}")

    def copy_blocks(self, pairs) -> None:
        """Copy block src to block dst for each (src, dst) row of `pairs`, in order."""
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        rc = lib().oracle_pool_copy_blocks(self._h, _ptr(pr), pr.shape[0])
        if rc != OK:
            raise ValueError(f"oracle_pool_copy_blocks: {rc}")

    def decode(self, q, block_tables, context_lens, scale: float, window: int = 0,
               seqs=None) -> np.ndarray:
        """fp64 paged decode attention; returns float32 [B, Hq, D] (rows outside `seqs` zero)."""
        q = _u16(q)
        B, Hq, D = q.shape
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        assert tables.shape[0] == B and lens.shape == (B,) and D == self.head_dim
        out = np.zeros((B, Hq, D), dtype=np.float32)
        sel = None if seqs is None else np.ascontiguousarray(seqs, dtype=np.int32)
        rc = lib().oracle_paged_decode(self._h, _ptr(q), Hq, _ptr(tables), tables.shape[1],
                                       _ptr(lens), B, float(scale), int(window), _ptr(sel),
                                       0 if sel is None else sel.shape[0], _ptr(out))
        if rc != OK:
            raise ValueError(f"oracle_paged_decode: {rc}")
        return out

    def prefill(self, q, cu_q_lens, block_tables, context_lens, scale: float,
                window: int = 0) -> np.ndarray:
        """fp64 paged prefill attention; q [T, Hq, D] bf16 -> float32 [T, Hq, D]."""
        q = _u16(q)
        T, Hq, D = q.shape
        cu = np.ascontiguousarray(cu_q_lens, dtype=np.int32)
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        B = lens.shape[0]
        assert cu.shape == (B + 1,) and cu[-1] == T and tables.shape[0] == B and D == self.head_dim
        out = np.zeros((T, Hq, D), dtype=np.float32)
        rc = lib().oracle_paged_prefill(self._h, _ptr(q), Hq, _ptr(cu), _ptr(tables), tables.shape[1],
                                        _ptr(lens), B, float(scale), int(window), _ptr(out))
        if rc != OK:
            raise ValueError(f"oracle_paged_prefill: {rc}")
        return out


def sha256(data: bytes) -> bytes:
    buf = np.frombuffer(bytes(data), dtype=np.uint8) if data else np.zeros(1, np.uint8)
    out = np.zeros(32, dtype=np.uint8)
    lib().oracle_sha256(_ptr(buf), len(data), _ptr(out))
    return out.tobytes()


# --------------------------------------------------------------- allocator --

class Allocator:
    """Host block pool bookkeeping (free queue, ref_cnt, hash map, preemption)."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self._h = lib().oracle_alloc_create(self.num_blocks, self.block_size)
        if not self._h:
            raise ValueError("oracle_alloc_create rejected its arguments")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.oracle_alloc_destroy(h)

    def admit(self, req_id: int, num_tokens: int | None = None, tokens=None,
              salt: bytes = b"", extra: bytes = b"") -> tuple[int, int]:
        """Returns (status, cached_tokens)."""
        toks = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        n = int(num_tokens if toks is None else toks.shape[0])
        sb = np.frombuffer(salt, np.uint8) if salt else None
        eb = np.frombuffer(extra, np.uint8) if extra else None
        cached = ctypes.c_int64(0)
        rc = lib().oracle_alloc_admit(self._h, int(req_id), _ptr(toks), n, _ptr(sb), len(salt),
                                      _ptr(eb), len(extra), ctypes.byref(cached))
        return rc, cached.value

    def append(self, req_id: int, n: int | None = None, tokens=None) -> int:
        toks = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        cnt = int(n if toks is None else toks.shape[0])
        return lib().oracle_alloc_append(self._h, int(req_id), _ptr(toks), cnt)

    def free(self, req_id: int) -> int:
        return lib().oracle_alloc_free(self._h, int(req_id))

    def fork(self, parent: int, child: int) -> int:
        return lib().oracle_alloc_fork(self._h, int(parent), int(child))

    def copies(self, take: bool = True) -> list[tuple[int, int]]:
        """Pending copy-on-write pairs (src, dst), oldest first (cleared when take)."""
        n = lib().oracle_alloc_copies(self._h, None, 0, 0)
        out = np.zeros((max(n, 1), 2), np.int32)
        lib().oracle_alloc_copies(self._h, _ptr(out), n, 1 if take else 0)
        return [(int(a), int(b)) for a, b in out[:n]]

    def preempt_newest(self) -> tuple[int, int]:
        rid = ctypes.c_int64(-1)
        rc = lib().oracle_alloc_preempt_newest(self._h, ctypes.byref(rid))
        return rc, rid.value

    def table(self, req_id: int) -> list[int]:
        n = ctypes.c_int64(0)
        rc = lib().oracle_alloc_table(self._h, int(req_id), None, 0, ctypes.byref(n))
        if rc != OK:
            raise KeyError(req_id)
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        lib().oracle_alloc_table(self._h, int(req_id), _ptr(out), n.value, ctypes.byref(n))
        return out[: n.value].tolist()

    def num_tokens(self, req_id: int) -> int:
        return int(lib().oracle_alloc_num_tokens(self._h, int(req_id)))

    def num_free(self) -> int:
        return int(lib().oracle_alloc_num_free(self._h))

    def free_queue(self) -> list[int]:
        n = lib().oracle_alloc_free_queue(self._h, None, 0)
        out = np.zeros(max(n, 1), dtype=np.int32)
        lib().oracle_alloc_free_queue(self._h, _ptr(out), n)
        return out[:n].tolist()

    def block(self, block_id: int) -> tuple[int, bytes | None]:
        """(ref_cnt, hash or None)."""
        ref = ctypes.c_int32(0)
        has = ctypes.c_int32(0)
        h = np.zeros(32, np.uint8)
        rc = lib().oracle_alloc_block_info(self._h, int(block_id), ctypes.byref(ref),
                                           ctypes.byref(has), _ptr(h))
        if rc != OK:
            raise IndexError(block_id)
        return ref.value, (h.tobytes() if has.value else None)

    def lookup(self, h: bytes) -> int:
        buf = np.frombuffer(bytes(h), np.uint8)
        return int(lib().oracle_alloc_lookup(self._h, _ptr(buf)))

    def map_entries(self) -> dict[bytes, int]:
        n = lib().oracle_alloc_map_size(self._h)
        hs = np.zeros((max(n, 1), 32), np.uint8)
        ids = np.zeros(max(n, 1), np.int32)
        lib().oracle_alloc_map_entries(self._h, _ptr(hs), _ptr(ids), n)
        return {hs[i].tobytes(): int(ids[i]) for i in range(n)}

    def stats(self) -> dict[str, int]:
        out = np.zeros(5, np.int64)
        lib().oracle_alloc_stats(self._h, _ptr(out))
        return dict(zip(["queries", "hits", "evictions", "preemptions", "running"],
                        out.tolist()))
