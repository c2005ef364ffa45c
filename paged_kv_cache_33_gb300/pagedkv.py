"""ctypes binding of libpagedkv.so (include/pagedkv.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; this module checks
tensor dtypes/devices, passes raw device pointers and the current torch
stream, and raises KVError on a non-OK status.  There is no CPU fallback: if
the library is missing or cannot load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

import torch

from . import build as _build

KV_OK = 0
STATUS = {0: "KV_OK", 1: "KV_ERR_INVALID_ARG", 2: "KV_ERR_OOM", 3: "KV_ERR_CUDA",
          4: "KV_ERR_UNSUPPORTED", 5: "KV_ERR_BAD_BLOCK_ID", 6: "KV_ERR_TIMEOUT",
          7: "KV_ERR_BAD_SLOT", 8: "KV_ERR_BAD_CONTEXT", 9: "KV_ERR_DRAIN_TIMEOUT",
          10: "KV_ERR_STALE_EXPONENT_MAP"}
DTYPES = {"bf16": 0, "fp8": 1, "fp4": 2}
FP4_RECORD_BYTES = 2304  # one 16-token sub-tile of a (block, KV head) in an FP4 pool

LIB_PATH = _build.LIB_PATH


class KVError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class _Desc(ctypes.Structure):
    _fields_ = [("base_dev", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
                ("block_size", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("strides", ctypes.c_int64 * 5), ("bytes", ctypes.c_uint64),
                ("device", ctypes.c_int32), ("scales_dev", ctypes.c_void_p),
                ("v_layout", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    """Load libpagedkv.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if _build.stale():
            _build.build()
        L = ctypes.CDLL(LIB_PATH)
        c, P = ctypes, ctypes.c_void_p
        sig = {
            "kv_pool_create": (c.c_int, [c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int,
                                         c.POINTER(P)]),
            "kv_pool_destroy": (c.c_int, [P]),
            "kv_pool_info": (c.c_int, [P, c.POINTER(_Desc)]),
            "kv_pool_exponent_map": (c.c_int, [P, c.POINTER(P), c.POINTER(c.c_int64)]),
            "kv_pool_refresh_exponent_map": (c.c_int, [P, P]),
            "kv_pool_set_scales": (c.c_int, [P, P, P, P]),
            "paged_kv_write": (c.c_int, [P, P, P, P, c.c_int64, P]),
            "paged_kv_copy_blocks": (c.c_int, [P, P, c.c_int64, P]),
            "paged_decode_workspace_bytes": (c.c_size_t, [P, c.c_int32, c.c_int32, c.c_int32,
                                                          c.c_int32]),
            "paged_decode_attention": (c.c_int, [P, P, c.c_int32, P, c.c_int32, P, c.c_int32,
                                                 c.c_int32, c.c_float, c.c_int32, P, P,
                                                 c.c_size_t, P]),
            "paged_decode_step": (c.c_int, [P, P, P, P, c.c_int64, P, c.c_int32, P, c.c_int32,
                                            P, c.c_int32, c.c_int32, c.c_float, c.c_int32, P,
                                            P, c.c_size_t, P]),
            "paged_prefill_attention": (c.c_int, [P, P, c.c_int32, P, P, c.c_int32, P,
                                                  c.c_int32, c.c_int32, c.c_int32, c.c_float,
                                                  c.c_int32, P, P]),
            "paged_decode_attention_noalloc": (c.c_int, [P, P, c.c_int32, P, c.c_int32, P,
                                                         c.c_int32, c.c_int32, c.c_float,
                                                         c.c_int32, P, P]),
            "kv_pool_set_partition_blocks": (c.c_int, [P, c.c_int32]),
            "kv_pool_set_timing_events": (c.c_int, [P, P, P]),
            "kv_pool_set_wait_limit": (c.c_int, [P, c.c_uint64]),
            "kv_pool_set_test_stall": (c.c_int, [P, c.c_int32]),
            "kv_pool_check_status": (c.c_int, [P, P]),
            "kv_status_str": (c.c_char_p, [c.c_int]),
            "kv_bm_create": (c.c_int, [c.c_int64, c.c_int32, c.POINTER(P)]),
            "kv_bm_destroy": (c.c_int, [P]),
            "kv_bm_admit": (c.c_int, [P, c.c_int64, P, c.c_int64, P, c.c_int32, P, c.c_int32,
                                      P]),
            "kv_bm_append": (c.c_int, [P, c.c_int64, P, c.c_int64]),
            "kv_bm_fork": (c.c_int, [P, c.c_int64, c.c_int64]),
            "kv_bm_free": (c.c_int, [P, c.c_int64]),
            "kv_bm_preempt_newest": (c.c_int, [P, P]),
            "kv_bm_take_copies": (c.c_int64, [P, P, c.c_int64]),
            "kv_bm_pending_copies": (c.c_int64, [P, P, c.c_int64]),
            "kv_bm_block_table": (c.c_int, [P, c.c_int64, P, c.c_int64, P]),
            "kv_bm_slot_mapping": (c.c_int, [P, c.c_int64, c.c_int64, c.c_int64, P]),
            "kv_bm_decode_inputs": (c.c_int, [P, P, c.c_int32, c.c_int32, P, P, P]),
            "kv_bm_num_tokens": (c.c_int64, [P, c.c_int64]),
            "kv_bm_num_free": (c.c_int64, [P]),
            "kv_bm_free_queue": (c.c_int64, [P, P, c.c_int64]),
            "kv_bm_block_info": (c.c_int, [P, c.c_int32, P, P, P]),
            "kv_bm_lookup": (c.c_int32, [P, P]),
            "kv_bm_map_entries": (c.c_int64, [P, P, P, c.c_int64]),
            "kv_bm_get_stats": (c.c_int, [P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
        return L


def _check(rc: int, where: str) -> None:
    if rc != KV_OK:
        raise KVError(rc, where)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _in(t: torch.Tensor, dtype: torch.dtype, name: str) -> ctypes.c_void_p:
    """A per-step input: a CUDA tensor, or a pinned host tensor, which the
    kernels read in place (mapped host memory; no host-to-device copy)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise TypeError(f"{name} must be a CUDA tensor or a pinned host tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return ctypes.c_void_p(t.data_ptr())
    return _dev(t, dtype, name)


def _out(t: torch.Tensor, name: str) -> ctypes.c_void_p:
    """An fp32 result buffer: a CUDA tensor, or a pinned host tensor, which
    the kernels write directly (mapped host memory; no device-to-host copy)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise TypeError(f"{name} must be a CUDA tensor or a pinned host tensor")
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError(f"{name} must be contiguous float32")
        return ctypes.c_void_p(t.data_ptr())
    return _dev(t, torch.float32, name)


class KVPool:
    """One layer's block pool on the current CUDA device (owns its memory)."""

    def __init__(self, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                 dtype: str = "bf16"):
        L = load()
        h = ctypes.c_void_p()
        _check(L.kv_pool_create(int(num_blocks), int(block_size), int(n_kv_heads),
                                int(head_dim), DTYPES[dtype], ctypes.byref(h)), "kv_pool_create")
        self._h = h
        self.device = torch.device("cuda", torch.cuda.current_device())  # the pool's GPU
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.n_kv_heads, self.head_dim, self.dtype = int(n_kv_heads), int(head_dim), dtype
        self._events = None

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise RuntimeError("pool destroyed")
        return self._h

    def destroy(self) -> None:
        if getattr(self, "_h", None) is not None and _lib is not None:
            _check(_lib.kv_pool_destroy(self._h), "kv_pool_destroy")
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def info(self) -> dict:
        d = _Desc()
        _check(load().kv_pool_info(self.handle, ctypes.byref(d)), "kv_pool_info")
        return {"base_dev": d.base_dev, "num_blocks": d.num_blocks, "block_size": d.block_size,
                "n_kv_heads": d.n_kv_heads, "head_dim": d.head_dim, "dtype": d.dtype,
                "strides": list(d.strides), "bytes": d.bytes, "device": d.device,
                "scales_dev": d.scales_dev, "v_layout": d.v_layout}

    def view(self) -> torch.Tensor:
        """The pool memory as a torch tensor, no copy: [NB, Hkv, 2, BS, D] (bf16 or
        uint8), or for FP4 pools the raw records [NB, Hkv, BS/16, 2304] uint8."""
        i = self.info()
        tdt, typestr = (torch.bfloat16, "<V2") if self.dtype == "bf16" else (torch.uint8, "|u1")
        shape = (self.num_blocks, self.n_kv_heads, 2, self.block_size, self.head_dim)
        if self.dtype == "fp4":
            shape = (self.num_blocks, self.n_kv_heads, self.block_size // 16, FP4_RECORD_BYTES)

        class _Buf:
            __cuda_array_interface__ = {"shape": shape, "typestr": "|u1" if tdt == torch.uint8
                                        else "<i2", "data": (i["base_dev"], False),
                                        "version": 3, "strides": None}
        t = torch.as_tensor(_Buf(), device=f"cuda:{i['device']}")
        return t.view(tdt) if tdt == torch.bfloat16 else t

    def exponent_map(self) -> torch.Tensor | None:
        """bf16 pools: the V exponent map as a uint8 tensor view
        [NB, Hkv, BS] (no copy); None for FP8 and FP4 pools."""
        ptr, n = ctypes.c_void_p(), ctypes.c_int64()
        _check(load().kv_pool_exponent_map(self.handle, ctypes.byref(ptr), ctypes.byref(n)),
               "kv_pool_exponent_map")
        if not ptr.value:
            return None
        shape = (self.num_blocks, self.n_kv_heads, self.block_size)

        class _Buf:
            __cuda_array_interface__ = {"shape": shape, "typestr": "|u1", "data": (ptr.value, False),
                                        "version": 3, "strides": None}
        return torch.as_tensor(_Buf(), device=f"cuda:{self.info()['device']}")

    def refresh_exponent_map(self, stream=None) -> None:
        """Recompute the V exponent map from the pool (after writing V through view())."""
        _check(load().kv_pool_refresh_exponent_map(self.handle, _stream(stream)),
               "kv_pool_refresh_exponent_map")

    def rows(self) -> torch.Tensor:
        """Inspection: the pool as [NB, Hkv, 2, BS, D] with every V tile in
        token-row order.  The raw view itself for row-major pools; a copy with
        the transposed V tiles turned back for pools that store them so; for
        FP4 pools the E2M1 code of every element (see fp4_rows)."""
        if self.dtype == "fp4":
            return self.fp4_rows()[0]
        raw = self.view()
        if self.info()["v_layout"] == 0:
            return raw
        bs, d = self.block_size, self.head_dim
        pos = torch.tensor([4 * ((t % 8) // 2) + t % 2 + 2 * (t // 8) for t in range(16)],
                           device=raw.device)
        # each V tile: bs/16 sub-tiles of [D][16] codes
        vt = raw[:, :, 1].reshape(self.num_blocks, self.n_kv_heads, bs // 16, d, 16)
        rows = vt[..., pos].transpose(3, 4)            # [NB, Hkv, sub, 16, D]
        out = raw.clone()
        out[:, :, 1] = rows.reshape(self.num_blocks, self.n_kv_heads, bs, d)
        return out

    def fp4_rows(self) -> tuple[torch.Tensor, torch.Tensor]:
        """Inspection of an FP4 pool: (codes [NB, Hkv, 2, BS, D], block scales
        [NB, Hkv, 2, BS, D/16]) as uint8, gathered from the records with the
        byte offsets include/pagedkv.h documents."""
        assert self.dtype == "fp4" and self.head_dim == 128
        rec = self.view()                                   # [NB, Hkv, S, 2304]
        byte, shift, sbyte = _fp4_maps(rec.device)
        NB, H, S = rec.shape[:3]
        codes = (rec[..., byte] >> shift) & 0xF             # [NB, H, S, 2, 16, 128]
        scales = rec[..., sbyte]                            # [NB, H, S, 2, 16, 8]
        codes = codes.permute(0, 1, 3, 2, 4, 5).reshape(NB, H, 2, S * 16, 128)
        scales = scales.permute(0, 1, 3, 2, 4, 5).reshape(NB, H, 2, S * 16, 8)
        return codes, scales

    def set_scales(self, k_scale: torch.Tensor, v_scale: torch.Tensor, stream=None) -> None:
        _check(load().kv_pool_set_scales(self.handle, _dev(k_scale, torch.float32, "k_scale"),
                                         _dev(v_scale, torch.float32, "v_scale"),
                                         _stream(stream)), "kv_pool_set_scales")

    def set_partition_blocks(self, n: int) -> None:
        _check(load().kv_pool_set_partition_blocks(self.handle, int(n)),
               "kv_pool_set_partition_blocks")

    def set_timing_events(self, start, stop) -> None:
        """Record CUDA events around each decode kernel (None, None disables)."""
        if start is None:
            _check(load().kv_pool_set_timing_events(self.handle, None, None), "timing")
            self._events = None
            return
        fresh = [ev for ev in (start, stop) if ev.cuda_event == 0]
        for ev in fresh:
            ev.record()   # torch creates the event lazily, on first record
        if fresh:
            torch.cuda.synchronize()
        _check(load().kv_pool_set_timing_events(self.handle, ctypes.c_void_p(start.cuda_event),
                                                ctypes.c_void_p(stop.cuda_event)), "timing")
        self._events = (start, stop)

    def set_wait_limit(self, limit_ns: int) -> None:
        """Bound of every wait in this pool's kernels (ns of wall time)."""
        _check(load().kv_pool_set_wait_limit(self.handle, int(limit_ns)), "kv_pool_set_wait_limit")

    def set_test_stall(self, enable: bool) -> None:
        """Test instrumentation: make one copy's wait run out in each decode."""
        _check(load().kv_pool_set_test_stall(self.handle, 1 if enable else 0),
               "kv_pool_set_test_stall")

    def check_status(self, stream=None) -> int:
        """Read and clear the device error word; returns the status code."""
        return int(load().kv_pool_check_status(self.handle, _stream(stream)))


def _fp4_maps(device):
    """Byte index and nibble shift of every (K/V, token, dim) code of an FP4
    record, and the byte of every (K/V, token, group) scale."""
    byte = torch.zeros(2, 16, 128, dtype=torch.long)
    shift = torch.zeros(2, 16, 128, dtype=torch.uint8)
    sbyte = torch.zeros(2, 16, 8, dtype=torch.long)
    for r in range(16):
        for d in range(128):
            e = d - d % 2
            byte[0, r, d] = ((r // 8) * 512 + 16 * (4 * (r % 8) + (e % 8) // 2) + 2 * (e // 16)
                             + (e % 16) // 8)
            shift[0, r, d] = 4 * (d % 2)
            byte[1, r, d] = (1024 + 16 * (32 * (d // 64) + 4 * (d % 8) + (r % 8) // 2)
                             + 4 * ((d // 16) % 4) + r // 8 + 2 * ((d % 16) // 8))
            shift[1, r, d] = 4 * (r % 2)
        for b in range(8):
            sbyte[0, r, b] = 2048 + 8 * r + b
            sbyte[1, r, b] = 2176 + 32 * ((r % 8) // 2) + 4 * b + r % 2 + 2 * (r // 8)
    return byte.to(device), shift.to(device), sbyte.to(device)


def _check_decode_shapes(pool: KVPool, q: torch.Tensor, block_tables: torch.Tensor,
                         context_lens: torch.Tensor, out: torch.Tensor | None) -> tuple:
    """The sizes the C ABI cannot see: it reads q at the pool's head_dim,
    context_lens and block_tables with the batch of q, and writes out as
    [B, Hq, D].  Raises ValueError on any mismatch; returns (B, Hq, D)."""
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    if D != pool.head_dim:
        raise ValueError(f"q has head_dim {D}, the pool {pool.head_dim}")
    if tuple(context_lens.shape) != (B,):
        raise ValueError(f"context_lens must be [{B}]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [B, max_blocks_per_seq]")
    if out is not None and tuple(out.shape) != (B, Hq, D):
        raise ValueError(f"out must be {(B, Hq, D)}")
    return B, Hq, D


# ----------------------------------------------------- C ABI named functions --

def kv_pool_create(num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                   dtype: str = "bf16") -> KVPool:
    return KVPool(num_blocks, block_size, n_kv_heads, head_dim, dtype)


def kv_pool_destroy(pool: KVPool) -> None:
    pool.destroy()


def kv_pool_set_scales(pool: KVPool, k_scale, v_scale, stream=None) -> None:
    pool.set_scales(k_scale, v_scale, stream)


def kv_pool_check_status(pool: KVPool, stream=None) -> int:
    return pool.check_status(stream)


def paged_kv_write(pool: KVPool, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                   stream=None) -> None:
    """Scatter k, v ([T, Hkv, D] bf16) to the slots in slot_mapping ([T] int64; <0 = skip)."""
    T = slot_mapping.shape[0]
    shape = (T, pool.n_kv_heads, pool.head_dim)
    if tuple(k.shape) != shape or tuple(v.shape) != shape:
        raise ValueError(f"k and v must be {shape}")
    _check(load().paged_kv_write(pool.handle, _in(k, torch.bfloat16, "k"),
                                 _in(v, torch.bfloat16, "v"),
                                 _in(slot_mapping, torch.int64, "slot_mapping"), T,
                                 _stream(stream)), "paged_kv_write")


def paged_kv_copy_blocks(pool: KVPool, pairs, stream=None) -> None:
    """Copy whole blocks src -> dst for each (src, dst) row of `pairs` (host
    data, e.g. BlockManager.copies()), with in-order semantics."""
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    _check(load().paged_kv_copy_blocks(pool.handle, _np_ptr(pr), pr.shape[0], _stream(stream)),
           "paged_kv_copy_blocks")


def paged_decode_workspace_bytes(pool: KVPool, batch: int, n_q_heads: int, max_context_len: int,
                                 sliding_window: int = 0) -> int:
    return int(load().paged_decode_workspace_bytes(pool.handle, int(batch), int(n_q_heads),
                                                   int(max_context_len), int(sliding_window)))


def paged_decode_attention(pool: KVPool, q: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: float, sliding_window: int = 0,
                           max_context_len: int | None = None, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode attention: q [B, Hq, D] bf16 -> out [B, Hq, D] fp32.

    `max_context_len` bounds context_lens (the host side sizes the launch with
    it); when omitted it is read from context_lens, which synchronises.  `out`
    may be a pinned host tensor: the kernels then write the result into host
    memory directly."""
    B, Hq, D = _check_decode_shapes(pool, q, block_tables, context_lens, out)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=pool.device)
    need = paged_decode_workspace_bytes(pool, B, Hq, max_context_len, sliding_window)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=pool.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().paged_decode_attention(
        pool.handle, _in(q, torch.bfloat16, "q"), Hq,
        _in(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _in(context_lens, torch.int32, "context_lens"), B, int(max_context_len), float(scale),
        int(sliding_window), _out(out, "out"), ws_ptr, ws_bytes, _stream(stream)),
        "paged_decode_attention")
    return out


def paged_decode_step(pool: KVPool, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                      q: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                      scale: float, sliding_window: int = 0, max_context_len: int | None = None,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """One decode step: write k, v ([T, Hkv, D] bf16) to `slot_mapping`, then
    attend q [B, Hq, D] over the pool; context_lens already count the new
    tokens.  Returns out [B, Hq, D] fp32 (a CUDA tensor, or the pinned host
    tensor given as `out`, which the kernels write directly)."""
    T = slot_mapping.shape[0]
    shape = (T, pool.n_kv_heads, pool.head_dim)
    if tuple(k.shape) != shape or tuple(v.shape) != shape:
        raise ValueError(f"k and v must be {shape}")
    B, Hq, D = _check_decode_shapes(pool, q, block_tables, context_lens, out)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=pool.device)
    need = paged_decode_workspace_bytes(pool, B, Hq, max_context_len, sliding_window)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=pool.device)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().paged_decode_step(
        pool.handle, _in(k, torch.bfloat16, "k"), _in(v, torch.bfloat16, "v"),
        _in(slot_mapping, torch.int64, "slot_mapping"), T,
        _in(q, torch.bfloat16, "q"), Hq,
        _in(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _in(context_lens, torch.int32, "context_lens"), B, int(max_context_len), float(scale),
        int(sliding_window), _out(out, "out"), ws_ptr, ws_bytes, _stream(stream)),
        "paged_decode_step")
    return out


def paged_prefill_attention(pool: KVPool, q: torch.Tensor, cu_q_lens: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                            sliding_window: int = 0, max_q_len: int | None = None,
                            max_context_len: int | None = None, out: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """Prefill / extend attention: q [T, Hq, D] bf16 (the new tokens of every
    sequence, split by cu_q_lens [B + 1] int32) -> out [T, Hq, D] fp32.  The
    host bounds are read from the tensors (a synchronisation) when omitted."""
    T, Hq, D = q.shape
    B = context_lens.shape[0]
    if max_q_len is None:
        max_q_len = int((cu_q_lens[1:] - cu_q_lens[:-1]).max().item()) if B else 0
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0
    if out is None:
        out = torch.empty(T, Hq, D, dtype=torch.float32, device=q.device)
    if block_tables.dim() != 2 or block_tables.shape[0] != B or cu_q_lens.shape[0] != B + 1:
        raise ValueError("block_tables must be [B, max_blocks_per_seq] and cu_q_lens [B + 1]")
    _check(load().paged_prefill_attention(
        pool.handle, _dev(q, torch.bfloat16, "q"), Hq, _dev(cu_q_lens, torch.int32, "cu_q_lens"),
        _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _dev(context_lens, torch.int32, "context_lens"), B, int(max_q_len),
        int(max_context_len), float(scale), int(sliding_window), _dev(out, torch.float32, "out"),
        _stream(stream)), "paged_prefill_attention")
    return out


def paged_decode_attention_noalloc(pool: KVPool, q: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: float, sliding_window: int,
                                   max_context_len: int, out: torch.Tensor, stream=None) -> None:
    """Decode attention whose split-K scratch is the library's static device
    array: nothing is allocated, so `out` ([B, Hq, D] fp32, a CUDA tensor or
    a pinned host tensor) and `max_context_len` must come from the caller."""
    if out is None:
        raise ValueError("out is required: this entry point allocates nothing")
    B, Hq, _ = _check_decode_shapes(pool, q, block_tables, context_lens, out)
    _check(load().paged_decode_attention_noalloc(
        pool.handle, _in(q, torch.bfloat16, "q"), Hq,
        _in(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
        _in(context_lens, torch.int32, "context_lens"), B, int(max_context_len), float(scale),
        int(sliding_window), _out(out, "out"), _stream(stream)),
        "paged_decode_attention_noalloc")


# ------------------------------------------------------------ block manager --

def _np_ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class BlockManager:
    """Host block manager of one pool (include/kv_block_manager.h).

    Return codes are the C ABI's: 0 ok, 1 bad argument / unknown request,
    2 not enough free blocks (nothing changed)."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        L = load()
        h = ctypes.c_void_p()
        _check(L.kv_bm_create(int(num_blocks), int(block_size), ctypes.byref(h)), "kv_bm_create")
        self.handle, self.num_blocks, self.block_size = h, int(num_blocks), int(block_size)

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib is not None:
            _lib.kv_bm_destroy(h)

    def admit(self, req_id: int, num_tokens: int | None = None, tokens=None,
              salt: bytes = b"", extra: bytes = b"") -> tuple[int, int]:
        """Returns (status, cached_tokens)."""
        toks = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        n = int(num_tokens if toks is None else toks.shape[0])
        sb = np.frombuffer(salt, np.uint8) if salt else None
        eb = np.frombuffer(extra, np.uint8) if extra else None
        cached = ctypes.c_int64(0)
        rc = load().kv_bm_admit(self.handle, int(req_id), _np_ptr(toks), n, _np_ptr(sb),
                                len(salt), _np_ptr(eb), len(extra), ctypes.byref(cached))
        return int(rc), cached.value

    def append(self, req_id: int, n: int | None = None, tokens=None) -> int:
        toks = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        cnt = int(n if toks is None else toks.shape[0])
        return int(load().kv_bm_append(self.handle, int(req_id), _np_ptr(toks), cnt))

    def fork(self, parent: int, child: int) -> int:
        return int(load().kv_bm_fork(self.handle, int(parent), int(child)))

    def free(self, req_id: int) -> int:
        return int(load().kv_bm_free(self.handle, int(req_id)))

    def preempt_newest(self) -> tuple[int, int]:
        rid = ctypes.c_int64(-1)
        rc = load().kv_bm_preempt_newest(self.handle, ctypes.byref(rid))
        return int(rc), rid.value

    def copies(self, take: bool = True) -> list[tuple[int, int]]:
        """Pending copy-on-write pairs (src, dst), oldest first (cleared when take)."""
        L = load()
        n = L.kv_bm_pending_copies(self.handle, None, 0)
        out = np.zeros((max(n, 1), 2), np.int32)
        if take:
            n = L.kv_bm_take_copies(self.handle, _np_ptr(out), n)
        else:
            L.kv_bm_pending_copies(self.handle, _np_ptr(out), n)
        return [(int(a), int(b)) for a, b in out[:n]]

    def table(self, req_id: int) -> list[int]:
        n = ctypes.c_int64(0)
        L = load()
        if L.kv_bm_block_table(self.handle, int(req_id), None, 0, ctypes.byref(n)) != KV_OK:
            raise KeyError(req_id)
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        L.kv_bm_block_table(self.handle, int(req_id), _np_ptr(out), n.value, ctypes.byref(n))
        return out[: n.value].tolist()

    def slot_mapping(self, req_id: int, first_pos: int, n: int) -> np.ndarray:
        out = np.zeros(max(int(n), 1), dtype=np.int64)
        _check(load().kv_bm_slot_mapping(self.handle, int(req_id), int(first_pos), int(n),
                                         _np_ptr(out)), "kv_bm_slot_mapping")
        return out[: int(n)]

    def decode_inputs(self, req_ids, max_blocks_per_seq: int):
        """(block_tables [B, mbs] int32, context_lens [B] int32, slot_mapping [B] int64)."""
        ids = np.ascontiguousarray(req_ids, dtype=np.int64)
        B = ids.shape[0]
        tables = np.zeros((max(B, 1), int(max_blocks_per_seq)), np.int32)
        lens = np.zeros(max(B, 1), np.int32)
        slots = np.zeros(max(B, 1), np.int64)
        _check(load().kv_bm_decode_inputs(self.handle, _np_ptr(ids), B, int(max_blocks_per_seq),
                                          _np_ptr(tables), _np_ptr(lens), _np_ptr(slots)),
               "kv_bm_decode_inputs")
        return tables[:B], lens[:B], slots[:B]

    def num_tokens(self, req_id: int) -> int:
        return int(load().kv_bm_num_tokens(self.handle, int(req_id)))

    def num_free(self) -> int:
        return int(load().kv_bm_num_free(self.handle))

    def free_queue(self) -> list[int]:
        L = load()
        n = L.kv_bm_free_queue(self.handle, None, 0)
        out = np.zeros(max(n, 1), dtype=np.int32)
        L.kv_bm_free_queue(self.handle, _np_ptr(out), n)
        return out[:n].tolist()

    def block(self, block_id: int) -> tuple[int, bytes | None]:
        """(ref_cnt, hash or None)."""
        ref, has = ctypes.c_int32(0), ctypes.c_int32(0)
        h = np.zeros(32, np.uint8)
        if load().kv_bm_block_info(self.handle, int(block_id), ctypes.byref(ref),
                                   ctypes.byref(has), _np_ptr(h)) != KV_OK:
            raise IndexError(block_id)
        return ref.value, (h.tobytes() if has.value else None)

    def lookup(self, h: bytes) -> int:
        buf = np.frombuffer(bytes(h), np.uint8)
        return int(load().kv_bm_lookup(self.handle, _np_ptr(buf)))

    def map_entries(self) -> dict[bytes, int]:
        L = load()
        n = L.kv_bm_map_entries(self.handle, None, None, 0)
        hs = np.zeros((max(n, 1), 32), np.uint8)
        ids = np.zeros(max(n, 1), np.int32)
        L.kv_bm_map_entries(self.handle, _np_ptr(hs), _np_ptr(ids), n)
        return {hs[i].tobytes(): int(ids[i]) for i in range(n)}

    def stats(self) -> dict[str, int]:
        out = np.zeros(6, np.int64)
        _check(load().kv_bm_get_stats(self.handle, _np_ptr(out)), "kv_bm_get_stats")
        return dict(zip(["queries", "hits", "evictions", "preemptions", "running",
                         "cow_copies"], out.tolist()))


def kv_status_str(status: int) -> str:
    return load().kv_status_str(int(status)).decode()


def library_path() -> str:
    return os.path.abspath(LIB_PATH)
