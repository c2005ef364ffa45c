"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument checks answer without touching a GPU."""

import ctypes
import os
import re

import pytest
import torch

from paged_kv_cache_33_gb300 import pagedkv

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions() -> list[str]:
    """Every function declared in include/*.h (return type at line start)."""
    names = []
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = open(os.path.join(INCLUDE, h)).read()
            names += re.findall(r"^(?:kv_status|size_t|int64_t|int32_t|const char\*)\s+(\w+)\(",
                                text, re.M)
    return names


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("kv_pool_create", "paged_kv_write", "paged_decode_attention",
              "paged_decode_step", "kv_pool_check_status", "kv_status_str",
              "kv_bm_create", "kv_bm_admit", "kv_bm_append", "kv_bm_fork",
              "kv_bm_take_copies", "kv_bm_decode_inputs"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = pagedkv.load()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings():
    assert pagedkv.kv_status_str(0) == "KV_OK"
    assert pagedkv.kv_status_str(5) == "KV_ERR_BAD_BLOCK_ID"
    assert pagedkv.kv_status_str(99) == "KV_ERR_UNKNOWN"
    for code, name in pagedkv.STATUS.items():
        assert pagedkv.kv_status_str(code) == name


@pytest.mark.parametrize("args,status", [
    ((0, 16, 8, 128, 0), 1),        # no blocks
    ((10, 0, 8, 128, 0), 1),        # no block size
    ((10, 16, 0, 128, 0), 1),       # no heads
    ((10, 16, 8, 128, 7), 1),       # unknown dtype
    ((10, 64, 8, 128, 0), 4),       # block size other than 16 or 32
    ((10, 16, 8, 96, 0), 4),        # head_dim not 64/128
    ((10, 16, 8, 64, 1), 4),        # FP8 needs head_dim 128
    ((10, 16, 8, 64, 2), 4),        # FP4 needs head_dim 128
])
def test_create_rejects_bad_shapes_before_any_cuda_call(args, status):
    L = pagedkv.load()
    h = ctypes.c_void_p()
    assert L.kv_pool_create(*args, ctypes.byref(h)) == status
    assert not h.value


def test_null_handles_are_rejected():
    L = pagedkv.load()
    assert L.kv_pool_destroy(None) == 1
    assert L.paged_kv_write(None, None, None, None, 1, None) == 1
    assert L.paged_decode_attention(None, None, 8, None, 4, None, 1, 64, 1.0, 0, None, None, 0,
                                    None) == 1
    assert L.paged_decode_step(None, None, None, None, 1, None, 8, None, 4, None, 1, 64, 1.0, 0,
                               None, None, 0, None) == 1
    assert L.paged_decode_workspace_bytes(None, 1, 8, 64, 0) == 0
    assert L.kv_pool_check_status(None, None) == 1
    assert L.kv_pool_set_partition_blocks(None, 8) == 1
    assert L.kv_pool_set_wait_limit(None, 1000000) == 1
    assert L.kv_pool_set_test_stall(None, 1) == 1
    assert L.kv_pool_refresh_exponent_map(None, None) == 1
    ptr, n = ctypes.c_void_p(), ctypes.c_int64()
    assert L.kv_pool_exponent_map(None, ctypes.byref(ptr), ctypes.byref(n)) == 1


def test_create_without_a_device_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    L = pagedkv.load()
    h = ctypes.c_void_p()
    assert L.kv_pool_create(10, 16, 8, 128, 0, ctypes.byref(h)) in (2, 3)
    assert not h.value


class _FakePool:
    """Only the sizes the bindings check before any call into the library."""
    n_kv_heads, head_dim = 2, 128


def _decode_args(B=3, Hq=8, D=128, mbs=4):
    return (torch.zeros(B, Hq, D, dtype=torch.bfloat16), torch.zeros(B, mbs, dtype=torch.int32),
            torch.ones(B, dtype=torch.int32), torch.zeros(B, Hq, D))


@pytest.mark.parametrize("bad", ["head_dim", "lens_short", "lens_2d", "tables", "out_small",
                                 "q_2d"])
@pytest.mark.parametrize("entry", ["attention", "step", "noalloc"])
def test_decode_bindings_check_the_sizes_the_abi_cannot_see(entry, bad):
    q, tables, lens, out = _decode_args()
    if bad == "head_dim":
        q = torch.zeros(3, 8, 64, dtype=torch.bfloat16)
    elif bad == "lens_short":
        lens = lens[:2]
    elif bad == "lens_2d":
        lens = lens.view(3, 1)
    elif bad == "tables":
        tables = tables[:2]
    elif bad == "out_small":
        out = out[:, :4]
    elif bad == "q_2d":
        q = q[0]
    pool = _FakePool()
    with pytest.raises(ValueError):
        if entry == "attention":
            pagedkv.paged_decode_attention(pool, q, tables, lens, 0.1, out=out, max_context_len=16)
        elif entry == "noalloc":
            pagedkv.paged_decode_attention_noalloc(pool, q, tables, lens, 0.1, 0, 16, out)
        else:
            kv = torch.zeros(3, 2, 128, dtype=torch.bfloat16)
            pagedkv.paged_decode_step(pool, kv, kv, torch.zeros(3, dtype=torch.int64), q, tables,
                                      lens, 0.1, out=out, max_context_len=16)


def test_noalloc_binding_requires_out():
    q, tables, lens, _ = _decode_args()
    with pytest.raises(ValueError):
        pagedkv.paged_decode_attention_noalloc(_FakePool(), q, tables, lens, 0.1, 0, 16, None)


def test_drain_timeout_status_is_named():
    assert pagedkv.STATUS[9] == "KV_ERR_DRAIN_TIMEOUT"
    assert pagedkv.kv_status_str(9) == "KV_ERR_DRAIN_TIMEOUT"


def test_stale_exponent_map_status_is_named():
    assert pagedkv.STATUS[10] == "KV_ERR_STALE_EXPONENT_MAP"
    assert pagedkv.kv_status_str(10) == "KV_ERR_STALE_EXPONENT_MAP"


def test_decode_bindings_marshal_their_arguments(monkeypatch):
    # The library replaced by a recorder (no GPU here): each binding must
    # pass the sizes taken from the tensors, in the C ABI's order.
    calls = {}

    class _Lib:
        def __getattr__(self, name):
            def f(*args):
                calls[name] = args
                return 0
            return f

    monkeypatch.setattr(pagedkv, "load", lambda: _Lib())
    monkeypatch.setattr(pagedkv, "_dev", lambda t, dtype, name: (name, tuple(t.shape)))
    monkeypatch.setattr(pagedkv, "_in", lambda t, dtype, name: (name, tuple(t.shape)))
    monkeypatch.setattr(pagedkv, "_out", lambda t, name: (name, tuple(t.shape)))
    monkeypatch.setattr(pagedkv, "_stream", lambda s: "stream")
    pool = _FakePool()
    pool.handle = "pool"
    q, tables, lens, out = _decode_args(B=3, Hq=8, mbs=4)
    pagedkv.paged_decode_attention_noalloc(pool, q, tables, lens, 0.5, 7, 16, out)
    assert calls["paged_decode_attention_noalloc"] == (
        "pool", ("q", (3, 8, 128)), 8, ("block_tables", (3, 4)), 4, ("context_lens", (3,)), 3, 16,
        0.5, 7, ("out", (3, 8, 128)), "stream")
    monkeypatch.setattr(pagedkv, "paged_decode_workspace_bytes", lambda *a: 0)
    pagedkv.paged_decode_attention(pool, q, tables, lens, 0.5, 7, max_context_len=16, out=out)
    args = calls["paged_decode_attention"]
    assert args[:10] == ("pool", ("q", (3, 8, 128)), 8, ("block_tables", (3, 4)), 4,
                         ("context_lens", (3,)), 3, 16, 0.5, 7)


def test_inputs_must_be_device_or_pinned_host_tensors():
    # a pageable host tensor cannot be read by the kernels in place
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(TypeError, match="pinned"):
        pagedkv._in(t, torch.int32, "context_lens")
