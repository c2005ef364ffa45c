"""Shared GPU-vs-oracle parity harness for the -m gpu tests.

Both sides receive the same seeded inputs from the workload generator: the
CUDA path through the C ABI (via the ctypes binding), the oracle through its
own write into its own pool.  Nothing the oracle sees comes from the GPU.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv
from paged_kv_cache_33_gb300.workloads import Workload

BF16_MAX_ABS = 2e-3   # acceptance for bf16 KV: max |err|
BF16_REL_L2 = 1e-3    # and relative L2
FP8_MAX_ABS = 3e-2    # acceptance for FP8 KV
# FP4 KV: the keys and values are dequantised exactly (f16), the queries are
# exact in f16 after a power-of-two scaling, scores accumulate in fp32; the
# softmax weights enter the P V product as f16 (relative rounding <= 2^-11),
# so against the oracle on the same codes the error is below the bf16 bar.
FP4_MAX_ABS = BF16_MAX_ABS
FP4_REL_L2 = BF16_REL_L2


def poison(pool: pagedkv.KVPool) -> None:
    """Fill the whole pool with NaN codes so any read of an unwritten slot shows."""
    v = pool.view()
    if pool.dtype == "bf16":
        v.view(torch.int16).fill_(0x7FC0)
    elif pool.dtype == "fp4":
        v.fill_(0xFF)          # codes -6 under NaN (0xFF) block scales
    else:
        v.fill_(0x7F)


def make_gpu_pool(w: Workload, poison_pool: bool = True) -> pagedkv.KVPool:
    pool = pagedkv.KVPool(w.num_blocks, w.block_size, w.n_kv_heads, w.head_dim, w.dtype)
    if poison_pool:
        poison(pool)
    if w.dtype in ("fp8", "fp4"):
        pool.set_scales(torch.from_numpy(w.k_scale).cuda(), torch.from_numpy(w.v_scale).cuda())
    return pool


def make_oracle_pool(w: Workload) -> oracle.Pool:
    op = oracle.Pool(w.num_blocks, w.block_size, w.n_kv_heads, w.head_dim, w.dtype)
    if w.dtype in ("fp8", "fp4"):
        op.set_scales(w.k_scale, w.v_scale)
    return op


def fill_both(w: Workload, pool: pagedkv.KVPool, opool: oracle.Pool | None, seqs=None,
              device_fill_rest: bool = False):
    """Write the cache (setup) then this step's tokens to both pools.

    With `seqs`, only those sequences (and any shared prefix) are generated on
    the CPU and given to both sides; with device_fill_rest the other
    sequences are filled on the GPU alone from device-generated data so the
    kernel runs the full workload."""
    if device_fill_rest and seqs is not None:
        d_setup, (dk, dv, ds) = w.fill_plan(device="cuda")
        for k, v, s in d_setup:
            pagedkv.paged_kv_write(pool, k, v, s.cuda())
        pagedkv.paged_kv_write(pool, dk, dv, ds.cuda())
    setup, (k_new, v_new, s_new) = w.fill_plan(seqs=seqs)
    if seqs is not None:
        keep = torch.zeros(w.batch, dtype=torch.bool)
        keep[list(seqs)] = True
        s_new = torch.where(keep, s_new, torch.full_like(s_new, -1))
    for k, v, s in setup:
        pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), s.cuda())
        if opool is not None:
            opool.write(k, v, s.numpy())
    pagedkv.paged_kv_write(pool, k_new.cuda(), v_new.cuda(), s_new.cuda())
    if opool is not None:
        opool.write(k_new, v_new, s_new.numpy())
    return setup, (k_new, v_new, s_new)


def written_slots(setup, step) -> np.ndarray:
    parts = [s.numpy() for _, _, s in setup] + [step[2].numpy()]
    s = np.concatenate(parts) if parts else np.zeros(0, np.int64)
    return s[s >= 0]


def compare_pools(pool: pagedkv.KVPool, opool: oracle.Pool, slots: np.ndarray,
                  max_rows: int = 200_000) -> None:
    """Bit-exact comparison of the K/V rows at `slots` (GPU layout vs the pages' layout)."""
    if len(slots) > max_rows:
        slots = np.random.default_rng(0).choice(slots, max_rows, replace=False)
    bs = pool.block_size
    assert opool.block_size == bs
    assert len(slots) == 0 or (slots.min() >= 0 and slots.max() < pool.num_blocks * bs)
    blk = torch.from_numpy(slots // bs)
    off = torch.from_numpy(slots % bs)
    if pool.dtype == "fp4":
        codes, scales = pool.fp4_rows()                # [NB, Hkv, 2, BS, D], [.., D/16]
        for gpu, ora in ((codes, opool.array()), (scales, opool.block_scales())):
            g = gpu[blk.cuda(), :, :, off.cuda(), :].permute(0, 2, 1, 3).cpu().numpy()
            o = ora[slots // bs, :, slots % bs]
            bad = np.nonzero((g != o).reshape(len(slots), -1).any(axis=1))[0]
            assert bad.size == 0, f"{bad.size} FP4 rows differ, first slot {slots[bad[0]]}"
        return
    v = pool.rows()
    g = v[blk.cuda(), :, :, off.cuda(), :]            # [n, Hkv, 2, D]
    g = g.permute(0, 2, 1, 3).contiguous().cpu()       # [n, 2, Hkv, D]
    if pool.dtype == "bf16":
        g = g.view(torch.int16).numpy().view(np.uint16)
    else:
        g = g.numpy()
    arr = opool.array()                                # [NB, 2, BS, Hkv, D]
    o = arr[slots // bs, :, slots % bs]                # [n, 2, Hkv, D]
    bad = np.nonzero((g != o).reshape(len(slots), -1).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first slot {slots[bad[0]]}"


def errors(out: np.ndarray, ref: np.ndarray) -> tuple[float, float]:
    diff = out.astype(np.float64) - ref.astype(np.float64)
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref.astype(np.float64)))
    rel = float(np.linalg.norm(diff)) / den if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(w: Workload, out: np.ndarray, ref: np.ndarray, label: str = "") -> tuple:
    assert np.isfinite(out).all(), f"{label}: non-finite output"
    max_abs, rel = errors(out, ref)
    if w.dtype == "bf16":
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, (label, max_abs, rel)
    elif w.dtype == "fp4":
        assert max_abs <= FP4_MAX_ABS and rel <= FP4_REL_L2, (label, max_abs, rel)
    else:
        assert max_abs <= FP8_MAX_ABS, (label, max_abs, rel)
    return max_abs, rel


def decode_gpu(w: Workload, pool: pagedkv.KVPool, q: torch.Tensor, tables=None, lens=None,
               window=None, max_context_len=None) -> torch.Tensor:
    tables = torch.from_numpy(w.block_tables if tables is None else tables).cuda()
    lens = torch.from_numpy(w.context_lens if lens is None else lens).cuda()
    return pagedkv.paged_decode_attention(
        pool, q.cuda(), tables, lens, w.scale, w.window if window is None else window,
        max_context_len=w.max_context_len if max_context_len is None else max_context_len)


def run_parity(w: Workload, seqs=None, part_blocks: int | None = None,
               device_fill_rest: bool = False, check_pool: bool = True) -> dict:
    pool = make_gpu_pool(w)
    if part_blocks:
        pool.set_partition_blocks(part_blocks)
    opool = make_oracle_pool(w)
    setup, step = fill_both(w, pool, opool, seqs=seqs, device_fill_rest=device_fill_rest)
    q = w.query()
    out = decode_gpu(w, pool, q)
    torch.cuda.synchronize()
    status = pool.check_status()
    assert status == pagedkv.KV_OK, pagedkv.STATUS.get(status)
    if check_pool:
        compare_pools(pool, opool, written_slots(setup, step))
    ref = opool.decode(q, w.block_tables, w.context_lens, w.scale, w.window, seqs=seqs)
    rows = list(range(w.batch)) if seqs is None else list(seqs)
    got = out.cpu().numpy()[rows]
    max_abs, rel = assert_close(w, got, ref[rows], f"{w.name}/{w.size}")
    print(f"PARITY {w.name}/{w.size} bs={w.block_size} seqs={len(rows)} part_blocks={part_blocks} "
          f"max_abs={max_abs:.3e} rel_l2={rel:.3e}")
    pool.destroy()
    return {"max_abs": max_abs, "rel_l2": rel}
