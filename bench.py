"""Benchmark of the paged decode hot path: one step = paged KV write of this
step's token per sequence + split-K paged decode attention (+ its reduce).

Prints ONE JSON line (rank 0).  `value` is KV-read GB/s: K+V bytes of the
attended tokens (exact context, per layer) of all ranks / the max-over-ranks
time of the timed steps, with every input resident in HBM.  `e2e` is the same
metric through the public API with the step's inputs copied from pinned host
memory and the output read back inside the timed region.  `roofline` gives the
decode kernel alone against the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 8b|70b|sw|tiny]
                  [--configs 70b,sw,fp8,fp4,long,tiny|none] [--impl ours|reference]
                  [--part-blocks P]

The headline workload (--config, default 8b) gives the top-level figures;
every workload named by --configs is then measured the same way (device
steps, decode kernel roofline, cold L2, end to end, clocks) and reported
under "configs", each with the oracle timed on a sample of its sequences
and the sample's error against the oracle.

Under torchrun every rank runs an independent replica on its own GPU (the
path has no exchange step); ranks meet at barriers around the timed region.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV-read GB/s and % of GB300 HBM peak; decode tokens/s/layer"
L2_BYTES = 129 * 1024 * 1024
DESCRIPTIONS = {
    "tiny": "tiny paged decode: 4 seqs ctx {5,16,33,70}, 2 q / 1 KV heads, head_dim 64, "
            "64-block permuted pool, 4-token write",
    "8b": "Llama-3-8B-shaped layer decode: batch 64, 32 q / 8 KV heads, head_dim 128, "
          "ctx U[128,4096], pool 1.2x needed with shuffled ids, "
          "1-token KV write per seq before attention",
    "70b": "Llama-3-70B-shaped layer decode: batch 128, 64 q / 8 KV heads, head_dim 128, "
           "ctx log-uniform [256,8192], 64-block shared prefix (ref_cnt 128)",
    "sw": "sliding-window layer decode: batch 32, 32 q / 8 KV heads, head_dim 128, "
          "window 4096, ctx U[4096,32768], only window blocks mapped",
    "long": "Llama-3-8B-shaped long-context decode: batch 16, 32 q / 8 KV heads, head_dim 128, "
            "ctx U[32768,65536], pool 1.2x needed with shuffled ids",
    "fp8": "FP8-E4M3 KV decode: batch 256, 32 q / 8 KV heads, head_dim 128, ctx U[1,16384], "
           "per-KV-head scales, block tables from the host block manager after 10k seeded "
           "alloc/free steps at 95% occupancy",
    "fp4": "FP4-E2M1 KV decode (E4M3 scale per 16 elements, per-KV-head scales): batch 256, "
           "32 q / 8 KV heads, head_dim 128, ctx U[1,16384], block tables from the host block "
           "manager after 10k seeded alloc/free steps at 95% occupancy",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="8b",
                    choices=["tiny", "8b", "70b", "sw", "fp8", "fp4", "long"])
    ap.add_argument("--block-size", type=int, default=16, choices=[16, 32],
                    help="tokens per pool block")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--part-blocks", type=int, default=0, help="split-K partition size (0 = auto)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the block-copy, prefill and host block-manager measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--configs", default="70b,sw,fp8,fp4,long,tiny",
                    help="comma-separated workloads measured after the headline one and "
                         "reported under 'configs' ('none' = only the headline)")
    ap.add_argument("--config-oracle-seconds", type=float, default=3.0,
                    help="oracle CPU time per workload under 'configs' (timing + parity sample)")
    return ap.parse_args(argv)


# ------------------------------------------------------------- host helpers --

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_33_gb300", "csrc")
    for name in ("decode.cu", "common.cuh", "internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str) -> float | None:
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on this exact kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(config)
    if not rec or rec.get("kernel_source_sha") != kernel_source_sha():
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples at 100 ms while running."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = device_index
        self.marks: dict[str, float] = {}
        if shutil.which("nvidia-smi") is None:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.out = open(self.path, "w")
        self.proc = subprocess.Popen(
            ["nvidia-smi", f"--id={device_index}", f"--query-gpu={self.FIELDS}",
             "--format=csv,noheader,nounits", "-lms", "100"],
            stdout=self.out, stderr=subprocess.DEVNULL)

    def mark(self, name: str) -> None:
        self.marks[name] = time.time()

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[1].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append({"t": ts, "sm": float(parts[2]), "max": float(parts[3]),
                                 "reasons": {"hw_slowdown": parts[6], "hw_thermal_slowdown": parts[7],
                                             "sw_thermal_slowdown": parts[8],
                                             "sw_power_cap": parts[9]}})
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        t0, t1 = self.marks.get("timed_start"), self.marks.get("timed_end")
        window = "timed"
        sel = [r for r in rows if t0 is not None and t0 - 1 <= r["t"] <= t1 + 1]
        if len(sel) < 3:
            sel, window = rows, "run"
        reasons = sorted({k for r in sel for k, v in r["reasons"].items() if v == "Active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in sel),
                "sm_max_mhz": max(r["max"] for r in sel), "reasons": reasons,
                "samples": len(sel), "window": window}


# ------------------------------------------------- bytes of one decode launch --

# The decode kernel's split of a launch's units into segments (decode.cu,
# struct Split): 25% of the units go to dynamic chunks once there are at least
# 8 per worker; the chunk regions take 60%, 30% and 10% of them in chunks of
# 16, 8 and 4 units, the rest in chunks of 4.
SPLIT_DYN_PCT = 25
SPLIT_CHUNKS = (16, 8, 4, 4)
SPLIT_REGION_PCT = (60, 30, 10)
MAX_DECODE_BATCH = 512          # sequences per decode launch
NOMINAL_HBM_GBS = 7900.0        # GB300 HBM3e spec-sheet bandwidth


def decode_workers(w, sm_count: int) -> int:
    """Warps of the persistent decode grid: 3 CTAs per SM, 4 warps each
    (2 for bf16 with 32-token blocks, with 6 CTAs per SM)."""
    return sm_count * 12


def blocks_per_unit(w) -> int:
    if w.block_size == 32:
        return 1
    return {"bf16": 1, "fp8": 2, "fp4": 3}[w.dtype]


def _split_segments(T: int, P: int):
    """seg_of(u) of the kernel's split of T units over P workers."""
    Td = T * SPLIT_DYN_PCT // 100 if T >= 8 * P else 0
    Ts = T - Td
    Ps = min(P, Ts)
    c0, c1, c2, c3 = SPLIT_CHUNKS
    r0 = Td * SPLIT_REGION_PCT[0] // 100 // c0 * c0
    r1 = Td * SPLIT_REGION_PCT[1] // 100 // c1 * c1
    r2 = Td * SPLIT_REGION_PCT[2] // 100 // c2 * c2
    s1, s2, s3 = Ts + r0, Ts + r0 + r1, Ts + r0 + r1 + r2
    t1, t2, t3 = r0 // c0, r0 // c0 + r1 // c1, r0 // c0 + r1 // c1 + r2 // c2

    def seg_of(u: int) -> int:
        if u < Ts:
            return ((u + 1) * Ps - 1) // Ts
        if u < s1:
            return Ps + (u - Ts) // c0
        if u < s2:
            return Ps + t1 + (u - s1) // c1
        if u < s3:
            return Ps + t2 + (u - s2) // c2
        return Ps + t3 + (u - s3) // c3
    return seg_of


def decode_launch_bytes(w, sm_count: int) -> dict:
    """Algorithmic bytes of the decode kernel and of its reduce, summed over
    the launches of one call.

    Decode: K/V of the attended tokens (the shared prefix once) + the queries
    + 4 B per block-table entry read per KV head + the outputs of pairs
    finished inside one segment + one partial (g*D unnormalised outputs and
    g (max, sum) pairs, fp32) per segment of a pair cut between segments.
    Reduce: reads those partials, writes the cut pairs' outputs.  Block-
    rounded K/V (whole blocks of every attended range) is given beside the
    exact figure."""
    bs, g, D = w.block_size, w.group, w.head_dim
    bpu = blocks_per_unit(w)
    P = decode_workers(w, sm_count)
    tok = w.kv_bytes_per_token_head() * w.n_kv_heads
    pieces = cut = whole = entries = blocks = 0
    for b0 in range(0, w.batch, MAX_DECODE_BATCH):
        nunits = []
        for b in range(b0, min(w.batch, b0 + MAX_DECODE_BATCH)):
            lo, ctx = w.attended_range(b)
            nblk = (ctx - 1) // bs - lo // bs + 1 if ctx > lo else 0
            blocks += nblk
            entries += nblk * w.n_kv_heads
            nunits.append(-(-nblk // bpu))
        T = sum(n * w.n_kv_heads for n in nunits)
        if T == 0:
            continue
        seg_of = _split_segments(T, P)
        u = 0
        for n in nunits:
            for _ in range(w.n_kv_heads):
                if n == 0:
                    continue
                c = seg_of(u + n - 1) - seg_of(u) + 1
                if c == 1:
                    whole += 1
                else:
                    cut += 1
                    pieces += c
                u += n
    piece_bytes = (g * D + 2 * g) * 4
    out_pair = g * D * 4
    q_bytes = w.batch * w.n_q_heads * D * 2
    decode = (w.kv_bytes_unique() + q_bytes + 4 * entries + whole * out_pair
              + pieces * piece_bytes + 8 * (whole + cut))
    return {"decode": decode, "reduce": pieces * piece_bytes + cut * out_pair,
            "kv_exact": w.kv_bytes_unique(), "kv_block_rounded": _block_rounded_unique(w),
            "partials": pieces, "cut_pairs": cut, "whole_pairs": whole,
            "partial_bytes": pieces * piece_bytes, "table_bytes": 4 * entries,
            "workers": P}


def _block_rounded_unique(w) -> int:
    """K/V bytes of every block an attended range touches, whole (the shared
    prefix's blocks once)."""
    bs = w.block_size
    per_block = bs * w.kv_bytes_per_token_head() * w.n_kv_heads
    prefix_blocks = w.shared_prefix_tokens // bs
    seen_prefix = 0
    n = 0
    for b in range(w.batch):
        lo, ctx = w.attended_range(b)
        if ctx <= lo:
            continue
        first, last = lo // bs, (ctx - 1) // bs
        if prefix_blocks:
            seen_prefix = max(seen_prefix, min(last + 1, prefix_blocks) if first < prefix_blocks else 0)
            first = max(first, prefix_blocks)
        n += max(0, last - first + 1)
    return (n + seen_prefix) * per_block


# ----------------------------------------------------------------- the step --

class Step:
    """Device-resident inputs of one decode step and the calls that run it."""

    def __init__(self, w, device, part_blocks: int = 0):
        import torch
        from paged_kv_cache_33_gb300 import pagedkv

        self.torch, self.pk, self.w = torch, pagedkv, w
        self.pool = pagedkv.KVPool(w.num_blocks, w.block_size, w.n_kv_heads, w.head_dim, w.dtype)
        if w.dtype in ("fp8", "fp4"):
            self.pool.set_scales(torch.from_numpy(w.k_scale).to(device),
                                 torch.from_numpy(w.v_scale).to(device))
        if part_blocks:
            self.pool.set_partition_blocks(part_blocks)
        setup, (k_new, v_new, s_new) = w.fill_plan(device=device)
        for k, v, s in setup:
            pagedkv.paged_kv_write(self.pool, k, v, s.to(device))
        self.k_new, self.v_new = k_new, v_new
        self.slots = s_new.to(device)
        self.q = w.query(device=device)
        self.tables = torch.from_numpy(w.block_tables).to(device)
        self.lens = torch.from_numpy(w.context_lens).to(device)
        self.out = torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=device)
        need = pagedkv.paged_decode_workspace_bytes(self.pool, w.batch, w.n_q_heads,
                                                    w.max_context_len, w.window)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        chunks = -(-w.batch // 512)  # sequences per decode launch are capped at 512
        self.launches = 1 + 2 * chunks  # KV write, then decode + reduce per launch
        torch.cuda.synchronize()
        if self.pool.check_status() != pagedkv.KV_OK:
            raise RuntimeError("pool fill reported a device error")

    def run(self, q=None, tables=None, lens=None, k=None, v=None, slots=None, out=None):
        """One step: the new tokens' K/V written, then attention over the pool."""
        pk, w = self.pk, self.w
        pk.paged_decode_step(self.pool, self.k_new if k is None else k,
                             self.v_new if v is None else v,
                             self.slots if slots is None else slots,
                             self.q if q is None else q,
                             self.tables if tables is None else tables,
                             self.lens if lens is None else lens, w.scale, w.window,
                             max_context_len=w.max_context_len,
                             out=self.out if out is None else out, workspace=self.ws)


def timed_device(step: Step, steps: int, warmup: int, dist_ctx, sampler) -> dict:
    """K steps with all inputs resident, timed with events around the whole
    region; then the same K steps again with the pool's hook bracketing every
    decode kernel launch, for the kernel's own average duration.  (The hook
    puts event records between the step's kernels, which gives up the
    write/decode overlap, so the step time comes from the first region.)"""
    torch = step.torch
    for _ in range(warmup):
        step.run()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record()
        b.record()
    torch.cuda.synchronize()
    dist_ctx.barrier()
    torch.cuda.synchronize()
    sampler.mark("timed_start")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    torch.cuda.nvtx.range_push("timed_steps")
    start.record()
    for _ in range(steps):
        step.run()
    stop.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    dist_ctx.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("kernel_timed_steps")
    for i in range(steps):
        step.pool.set_timing_events(*ev[i])
        step.run()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    sampler.mark("timed_end")
    dist_ctx.barrier()
    step.pool.set_timing_events(None, None)
    status = step.pool.check_status()
    if status != step.pk.KV_OK:
        raise RuntimeError(f"device error during the timed steps: {step.pk.STATUS[status]}")
    elapsed = start.elapsed_time(stop) / 1e3
    kernel = sum(a.elapsed_time(b) for a, b in ev) / 1e3 / steps
    return {"elapsed_s": elapsed, "wall_s": wall, "decode_kernel_s": kernel}


def timed_cold(step: Step, iters: int) -> float:
    """Seconds per step with L2 flushed before each one, outside the events
    that time the step: a 256 MB buffer (about twice the L2) is written, then
    a second one read, so the written lines are evicted (and written back)
    before the step starts and L2 holds only clean lines.  The main figures
    stream inputs larger than L2 back to back; this one also removes what a
    step leaves in L2 for the next (the 70b workload's shared prefix, the
    block tables, the queries) and the overlap between consecutive steps."""
    torch = step.torch
    n = 256 * 1024 * 1024
    flush_w = torch.empty(n, dtype=torch.uint8, device=step.q.device)
    flush_r = torch.ones(n // 4, dtype=torch.int32, device=step.q.device)

    def flush():
        flush_w.fill_(1)
        flush_r.sum()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    for _ in range(3):
        flush()
        step.run()
    torch.cuda.synchronize()
    for a, b in ev:
        flush()
        a.record()
        step.run()
        b.record()
    torch.cuda.synchronize()
    del flush_w, flush_r
    return sum(a.elapsed_time(b) for a, b in ev) / 1e3 / iters


def timed_e2e(step: Step, steps: int, warmup: int, dist_ctx) -> dict:
    """Same steps through the public API with host inputs and a host result.
    Every step's inputs -- q, the new K/V, slots, block tables and context
    lengths, laid out back to back in one pinned host buffer -- are passed to
    paged_decode_step as host memory, which the kernels read in place over
    the host link, and the kernels write the step's output into a pinned host
    buffer: the whole host-to-device and device-to-host traffic of the step
    happens inside the call, with no separate copy.  `staged_s` times the
    same steps with the inputs first copied to device memory by one
    host-to-device copy per step (torch), for comparison."""
    torch, w = step.torch, step.w
    srcs = {"q": step.q, "k": step.k_new, "v": step.v_new, "slots": step.slots,
            "tables": step.tables, "lens": step.lens}
    offs, total = {}, 0
    for name, t in srcs.items():
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=step.q.device)

    def view(buf, name):
        t = srcs[name]
        n = t.numel() * t.element_size()
        return buf[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)

    for name, t in srcs.items():
        view(host_buf, name).copy_(t.cpu())
    host = {name: view(host_buf, name) for name in srcs}
    dev = {name: view(dev_buf, name) for name in srcs}
    out_host = torch.empty(step.out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in srcs.values())
    d2h = out_host.numel() * out_host.element_size()

    def in_place():
        step.run(q=host["q"], tables=host["tables"], lens=host["lens"], k=host["k"],
                 v=host["v"], slots=host["slots"], out=out_host)

    def staged():
        dev_buf.copy_(host_buf, non_blocking=True)
        step.run(q=dev["q"], tables=dev["tables"], lens=dev["lens"], k=dev["k"], v=dev["v"],
                 slots=dev["slots"], out=out_host)

    times = {}
    for label, one in (("in_place", in_place), ("staged", staged)):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        dist_ctx.barrier()
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        torch.cuda.synchronize()
        times[label] = time.perf_counter() - t0
        dist_ctx.barrier()
    return {"elapsed_s": times["in_place"], "staged_s": times["staged"], "h2d": h2d, "d2h": d2h}


# ----------------------------------------------------------------- extras --

def _event_time(torch, fn, iters: int) -> float:
    """Seconds per call of fn, CUDA events on the current stream, after warm-up."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / iters


def measure_extras(step: Step, peaks: dict, device) -> dict:
    """The other operations of the library, each against its own roofline:
    copy-on-write block copies (HBM), prefill attention (tensor cores), and
    the host block manager's per-step work.  Runs after the timed steps, each
    on pools of its own."""
    import numpy as np
    torch, pk, w = step.torch, step.pk, step.w
    out = {}
    # -- paged_kv_copy_blocks: disjoint random pairs, 268 MB moved per call
    #    (134 MB read, 134 MB written), each call timed alone after an L2
    #    flush, on a bf16 pool (64 KB blocks) and on an FP8 pool (32 KB blocks)
    flush_w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    flush_r = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device=device)
    for key, dt, nblocks, npairs in (("paged_kv_copy_blocks", "bf16", 4096, 2048),
                                     ("paged_kv_copy_blocks_fp8", "fp8", 8192, 4096)):
        cpool = pk.KVPool(nblocks, 16, 8, 128, dt)
        pairs = (np.random.default_rng(9).permutation(nblocks)[:2 * npairs].astype(np.int32)
                 .reshape(npairs, 2))
        blk = 8 * 16 * 128 * 2 * (2 if dt == "bf16" else 1)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(20)]
        for i in range(23):
            flush_w.fill_(1)
            flush_r.sum()
            if i >= 3:
                ev[i - 3][0].record()
            pk.paged_kv_copy_blocks(cpool, pairs)
            if i >= 3:
                ev[i - 3][1].record()
        torch.cuda.synchronize()
        t = statistics.median(a.elapsed_time(b) for a, b in ev) / 1e3
        gbs = 2 * blk * npairs / t / 1e9
        out[key] = {
            "dtype": dt, "pairs": npairs, "block_bytes": blk, "launches": -(-npairs // 2048),
            "us_per_call": t * 1e6, "achieved": gbs, "unit": "GB/s", "bound": "hbm",
            "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"], "bytes_per_pair": 2 * blk,
            "note": "median of 20 calls, each after an L2 flush (256 MB written, another 256 MB "
                    "read); 268 MB moved per call"}
        if cpool.check_status() != pk.KV_OK:
            raise RuntimeError("device error in the block copies")
        cpool.destroy()
    del flush_w, flush_r
    # -- paged_prefill_attention: 8B-shaped full causal prefill, 4 x 2048 tokens
    #    (short prompts: per-CTA set-up weighs more) and 4 x 8192 tokens, over
    #    bf16, FP8 and FP4 pools.  The FP8 products run at twice the bf16 rate
    #    (the nominal ratio, 4.5 / 2.25 PFLOP/s dense, applied to the measured
    #    bf16 peak); the bf16 and FP4 kernels' are bf16 / f16 ones (the bf16
    #    rate).  Issued tensor work per algorithmic flop, in units of the peak
    #    used: bf16 1, FP8 2 (Q K^T twice on E4M3; P V once on f16, at half
    #    the E4M3 rate), FP4 1
    bf16_peak = peaks["bf16_tflops"]
    for key, dt, (B, ctx) in (("paged_prefill_attention", "bf16", (4, 2048)),
                              ("paged_prefill_attention_long", "bf16", (4, 8192)),
                              ("paged_prefill_attention_fp8", "fp8", (4, 2048)),
                              ("paged_prefill_attention_fp8_long", "fp8", (4, 8192)),
                              ("paged_prefill_attention_fp4", "fp4", (4, 2048)),
                              ("paged_prefill_attention_fp4_long", "fp4", (4, 8192))):
        hq, hkv = 32, 8
        nblk = ctx // 16
        ppool = pk.KVPool(B * nblk, 16, hkv, 128, dt)
        if dt in ("fp8", "fp4"):   # randn keys and values: |x| < 4.5 for these sizes
            sc = torch.full((hkv,), 4.5 / (448 if dt == "fp8" else 6 * 448), device=device)
            ppool.set_scales(sc, sc)
        tables = torch.from_numpy(np.random.default_rng(3).permutation(B * nblk).astype(np.int32)
                                  .reshape(B, nblk)).to(device)
        g = torch.Generator(device=device).manual_seed(5)
        kk = torch.randn(B * ctx, hkv, 128, device=device, generator=g).to(torch.bfloat16)
        pos = torch.arange(ctx, device=device)
        slots = (tables[:, pos // 16].long() * 16 + pos % 16).reshape(-1)
        pk.paged_kv_write(ppool, kk, kk, slots)
        q = torch.randn(B * ctx, hq, 128, device=device, generator=g).to(torch.bfloat16)
        cu = torch.arange(0, B * ctx + 1, ctx, dtype=torch.int32, device=device)
        lens = torch.full((B,), ctx, dtype=torch.int32, device=device)
        pout = torch.empty(B * ctx, hq, 128, device=device)
        t = _event_time(torch, lambda: pk.paged_prefill_attention(
            ppool, q, cu, tables, lens, 128 ** -0.5, 0, max_q_len=ctx, max_context_len=ctx,
            out=pout), 20)
        flops = 4.0 * 128 * hq * B * (ctx * (ctx + 1) // 2)   # QK and PV over the causal keys
        tf = flops / t / 1e12
        peak = bf16_peak * (2.0 if dt == "fp8" else 1.0)
        issued = {"bf16": 1.0, "fp8": 2.0, "fp4": 1.0}[dt]
        out[key] = {
            "workload": f"full causal prefill, {B} x {ctx} tokens, {hq} q / {hkv} KV heads, "
                        f"head_dim 128, 16-token blocks, {dt} pool",
            "dtype": dt,
            "us_per_call": t * 1e6, "achieved": tf, "unit": "TFLOP/s", "bound": "tensor",
            "peak": peak, "frac": tf / peak, "flops_per_call": flops,
            "issued_tensor_flops_per_call": issued * flops, "issued_frac": issued * tf / peak,
            "peak_source": peaks["source"] + " (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst"
                           + (", x 2 for E4M3 operands)" if dt == "fp8" else ")")}
        if ppool.check_status() != pk.KV_OK or step.pool.check_status() != pk.KV_OK:
            raise RuntimeError("device error in the extra measurements")
        ppool.destroy()
        del kk, q, pout, tables, slots
    # -- host block manager: one decode step's inputs for the bench batch, and
    #    admit / append / free churn
    need = sum(-(-int(c) // w.block_size) for c in w.context_lens)
    bm = pk.BlockManager(need + 64, w.block_size)
    for b in range(w.batch):
        if bm.admit(b, num_tokens=max(1, int(w.context_lens[b])))[0] != 0:
            raise RuntimeError("host block manager: admission failed")
    ids = np.arange(w.batch, dtype=np.int64)
    t0 = time.perf_counter()
    for _ in range(200):
        bm.decode_inputs(ids, w.max_blocks_per_seq)
    t_inputs = (time.perf_counter() - t0) / 200
    t0 = time.perf_counter()
    nops = 0
    for i in range(2000):
        rid = 10_000 + i
        if bm.admit(rid, num_tokens=300)[0] == 0:
            bm.append(rid, n=20)
            bm.free(rid)
            nops += 3
    t_ops = time.perf_counter() - t0
    out["host_block_manager"] = {
        "decode_inputs_us": t_inputs * 1e6, "batch": w.batch,
        "admit_append_free_ops_per_s": nops / t_ops if t_ops > 0 else None,
        "note": "host CPU time through the ctypes binding (includes marshalling)"}
    return out


# ------------------------------------------------------------ distributed --

class DistCtx:
    def __init__(self, want: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            backend = os.environ.get("PAGEDKV_DIST_BACKEND", "nccl")
            if backend == "nccl":
                import torch
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x: float, op: str) -> float:
        if self.dist is None:
            return x
        import torch
        backend = self.dist.get_backend()
        t = torch.tensor([float(x)], dtype=torch.float64,
                         device="cuda" if backend == "nccl" else "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX if op == "max" else self.dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def aggregate(dist_ctx: DistCtx, units: float, elapsed: float) -> tuple[float, float]:
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    return dist_ctx.sum(units), dist_ctx.max(elapsed)


# ------------------------------------------------------------ CPU baseline --

class OracleSampler:
    """Times the oracle (single-threaded fp64) on bounded samples of the
    workload: sequences in seeded order, each filled into the oracle's pool on
    its first visit (untimed) and decoded (timed), cycling through the batch
    again when it is exhausted.  Given the GPU's output of the same step, it
    also compares every sequence it decodes with it (outside the timing)."""

    def __init__(self, w, gpu_out=None, gen_device="cpu"):
        import numpy as np

        import oracle

        self.w = w
        # inputs drawn by the workload's seeded generators on this device (the
        # GPU leg draws its inputs on the GPU: the same seeds on another
        # device's generator give other numbers)
        self.gen_device = gen_device
        self.order = np.random.default_rng(0).permutation(w.batch)
        self.pool = oracle.Pool(w.num_blocks, w.block_size, w.n_kv_heads, w.head_dim, w.dtype)
        if w.dtype in ("fp8", "fp4"):
            self.pool.set_scales(w.k_scale, w.v_scale)
        self.q = w.query(device=gen_device).cpu()
        self.filled: set[int] = set()
        self.decodes = 0
        self.token_bytes = w.n_kv_heads * w.kv_bytes_per_token_head()
        self.gpu_out = gpu_out
        self.checked: set[int] = set()
        self.err_max = 0.0
        self.err_sq = 0.0
        self.ref_sq = 0.0
        self.finite = True

    def _fill(self, b: int) -> None:
        w = self.w
        setup, (k_new, v_new, s_new) = w.fill_plan(seqs=[b], device=self.gen_device)
        for k, v, s in setup:
            self.pool.write(k.cpu(), v.cpu(), s.numpy())
        keep = s_new.clone()
        keep[[i for i in range(w.batch) if i != b]] = -1
        self.pool.write(k_new.cpu(), v_new.cpu(), keep.numpy())
        self.filled.add(b)

    def run(self, budget_s: float, max_seqs: int | None = None) -> tuple[int, float, int]:
        """Decode sequences until ~budget_s of timed work (at least one, at
        most max_seqs); returns (K/V bytes read, seconds, sequences decoded)."""
        import numpy as np
        w = self.w
        done, t, n = 0, 0.0, 0
        while (n == 0 or t < budget_s) and (max_seqs is None or n < max_seqs):
            b = int(self.order[self.decodes % w.batch])
            if b not in self.filled:
                self._fill(b)
            t0 = time.perf_counter()
            o = self.pool.decode(self.q, w.block_tables, w.context_lens, w.scale, w.window,
                                 seqs=[b])
            t += time.perf_counter() - t0
            if self.gpu_out is not None and b not in self.checked:
                ref = o[b].astype(np.float64)
                got = self.gpu_out[b].astype(np.float64)
                self.finite = self.finite and bool(np.isfinite(got).all())
                d = got - ref
                self.err_max = max(self.err_max, float(np.abs(d).max()) if d.size else 0.0)
                self.err_sq += float((d * d).sum())
                self.ref_sq += float((ref * ref).sum())
                self.checked.add(b)
            lo, ctx = w.attended_range(b)
            done += (ctx - lo) * self.token_bytes
            self.decodes += 1
            n += 1
        return done, t, n

    def parity(self) -> dict | None:
        if self.gpu_out is None:
            return None
        tol = {"bf16": (2e-3, 1e-3), "fp8": (3e-2, None), "fp4": (2e-3, 1e-3)}[self.w.dtype]
        rel = (self.err_sq / self.ref_sq) ** 0.5 if self.ref_sq > 0 else 0.0
        ok = self.finite and self.err_max <= tol[0] and (tol[1] is None or rel <= tol[1])
        return {"sequences": len(self.checked), "max_abs_err": self.err_max, "rel_l2_err": rel,
                "tol_max_abs": tol[0], "tol_rel_l2": tol[1], "pass": ok,
                "against": "fp64 oracle on the same seeded inputs, sequences in the sample"}


def host_info() -> dict:
    """The host the CPU figures were taken on: logical CPUs and the CPU model
    (the first model line of /proc/cpuinfo, when the kernel gives one)."""
    import platform
    model, ids = None, {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key = key.strip().lower()
                if key in ("model name", "cpu model", "hardware") and model is None:
                    model = val.strip()
                elif key in ("cpu implementer", "cpu part") and key not in ids:
                    ids[key] = val.strip()   # Arm cores name themselves by these ids
    except OSError:
        pass
    if model is None and ids:
        model = ", ".join(f"{k} {v}" for k, v in ids.items())
    return {"logical_cpus": os.cpu_count(), "machine": platform.machine(), "model": model}


def oracle_workload(name: str, block_size: int, gpu_w=None):
    """The workload rebuilt from its seeds with the oracle's own allocator
    (for the churned pools), so the CPU legs depend on oracle/ alone; when
    the GPU leg's workload is given, its block tables must be identical."""
    import numpy as np

    import oracle
    from paged_kv_cache_33_gb300 import workloads as W
    w = W.make(name, "full", make_allocator=oracle.Allocator, block_size=block_size)
    if gpu_w is not None and not (np.array_equal(w.block_tables, gpu_w.block_tables) and
                                  np.array_equal(w.context_lens, gpu_w.context_lens)):
        raise RuntimeError(f"{name}: the oracle allocator's tables differ from the GPU leg's")
    return w


def oracle_sample(w, budget_s: float, gpu_out=None, max_seqs: int | None = None,
                  gen_device="cpu") -> dict:
    """The cpu_baseline object: the oracle on ~budget_s of the workload, and
    (given the GPU output of the step, whose inputs were drawn on
    `gen_device`) the error of that output on the sampled sequences."""
    sampler = OracleSampler(w, gpu_out, gen_device)
    done, t, n = sampler.run(budget_s, max_seqs)
    out = {"value": done / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "host": host_info(),
           "sample": f"{n} sequence decodes in seeded order ({n / w.batch:.2f} passes over the "
                     f"{w.batch} sequences, {done / 1e6:.1f} MB of K/V), single-threaded fp64 "
                     f"oracle, {t:.1f} s"}
    par = sampler.parity()
    if par is not None:
        out["parity"] = par
    return out


def _fanout_worker(rank: int, n: int, config: str, block_size: int, budget_s: float, queue) -> None:
    """One process of the all-cores oracle figure: the workload rebuilt from
    its seeds, the sampler started at this process's share of the seeded
    sequence order."""
    import numpy as np

    sys.path.insert(0, ROOT)
    w = oracle_workload(config, block_size)
    sampler = OracleSampler(w)
    sampler.order = np.roll(sampler.order, -(rank * w.batch) // n)
    queue.put(sampler.run(budget_s))


def oracle_fanout(config: str, block_size: int, budget_s: float) -> dict:
    """The oracle, unchanged, run as one process per logical CPU on disjoint
    starting points of the sequence order, all at once (spawned processes,
    so no CUDA state is inherited); the figure is the sum of the processes'
    decode rates.  A reported baseline, not a target."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    n = max(1, os.cpu_count() or 1)
    queue = ctx.Queue()
    procs = [ctx.Process(target=_fanout_worker, args=(r, n, config, block_size, budget_s, queue))
             for r in range(n)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=1800) for _ in procs]
    for p in procs:
        p.join()
    rate = sum(done / t for done, t, _ in results if t > 0)
    decodes = sum(k for _, _, k in results)
    return {"value": rate / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "host": host_info(),
            "sample": f"{n} processes of the single-threaded fp64 oracle at once, each ~{budget_s:.0f} s "
                      f"of decodes from its own start in the seeded sequence order ({decodes} "
                      "sequence decodes in all); sum of their rates"}


def run_reference(args) -> None:
    """The reference arm: the oracle itself, timed on this host's cores.  Each
    step is a bounded sample (the whole run takes ~150 s of oracle work)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_33_gb300 import workloads as W
    w = W.make(args.config, "full", make_allocator=oracle.Allocator, block_size=args.block_size)
    per_step_budget = min(6.0, 150.0 / max(1, args.steps + args.warmup))
    sampler = OracleSampler(w)
    for _ in range(args.warmup):
        sampler.run(per_step_budget)
    tot_b, tot_t, tot_n = 0, 0.0, 0
    for _ in range(args.steps):
        b, t, n = sampler.run(per_step_budget)
        tot_b += b
        tot_t += t
        tot_n += n
    value = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{DESCRIPTIONS[args.config]}, {w.block_size}-token blocks",
                       "name": args.config,
                       "batch": w.batch, "parallelism": "none (host oracle)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "host": host_info(),
                             "sample": f"each step: sequences of the {args.config} workload in "
                                       f"seeded order for ~{per_step_budget:.2f} s of "
                                       f"single-threaded fp64 oracle work ({tot_n} sequence "
                                       "decodes in all)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------- main --

def measure(name: str, args, dist_ctx: DistCtx, device, peaks: dict) -> tuple[dict, "Step"]:
    """One workload on this rank's GPU: device-resident steps (value, step
    time, the decode kernel's own time and roofline), cold-L2 steps, end to
    end through the public API with host buffers, and the clocks seen."""
    import torch

    from paged_kv_cache_33_gb300 import pagedkv
    from paged_kv_cache_33_gb300 import workloads as W
    # the churned pools' tables come from the library's own block manager
    w = W.make(name, "full", make_allocator=pagedkv.BlockManager, block_size=args.block_size)
    step = Step(w, device, args.part_blocks)
    sampler = ClockSampler(dist_ctx.local_rank)
    dev = timed_device(step, args.steps, args.warmup, dist_ctx, sampler)
    clocks = sampler.stop()
    e2e_steps = max(10, min(args.steps, 500))
    e2e = timed_e2e(step, e2e_steps, min(args.warmup, 10), dist_ctx)
    cold_s = dist_ctx.max(timed_cold(step, max(5, min(args.steps, 50))))

    kv_bytes = w.kv_bytes_attended()
    unique = w.kv_bytes_unique()
    total_bytes, elapsed = aggregate(dist_ctx, kv_bytes * args.steps, dev["elapsed_s"])
    e2e_bytes, e2e_elapsed = aggregate(dist_ctx, kv_bytes * e2e_steps, e2e["elapsed_s"])
    kernel_s = dist_ctx.max(dev["decode_kernel_s"])
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    lb = decode_launch_bytes(w, sm_count)
    algo = lb["decode"]
    achieved = algo / kernel_s / 1e9
    step_s = elapsed / args.steps
    key = name if w.block_size == 16 else f"{name}-bs{w.block_size}"
    traffic = recorded_traffic(key)
    result = {
        "metric": METRIC, "value": total_bytes / elapsed / 1e9, "unit": "GB/s",
        "n_gpus": dist_ctx.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{DESCRIPTIONS[name]}, {w.block_size}-token blocks",
                   "name": name,
                   "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                   "head_dim": w.head_dim, "block_size": w.block_size,
                   "num_blocks": w.num_blocks, "window": w.window,
                   "kv_bytes_attended_per_step": kv_bytes, "kv_bytes_unique_per_step": unique,
                   "kv_bytes_block_rounded_per_step": lb["kv_block_rounded"],
                   "l2": (f"inputs larger than L2: {unique / 1e6:.0f} MB of distinct K/V per "
                          f"step vs {L2_BYTES / 1e6:.0f} MB L2, no flush" if unique > L2_BYTES
                          else f"{unique / 1e6:.3f} MB of K/V per step fits in L2: back-to-back "
                               "steps are L2-resident; cold_l2 flushes before every step"),
                   "parallelism": f"replicas x{dist_ctx.world} (no collective on the path)"},
        "cold_l2": {"ms_per_step": cold_s * 1e3,
                    "value": dist_ctx.world * kv_bytes / cold_s / 1e9, "unit": "GB/s",
                    "note": "each step alone, L2 flushed (256 MB written, another 256 MB read) "
                            "before it, outside its events"},
        "pct_of_hbm_peak": 100.0 * achieved / peaks["hbm_gbs"],
        "tokens_per_s_per_layer": dist_ctx.world * w.batch / step_s,
        "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy)",
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": algo,
                     "algorithmic_bytes_detail": {
                         "kv_exact": lb["kv_exact"], "kv_block_rounded": lb["kv_block_rounded"],
                         "queries": w.batch * w.n_q_heads * w.head_dim * 2,
                         "table_entries": lb["table_bytes"],
                         "partials_written": lb["partial_bytes"], "partial_pieces": lb["partials"],
                         "cut_pairs": lb["cut_pairs"], "whole_pairs": lb["whole_pairs"]},
                     "reduce_bytes_per_launch": lb["reduce"],
                     "kernel_ms": kernel_s * 1e3,
                     "traffic": traffic,
                     "traffic_over_algorithmic": traffic / algo if traffic else None},
        "e2e": {"value": e2e_bytes / e2e_elapsed / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "steps": e2e_steps,
                "how": "paged_decode_step with every per-step input in pinned host memory, read "
                       "in place by the kernels, and the output written into pinned host memory",
                "staged_value": e2e_bytes / dist_ctx.max(e2e["staged_s"]) / 1e9,
                "staged_how": "the same with the inputs copied to device memory first (one "
                              "host-to-device copy per step)"},
        "clocks": clocks,
        "gpu_launches": step.launches * args.steps,
    }
    return result, step


def config_entry(r: dict) -> dict:
    """The per-workload object under "configs": the headline keys that
    describe one workload's measurement."""
    keys = ("value", "unit", "ms_per_step", "dtype", "config", "cold_l2", "pct_of_hbm_peak",
            "tokens_per_s_per_layer", "roofline", "e2e", "clocks", "gpu_launches",
            "cpu_baseline")
    return {k: r[k] for k in keys if k in r}


def main(argv=None) -> None:
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    from paged_kv_cache_33_gb300 import pagedkv

    dist_ctx = DistCtx(args.gpus)
    torch.cuda.set_device(dist_ctx.local_rank)
    device = torch.device("cuda", dist_ctx.local_rank)
    pagedkv.load()
    peaks = measured_peaks()
    result, step = measure(args.config, args, dist_ctx, device, peaks)
    if dist_ctx.rank == 0 and not args.no_extras:
        result["extras"] = measure_extras(step, peaks, device)
    if dist_ctx.rank == 0 and not args.no_cpu_baseline:
        gpu_out = step.out.cpu().numpy()
        ow = oracle_workload(args.config, step.w.block_size, step.w)
        result["cpu_baseline"] = oracle_sample(ow, args.cpu_baseline_seconds, gpu_out,
                                               gen_device=device)
        result["cpu_baseline_all_cores"] = oracle_fanout(args.config, step.w.block_size,
                                                         args.cpu_baseline_seconds)
    step.pool.destroy()
    del step
    names = [] if args.configs in ("", "none") else [c for c in args.configs.split(",")
                                                      if c and c != args.config]
    if names:
        result["configs"] = {}
    for name in names:
        torch.cuda.empty_cache()
        r, st = measure(name, args, dist_ctx, device, peaks)
        if dist_ctx.rank == 0 and not args.no_cpu_baseline:
            gpu_out = st.out.cpu().numpy()
            ow = oracle_workload(name, st.w.block_size, st.w)
            r["cpu_baseline"] = oracle_sample(ow, args.config_oracle_seconds, gpu_out,
                                              max_seqs=32, gen_device=device)
        st.pool.destroy()
        del st
        result["configs"][name] = config_entry(r)
    dist_ctx.barrier()
    if dist_ctx.rank == 0:
        print(json.dumps(result))
    dist_ctx.close()


if __name__ == "__main__":
    main()
