"""Host-side logic of bench.py: multi-rank aggregation over gloo (2 ranks on
the CPU) and the JSON contract of the reference arm."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "PAGEDKV_DIST_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    ctx = bench.DistCtx(world)
    units, elapsed = bench.aggregate(ctx, units=100.0 * (rank + 1), elapsed=1.0 + rank)
    ctx.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"units": units, "elapsed": elapsed}, f)
    ctx.close()


def test_two_gloo_ranks_sum_units_and_take_the_slowest_time(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["units"] == 300.0 and d["elapsed"] == 2.0


def test_reference_arm_prints_one_json_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    host = d["cpu_baseline"]["host"]
    assert host["logical_cpus"] == os.cpu_count() and host["machine"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert res.returncode == 0 and res.stdout.strip() == ""


def _units_by_segment(T, P):
    sys.path.insert(0, ROOT)
    import bench
    seg_of = bench._split_segments(T, P)
    return [seg_of(u) for u in range(T)]


def test_split_model_segments_are_contiguous_and_cover_every_unit():
    for T, P in [(10, 1824), (5000, 1824), (14597, 1824), (40000, 1824), (123, 7)]:
        segs = _units_by_segment(T, P)
        assert segs[0] == 0
        assert all(b - a in (0, 1) for a, b in zip(segs, segs[1:]))   # contiguous, in order
        if T >= 8 * P:   # 25% dynamic: static shares then chunks of 16, 8, 4
            Ts = T - T * 25 // 100
            assert len(set(segs[:Ts])) == P
            assert segs[Ts:Ts + 16] == [P] * 16
        else:            # static shares only
            assert len(set(segs)) == min(T, P)


def test_launch_bytes_of_the_tiny_workload_by_hand():
    # ctx {5, 16, 33, 70} in 16-token blocks, 1 KV head: 1, 1, 3 and 5 units,
    # 10 units for 1824 workers, so every unit is its own segment: the 3- and
    # 5-unit pairs are cut into 8 pieces, the other two finish whole.
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_33_gb300 import workloads as W
    w = W.make("tiny")
    lb = bench.decode_launch_bytes(w, 152)
    assert (lb["partials"], lb["cut_pairs"], lb["whole_pairs"]) == (8, 2, 2)
    piece = (2 * 64 + 2 * 2) * 4
    kv = (5 + 16 + 33 + 70) * 2 * 64 * 2
    assert lb["kv_exact"] == kv
    assert lb["kv_block_rounded"] == (1 + 1 + 3 + 5) * 16 * 2 * 64 * 2
    assert lb["decode"] == kv + 4 * 2 * 64 * 2 + 4 * 10 + 2 * 2 * 64 * 4 + 8 * piece + 8 * 4
    assert lb["reduce"] == 8 * piece + 2 * 2 * 64 * 4


def test_block_rounded_bytes_count_the_shared_prefix_once():
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_33_gb300 import workloads as W
    w = W.make("70b", "small")
    per_block = 16 * 8 * 128 * 2 * 2
    blocks = 64 if w.context_lens.max() >= 1024 else -(-int(w.context_lens.max()) // 16)
    blocks += sum(max(0, -(-int(c) // 16) - 64) for c in w.context_lens)
    assert bench._block_rounded_unique(w) == blocks * per_block
