"""GPU tests of paged_decode_step: the KV write of a step's new tokens fused
with the attention over the pool that then holds them.

The fused call must give the same pool and, bit for bit, the same output as
paged_kv_write followed by paged_decode_attention (both kernels are
deterministic: the split points of the work do not depend on timing), and
both must match the fp64 oracle within the decode tolerance.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_33_gb300 import pagedkv
from paged_kv_cache_33_gb300 import workloads as W

from _parity import assert_close, compare_pools, make_gpu_pool, make_oracle_pool, written_slots

pytestmark = pytest.mark.gpu


def _workload(name, size):
    return W.make(name, size, make_allocator=oracle.Allocator if name in ("fp8", "fp4") else None)


def _setup(w, pool, opool=None):
    setup, step = w.fill_plan()
    for k, v, s in setup:
        pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), s.cuda())
        if opool is not None:
            opool.write(k, v, s.numpy())
    return setup, step


def _inputs(w):
    return (w.query().cuda(), torch.from_numpy(w.block_tables).cuda(),
            torch.from_numpy(w.context_lens).cuda())


def _two_ways(w, hook=False):
    """(fused output, separate-calls output, fused pool, oracle pool, written slots)."""
    q, tables, lens = _inputs(w)
    opool = make_oracle_pool(w)
    fused = make_gpu_pool(w)
    setup, (k, v, s) = _setup(w, fused, opool)
    opool.write(k, v, s.numpy())
    if hook:
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        fused.set_timing_events(*ev)
    out_f = pagedkv.paged_decode_step(fused, k.cuda(), v.cuda(), s.cuda(), q, tables, lens,
                                      w.scale, w.window, max_context_len=w.max_context_len)
    if hook:
        fused.set_timing_events(None, None)
    sep = make_gpu_pool(w)
    _setup(w, sep)
    pagedkv.paged_kv_write(sep, k.cuda(), v.cuda(), s.cuda())
    out_s = pagedkv.paged_decode_attention(sep, q, tables, lens, w.scale, w.window,
                                           max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    for p in (fused, sep):
        assert p.check_status() == pagedkv.KV_OK
    assert torch.equal(fused.view().view(torch.uint8), sep.view().view(torch.uint8))
    sep.destroy()
    return out_f, out_s, fused, opool, written_slots(setup, (k, v, s))


@pytest.mark.parametrize("name", ["tiny", "8b", "70b", "sw", "fp8", "fp4"])
def test_step_equals_write_then_attention(name):
    w = W.make("tiny") if name == "tiny" else _workload(name, "small")
    out_f, out_s, fused, opool, slots = _two_ways(w)
    assert torch.equal(out_f, out_s)
    compare_pools(fused, opool, slots)
    ref = opool.decode(w.query(), w.block_tables, w.context_lens, w.scale, w.window)
    max_abs, rel = assert_close(w, out_f.cpu().numpy(), ref, f"step {w.name}")
    print(f"PARITY step {w.name}/{w.size} max_abs={max_abs:.3e} rel_l2={rel:.3e}")
    fused.destroy()


def test_step_with_timing_hook():
    # the hook launches the decode after the write instead of overlapping it
    w = _workload("70b", "small")
    out_f, out_s, fused, _, _ = _two_ways(w, hook=True)
    assert torch.equal(out_f, out_s)
    fused.destroy()


def test_repeated_steps_reuse_the_workspace():
    # the write kernel of each step clears the decode's work counter
    w = _workload("8b", "small")
    q, tables, lens = _inputs(w)
    pool = make_gpu_pool(w)
    _, (k, v, s) = _setup(w, pool)
    k, v, s = k.cuda(), v.cuda(), s.cuda()
    need = pagedkv.paged_decode_workspace_bytes(pool, w.batch, w.n_q_heads, w.max_context_len,
                                                w.window)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    outs = [pagedkv.paged_decode_step(pool, k, v, s, q, tables, lens, w.scale, w.window,
                                      max_context_len=w.max_context_len, workspace=ws)
            for _ in range(3)]
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    pool.destroy()


@pytest.mark.parametrize("name", ["8b", "fp8"])
def test_result_written_into_pinned_host_memory(name):
    # the kernels write a pinned host `out` directly (mapped host memory): the
    # same bits as a device result, for the fused step and the plain call
    w = _workload(name, "small")
    q, tables, lens = _inputs(w)
    pool = make_gpu_pool(w)
    _, (k, v, s) = _setup(w, pool)
    k, v, s = k.cuda(), v.cuda(), s.cuda()
    host = torch.full((w.batch, w.n_q_heads, w.head_dim), float("nan")).pin_memory()
    dev = pagedkv.paged_decode_step(pool, k, v, s, q, tables, lens, w.scale, w.window,
                                    max_context_len=w.max_context_len)
    got = pagedkv.paged_decode_step(pool, k, v, s, q, tables, lens, w.scale, w.window,
                                    max_context_len=w.max_context_len, out=host)
    torch.cuda.synchronize()
    assert got is host
    assert torch.equal(host, dev.cpu())
    host2 = torch.full_like(host, float("nan")).pin_memory()
    pagedkv.paged_decode_attention(pool, q, tables, lens, w.scale, w.window,
                                   max_context_len=w.max_context_len, out=host2)
    torch.cuda.synchronize()
    assert torch.equal(host2, dev.cpu())
    assert pool.check_status() == pagedkv.KV_OK
    with pytest.raises(TypeError):  # pageable host memory is not accepted
        pagedkv.paged_decode_attention(pool, q, tables, lens, w.scale, w.window,
                                       max_context_len=w.max_context_len,
                                       out=torch.empty_like(host2))
    with pytest.raises(ValueError):
        pagedkv.paged_decode_attention(pool, q, tables, lens, w.scale, w.window,
                                       max_context_len=w.max_context_len, out=host2[:1])
    pool.destroy()


def test_step_over_more_sequences_than_one_launch():
    # 600 sequences: two decode launches, the write fused into the first only
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 70, size=600).astype(np.int32)
    hkv, hq, d = 2, 8, 128
    nblk = [-(-int(c) // 16) for c in lens]
    nb = sum(nblk) + 5
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((600, max(nblk)), -1, dtype=np.int32)
    at = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[at:at + n]
        at += n
    pool = pagedkv.KVPool(nb, 16, hkv, d, "bf16")
    opool = oracle.Pool(nb, 16, hkv, d, "bf16")
    g = torch.Generator().manual_seed(11)
    T = int(lens.sum())
    k = torch.randn(T, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(T, hkv, d, generator=g).to(torch.bfloat16)
    pos = np.concatenate([np.arange(c) for c in lens])
    seq = np.repeat(np.arange(600), lens)
    slots = (tables[seq, pos // 16].astype(np.int64) * 16 + pos % 16)
    last = np.cumsum(lens) - 1                       # each sequence's newest token
    old = np.setdiff1d(np.arange(T), last)
    pagedkv.paged_kv_write(pool, k[old].cuda(), v[old].cuda(), torch.from_numpy(slots[old]).cuda())
    opool.write(k, v, slots)
    q = torch.randn(600, hq, d, generator=g).to(torch.bfloat16)
    scale = d ** -0.5
    out = pagedkv.paged_decode_step(pool, k[last].cuda(), v[last].cuda(),
                                    torch.from_numpy(slots[last]).cuda(), q.cuda(),
                                    torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                                    scale, 0, max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.decode(q, tables, lens, scale, 0)
    w = W.make("tiny")  # bf16 tolerance
    assert_close(w, out.cpu().numpy(), ref, "600 sequences")
    pool.destroy()


def test_step_with_empty_batch_writes_only():
    w = W.make("tiny")
    pool = make_gpu_pool(w)
    opool = make_oracle_pool(w)
    setup, (k, v, s) = _setup(w, pool, opool)
    opool.write(k, v, s.numpy())
    empty_q = torch.empty(0, w.n_q_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
    out = pagedkv.paged_decode_step(pool, k.cuda(), v.cuda(), s.cuda(), empty_q,
                                    torch.zeros(0, 1, dtype=torch.int32, device="cuda"),
                                    torch.zeros(0, dtype=torch.int32, device="cuda"),
                                    w.scale, 0, max_context_len=0)
    torch.cuda.synchronize()
    assert out.shape[0] == 0
    assert pool.check_status() == pagedkv.KV_OK
    compare_pools(pool, opool, written_slots(setup, (k, v, s)))
    pool.destroy()


def test_step_with_no_new_tokens_is_attention():
    w = _workload("sw", "small")
    q, tables, lens = _inputs(w)
    pool = make_gpu_pool(w)
    _, (k, v, s) = _setup(w, pool)
    pagedkv.paged_kv_write(pool, k.cuda(), v.cuda(), s.cuda())
    none_k = torch.empty(0, w.n_kv_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
    none_s = torch.empty(0, dtype=torch.int64, device="cuda")
    out_f = pagedkv.paged_decode_step(pool, none_k, none_k, none_s, q, tables, lens, w.scale,
                                      w.window, max_context_len=w.max_context_len)
    out_a = pagedkv.paged_decode_attention(pool, q, tables, lens, w.scale, w.window,
                                           max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    assert torch.equal(out_f, out_a)
    pool.destroy()


def test_step_reports_a_bad_slot():
    w = W.make("tiny")
    q, tables, lens = _inputs(w)
    pool = make_gpu_pool(w, poison_pool=False)
    _, (k, v, s) = _setup(w, pool)
    bad = s.clone()
    bad[0] = w.num_blocks * 16 + 3
    pagedkv.paged_decode_step(pool, k.cuda(), v.cuda(), bad.cuda(), q, tables, lens, w.scale,
                              0, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert pool.check_status() == 7              # KV_ERR_BAD_SLOT
    pool.destroy()


@pytest.mark.parametrize("name", ["tiny", "8b", "sw", "fp8", "fp4"])
def test_inputs_in_pinned_host_memory_give_the_same_step(name):
    # Every per-step input (new K/V, slots, queries, tables, lengths) read in
    # place from pinned host memory, the output written into pinned host
    # memory: same pool and, bit for bit, the same output as device inputs.
    w = _workload(name, "small")
    q, tables, lens = _inputs(w)
    dev_pool, host_pool = make_gpu_pool(w), make_gpu_pool(w)
    _, (k, v, s) = _setup(w, dev_pool)
    _setup(w, host_pool)
    ref = pagedkv.paged_decode_step(dev_pool, k.cuda(), v.cuda(), s.cuda(), q, tables, lens,
                                    w.scale, w.window, max_context_len=w.max_context_len)
    pin = lambda t: t.cpu().contiguous().pin_memory()
    out = torch.full(tuple(ref.shape), float("nan")).pin_memory()
    pagedkv.paged_decode_step(host_pool, pin(k), pin(v), pin(s), pin(q), pin(tables), pin(lens),
                              w.scale, w.window, max_context_len=w.max_context_len, out=out)
    torch.cuda.synchronize()
    assert dev_pool.check_status() == pagedkv.KV_OK and host_pool.check_status() == pagedkv.KV_OK
    assert torch.equal(out, ref.cpu())
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t   # NaN-poisoned
    assert torch.equal(bits(host_pool.view()), bits(dev_pool.view()))
    # and the attention alone, reading host inputs
    out2 = pagedkv.paged_decode_attention(host_pool, pin(q), pin(tables), pin(lens), w.scale,
                                          w.window, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out2.cpu(), ref.cpu())
    dev_pool.destroy()
    host_pool.destroy()


def test_step_replays_from_a_cuda_graph():
    # The fused step (write, decode as its programmatic dependent, reduce)
    # has no host synchronisation: captured once into a CUDA graph it
    # replays with whatever the captured input buffers hold, bit for bit as
    # a direct call on the same inputs.
    w = _workload("8b", "small")
    q, tables, lens = _inputs(w)
    pool, ref_pool = make_gpu_pool(w), make_gpu_pool(w)
    _, (k, v, s) = _setup(w, pool)
    _setup(w, ref_pool)
    k, v, s = k.cuda(), v.cuda(), s.cuda()
    need = pagedkv.paged_decode_workspace_bytes(pool, w.batch, w.n_q_heads, w.max_context_len,
                                                w.window)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty(w.batch, w.n_q_heads, w.head_dim, device="cuda")
    run = lambda: pagedkv.paged_decode_step(pool, k, v, s, q, tables, lens, w.scale, w.window,
                                            max_context_len=w.max_context_len, out=out,
                                            workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()                                   # first call outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    gen = torch.Generator().manual_seed(11)
    for _ in range(3):
        q.copy_(torch.randn(q.shape, generator=gen).bfloat16())   # new queries, same buffer
        graph.replay()
        ref = pagedkv.paged_decode_step(ref_pool, k, v, s, q, tables, lens, w.scale, w.window,
                                        max_context_len=w.max_context_len)
        torch.cuda.synchronize()
        assert pool.check_status() == pagedkv.KV_OK and ref_pool.check_status() == pagedkv.KV_OK
        assert torch.equal(out, ref)
    pool.destroy()
    ref_pool.destroy()


def test_step_with_sixteen_query_heads_per_kv_head():
    # a group of 16 runs the decode as two passes of 8 heads; the fused call
    # must match the write followed by the attention, bit for bit, and the
    # oracle within the bf16 bar
    lens = np.array([3, 16, 40, 129, 500], dtype=np.int32)
    bs, hkv, hq = 16, 2, 32
    nblk = [-(-int(c) // bs) for c in lens]
    nb = sum(nblk) + 3
    perm = np.random.default_rng(21).permutation(nb).astype(np.int32)
    tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[off:off + n]
        off += n
    w = W.Workload("g16", "small", len(lens), hq, hkv, 128, bs, nb, 0, "bf16", 128 ** -0.5, lens,
                   tables, (lens - 1).astype(np.int64), data_seed=4242)
    out_f, out_s, fused, opool, written = _two_ways(w)
    assert torch.equal(out_f, out_s)
    ref = opool.decode(w.query(), w.block_tables, w.context_lens, w.scale, w.window)
    assert_close(w, out_f.cpu().numpy(), ref, "g16 fused")
    fused.destroy()
