"""The timeout path of the decode kernel, exercised without a GPU fault.

With the pool's test stall enabled, the first copy of worker 0 expects 16
bytes more than it brings, so that warp's wait (bounded to 2 ms here) runs
out: the kernel records KV_ERR_TIMEOUT, supplies the 16 missing bytes to
that barrier itself, drains the copies it issued (every copy lands, so the
drain completes and no KV_ERR_DRAIN_TIMEOUT is recorded) and returns.  The
host reads the status, and the same context then computes a correct step.
"""

import pytest
import torch

from paged_kv_cache_33_gb300 import pagedkv
from paged_kv_cache_33_gb300 import workloads as W

from _parity import assert_close, decode_gpu, fill_both, make_gpu_pool, make_oracle_pool

pytestmark = pytest.mark.gpu

KV_ERR_TIMEOUT = 6


@pytest.mark.parametrize("name", ["8b", "sw"])
def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable(name):
    w = W.make(name, "small")
    pool = make_gpu_pool(w)
    opool = make_oracle_pool(w)
    fill_both(w, pool, opool)
    q = w.query()
    pool.set_wait_limit(2_000_000)
    pool.set_test_stall(True)
    decode_gpu(w, pool, q)
    torch.cuda.synchronize()
    assert pool.check_status() == KV_ERR_TIMEOUT
    pool.set_test_stall(False)
    out = decode_gpu(w, pool, q)
    torch.cuda.synchronize()
    assert pool.check_status() == pagedkv.KV_OK
    ref = opool.decode(q, w.block_tables, w.context_lens, w.scale, w.window)
    assert_close(w, out.cpu().numpy(), ref, f"{name} after a timeout")
    pool.destroy()


def test_wait_limit_bounds():
    pool = pagedkv.KVPool(4, 16, 1, 64)
    with pytest.raises(pagedkv.KVError):
        pool.set_wait_limit(10)              # below 100 us
    pool.set_wait_limit(1_000_000_000)
    pool.destroy()
