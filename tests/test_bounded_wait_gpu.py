"""The kernels' bounded waits, run out on purpose.

Every wait a kernel of libpa makes gives up after a time limit instead of
hanging: the attention loop's mbarrier waits for its tile copies, and the
merge launch's poll for partial results that the attention launch writes.
Here each is made to run out with a 1 ms limit, on something that nothing
will ever complete (an mbarrier nobody arrives on; partials no attention
launch writes), and the test checks that the kernel returned, that the status
word reports PA_STATUS_TIMEOUT, and that the context stays usable: the next
decode is bit-identical to one made before.  Nothing here faults, traps or
waits without bound.
"""
import time

import pytest
import torch

from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W

from _helpers import to_cuda

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000   # 1 ms


def test_mbarrier_wait_gives_up_and_reports_timeout():
    assert _abi.pa_get_status()[0] == 0
    t = time.perf_counter()
    _abi.pa_test_wait_timeout(LIMIT_NS)
    rc, bits = _abi.pa_get_status()
    dt = time.perf_counter() - t
    assert rc == _abi.PA_ERR_TIMEOUT and bits & _abi.PA_STATUS_TIMEOUT, (rc, bits)
    assert dt < 1.0, dt                       # gave up after its limit, not the 2 s default
    assert _abi.pa_get_status() == (0, 0)     # the read cleared it
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2  # the context still works


def test_merge_poll_gives_up_then_decode_is_exact():
    w = to_cuda(W.make_workload("qwen2_5_1_5b", seed=5))
    splits = 37                               # 148 workers: most sequences are split
    ws = _abi.alloc_workspace(w.B, w.Hq, w.D, splits, "cuda")
    ref = torch.empty_like(w.q)
    _abi.pa_decode(ref, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                   w.max_context_len, w.scale, splits, ws)
    assert _abi.pa_get_status() == (0, 0)
    assert int(ws.count_nonzero()) == 0       # the call left the workspace zero-filled

    out = torch.full_like(w.q, 7.0)
    t = time.perf_counter()
    _abi.pa_test_merge_timeout(out, w.context_lens, w.max_context_len, w.Hkv, splits, ws,
                               LIMIT_NS)
    rc, bits = _abi.pa_get_status()
    dt = time.perf_counter() - t
    assert rc == _abi.PA_ERR_TIMEOUT and bits & _abi.PA_STATUS_TIMEOUT, (rc, bits)
    assert dt < 1.0, dt
    assert bool(torch.all(out == 7.0))        # a merge that gave up writes no output
    assert int(ws.count_nonzero()) == 0       # ... and nothing into the workspace

    again = torch.empty_like(w.q)
    _abi.pa_decode(again, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                   w.max_context_len, w.scale, splits, ws)
    assert _abi.pa_get_status() == (0, 0)
    assert torch.equal(again, ref)


def test_wait_limits_are_checked_on_the_host():
    for bad in (0, 3_000_000_000):
        with pytest.raises(_abi.PAError) as e:
            _abi.pa_test_wait_timeout(bad)
        assert e.value.code == _abi.PA_ERR_INVALID_ARG
