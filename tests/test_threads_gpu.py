"""Decodes from several host threads at once.

The library's host state is per device (status word, SM count) or per host
thread (tensor-map cache); the decode kernel's dynamic shared-memory limit,
though, is one attribute of the function for the whole process.  Two threads
that alternate a 512-sequence batch (the largest launch layout) with a
1-sequence batch, each on its own stream and workspace, must both get
results identical to the same calls made from one thread.
"""
import threading

import pytest
import torch

from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W

from _helpers import to_cuda

pytestmark = pytest.mark.gpu


def _batch(n_seqs, seed):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, 200, (n_seqs,), generator=g)
    return to_cuda(W.make_workload("smollm2_360m", seed=seed, lens_override=lens))


def _decode(w, out, ws, splits):
    _abi.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                   w.max_context_len, w.scale, splits, ws)


@pytest.mark.parametrize("order", ["big_first", "small_first"])
def test_two_threads_alternating_batch_sizes(order):
    splits = 24
    big, small = _batch(512, 11), _batch(1, 12)
    jobs = [big, small] if order == "big_first" else [small, big]
    refs = []
    for w in jobs:
        ws = _abi.alloc_workspace(w.B, w.Hq, w.D, splits, "cuda")
        ref = torch.empty_like(w.q)
        _decode(w, ref, ws, splits)
        refs.append(ref)
    assert _abi.pa_get_status() == (0, 0)

    errors = []
    barrier = threading.Barrier(len(jobs))

    def worker(i):
        w = jobs[i]
        stream = torch.cuda.Stream()
        ws = _abi.alloc_workspace(w.B, w.Hq, w.D, splits, "cuda")
        torch.cuda.synchronize()
        try:
            with torch.cuda.stream(stream):
                for it in range(16):
                    barrier.wait(timeout=60)
                    out = torch.empty_like(w.q)
                    _decode(w, out, ws, splits)
                    stream.synchronize()
                    if not torch.equal(out, refs[i]):
                        errors.append((i, it, "mismatch"))
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append((i, repr(e)))
            barrier.abort()

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert _abi.pa_get_status() == (0, 0)
