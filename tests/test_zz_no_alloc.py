"""pa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (its scratch is a static array inside the library).

Its output must match pa_decode's (which uses a caller-allocated workspace)
within the decode tolerances, on two calls in a row: the second call runs on
the scratch the first one left behind.  This file is collected last, so a run
that stops at the first failure has run every other test first; it also
passes on its own in a fresh process (the first call sets the scratch up).
"""
import pytest
import torch

from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W

from _helpers import TOL, to_cuda

pytestmark = pytest.mark.gpu


def _reference(w, splits):
    out = torch.empty_like(w.q)
    ws = _abi.alloc_workspace(w.B, w.Hq, w.D, splits, w.q.device)
    _abi.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                   w.max_context_len, w.scale, splits, ws)
    return out


@pytest.mark.parametrize("name,splits", [("qwen2_5_7b", 0), ("smollm2_360m", 0),
                                         ("qwen2_5_1_5b", 37)])
def test_noalloc_matches_pa_decode_on_two_calls_in_a_row(name, splits):
    w = to_cuda(W.make_workload(name, seed=3))
    ref = _reference(w, splits)
    assert _abi.pa_get_status() == (0, 0)
    for call in range(2):
        out = torch.full_like(w.q, float("nan"))
        _abi.pa_decode_noalloc(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                               w.max_context_len, w.scale, splits)
        assert _abi.pa_get_status() == (0, 0), call
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= TOL[w.dtype], (name, call, err)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = to_cuda(W.make_workload("tiny", seed=0))
    out = torch.empty_like(w.q)
    with pytest.raises(_abi.PAError) as e:
        # 100000 CTAs x 4 warps of partial rows need far more than the static array
        _abi.pa_decode_noalloc(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                               w.max_context_len, w.scale, 100000)
    assert e.value.code == _abi.PA_ERR_SCRATCH_LIMIT
