"""pa_decode (16-bit pools) on the GPU against the fp64 oracle.

Whole batches of the four 16-bit workloads (append + decode, in the launch
configuration the benchmark times), random small shapes that span several
partitions and a ragged last block, invariance to how the batch is split
across CTAs, and the edge
cases: context_len 0 and 1, NaN in unfilled rows, bad block ids and lengths.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import TOL, max_err, oracle_step, to_cuda, to_np16

pytestmark = pytest.mark.gpu


def _step_for(w, split_ctas=0):
    return DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, split_ctas=split_ctas)


@pytest.mark.parametrize("name,seed", [("tiny", 0), ("tiny", 1), ("smollm2_360m", 0),
                                       ("smollm2_360m", 3), ("qwen2_5_1_5b", 0),
                                       ("qwen2_5_7b", 0), ("qwen2_5_7b", 4)])
def test_full_step_matches_oracle(name, seed):
    w = W.make_workload(name, seed=seed)
    ref = oracle_step(w)
    to_cuda(w)
    step = _step_for(w)
    out = torch.empty_like(w.q)
    step(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert _abi.pa_get_status() == (0, 0)
    err = max_err(out, ref)
    assert err <= TOL[w.dtype], (name, seed, step.split_ctas, err)


def _random_workload(seed, B, Hq, Hkv, D, dtype, max_len, fill="zero"):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, max_len + 1, (B,), generator=g)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 3
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    mbs = int(nblk.max())
    tables = torch.full((B, mbs), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    tdt = W.TORCH_DTYPE[dtype]
    last = lens - 1
    slots = tables[torch.arange(B), last // 16].to(torch.int64) * 16 + last % 16
    return W.Workload(
        name="random", B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, kv=dtype, block_size=16,
        num_blocks=NB, max_context_len=int(lens.max()), context_lens=lens.to(torch.int32),
        block_tables=tables, slot_mapping=slots,
        q=torch.randn(B, Hq, D, generator=g).to(tdt),
        k_cache=torch.randn(NB, Hkv, 16, D, generator=g).to(tdt),
        v_cache=torch.randn(NB, Hkv, 16, D, generator=g).to(tdt),
        k_new=torch.randn(B, Hkv, D, generator=g).to(tdt),
        v_new=torch.randn(B, Hkv, D, generator=g).to(tdt),
        scale=float(np.float32(1 / math.sqrt(D))), seed=seed)


CASES = [
    # seed, B, Hq, Hkv, D, dtype, max_len, CTAs the batch is split across
    (10, 5, 8, 2, 64, "f16", 300, 16),
    (11, 3, 7, 1, 128, "f16", 700, 5),
    (12, 6, 15, 5, 64, "bf16", 500, 33),
    (13, 4, 28, 4, 128, "f16", 1000, 304),
    (14, 2, 12, 2, 128, "bf16", 2100, 7),
    (15, 7, 4, 4, 128, "f16", 90, 1000),     # MHA (group 1); more CTAs than blocks
    (16, 3, 16, 2, 64, "f16", 333, 3),       # group of 8
    (17, 8, 6, 3, 128, "bf16", 40, 1),       # one CTA: every sequence whole
]


@pytest.mark.parametrize("case", CASES)
def test_random_shapes_match_oracle(case):
    seed, B, Hq, Hkv, D, dtype, max_len, part = case
    w = _random_workload(seed, B, Hq, Hkv, D, dtype, max_len)
    ref = oracle_step(w)
    to_cuda(w)
    out = torch.empty_like(w.q)
    _step_for(w, part)(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert _abi.pa_get_status() == (0, 0)
    assert max_err(out, ref) <= TOL[dtype]


def test_split_invariance():
    w = W.make_workload("qwen2_5_1_5b", seed=2)
    ref = oracle_step(w)
    to_cuda(w)
    outs = []
    k0, v0 = w.k_cache.clone(), w.v_cache.clone()
    for splits in (1, 2, 7, 64, 304, 999, 7207):   # the last: more warps than blocks
        w.k_cache.copy_(k0)
        w.v_cache.copy_(v0)
        out = torch.empty_like(w.q)
        _step_for(w, splits)(w.q, w.k_new, w.v_new, w.slot_mapping, out)
        assert _abi.pa_get_status() == (0, 0)
        assert max_err(out, ref) <= TOL["f16"], splits
        outs.append(out.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2 * TOL["f16"]


@pytest.mark.parametrize("splits", [1, 4, 5, 8, 9, 12, 16, 17, 20])
def test_merge_rounds_match_oracle(splits):
    """One sequence of 4096 tokens on two kv heads, split over 4 x splits
    warps: each segment comes in about 2 x splits pieces, so the merge's
    rounds (two piece groups of 8 when its grid is small) are crossed at
    every boundary -- part-full groups, an empty second group, several
    rounds.  Equal to the oracle, and the workspace left zero-filled."""
    w = W.make_workload("qwen2_5_1_5b", seed=21, lens_override=[4096])
    ref = oracle_step(w)
    to_cuda(w)
    step = _step_for(w, splits)
    out = torch.empty_like(w.q)
    step(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert _abi.pa_get_status() == (0, 0)
    assert max_err(out, ref) <= TOL["f16"]
    torch.cuda.synchronize()
    assert int(step.workspace.count_nonzero()) == 0


def test_deterministic():
    w = to_cuda(W.make_workload("qwen2_5_7b", seed=0))
    step = _step_for(w)
    a, b = torch.empty_like(w.q), torch.empty_like(w.q)
    step.decode(w.q, a)
    step.decode(w.q, b)
    assert torch.equal(a, b)


def test_nan_in_unfilled_rows_is_ignored():
    w = W.make_workload("tiny", seed=3, fill="nan")
    kp, vp = to_np16(w.k_cache).copy(), to_np16(w.v_cache).copy()
    kp[np.isnan(kp)] = 0
    vp[np.isnan(vp)] = 0
    oracle.cache_append(to_np16(w.k_new), to_np16(w.v_new), kp, vp, w.slot_mapping.numpy(), 16)
    ref = oracle.decode(to_np16(w.q), kp, vp, w.block_tables.numpy(), w.context_lens.numpy(),
                        w.scale)
    to_cuda(w)
    out = torch.empty_like(w.q)
    _step_for(w, 9)(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert torch.isfinite(out).all()
    assert max_err(out, ref) <= TOL["f16"]


def test_context_len_one_returns_v0_and_zero_returns_zeros():
    w = to_cuda(W.make_workload("tiny", seed=0))
    lens = torch.tensor([1, 0, 1, 0], dtype=torch.int32, device="cuda")
    out = torch.full_like(w.q, 7.0)
    _abi.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.max_context_len,
                   w.scale, 5, _abi.alloc_workspace(4, 8, 64, 5, "cuda"))
    assert _abi.pa_get_status() == (0, 0)
    for b in (0, 2):
        blk = int(w.block_tables[b, 0])
        for hq in range(8):
            assert torch.equal(out[b, hq], w.v_cache[blk, hq // 4, 0])
    assert not out[1].any() and not out[3].any()


def test_bad_block_id_and_length_are_reported_not_read():
    w = to_cuda(W.make_workload("tiny", seed=0))
    bt = w.block_tables.clone()
    bt[3, 2] = w.num_blocks + 1000          # outside the pool
    out = torch.empty_like(w.q)
    ws = _abi.alloc_workspace(4, 8, 64, 6, "cuda")
    _abi.pa_decode(out, w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.max_context_len,
                   w.scale, 6, ws)
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_BOUNDS and bits & _abi.PA_STATUS_BAD_BLOCK
    lens = w.context_lens.clone()
    lens[1] = w.max_context_len + 5          # longer than the stated bound
    _abi.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.max_context_len,
                   w.scale, 6, ws)
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_BOUNDS and bits == _abi.PA_STATUS_BAD_LEN
    assert not out[1].any()
    # the context stays usable
    _abi.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                   w.max_context_len, w.scale, 6, ws)
    assert _abi.pa_get_status() == (0, 0)
