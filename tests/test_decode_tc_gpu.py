"""The decode launch on the fifth-generation tensor cores (17 to 32 query rows
per (sequence, kv head) over 16-bit pools at head_dim 128: multi-query
attention with 32 q heads on one kv head, 4 query tokens of a 7-head group,
query groups of 20).  The general cases of that row range run in
test_query_tiles_gpu.py and test_multiquery_gpu.py; these add the full-size
batches on sampled sequences, the fused append + decode step in bf16 with an
early prologue, the device-side handshake (equal results, and an upload
that never arrives), empty and one-token contexts, a bad block id,
run-to-run determinism, and a sweep over 17 to 32 rows (odd groups, up to
32 query tokens, windows, NaN in unused pool rows) -- every result against
the fp64 oracle.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import TOL, max_err, to_cuda, to_np16

pytestmark = pytest.mark.gpu


def _sample_rows(lens, seed, n=32):
    """The 8 shortest and 8 longest sequences, and n - 16 drawn between."""
    order = np.argsort(lens, kind="stable")
    picked = np.random.default_rng(seed).choice(order[8:-8], size=n - 16, replace=False)
    rows = sorted({int(x) for x in np.concatenate([order[:8], order[-8:], picked])})
    assert len(rows) == n
    return rows


@pytest.mark.parametrize("config,nq,early", [("mqa_32x1", 1, True), ("qwen2_5_7b", 4, True),
                                              ("qwen2_5_7b", 4, False)])
def test_full_batch_matches_oracle_on_sampled_sequences(config, nq, early):
    w = to_cuda(W.make_workload(config, seed=3))
    g = torch.Generator(device="cuda").manual_seed(11)
    q = (torch.randn(w.B, nq, w.Hq, w.D, generator=g, device="cuda").to(w.q.dtype) if nq > 1
         else w.q)
    step = DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, early_prologue=early, queries_per_seq=nq)
    out = torch.full_like(q, float("nan"))
    step.decode(q, out)
    assert _abi.pa_get_status() == (0, 0)
    assert int(step.workspace.count_nonzero()) == 0
    lens = w.context_lens.cpu().numpy()
    rows = _sample_rows(lens, 5)
    sub_t, sub_l, (kp, vp) = W.extract_rows(w.block_tables.cpu().numpy(), lens, rows,
                                            [w.k_cache, w.v_cache])
    ref = oracle.decode(to_np16(q[rows]), kp, vp, sub_t, sub_l, w.scale)
    assert max_err(out[rows], ref) <= TOL["f16"]


def test_fused_step_bf16_with_early_prologue():
    B, Hq, Hkv, D = 6, 32, 1, 128
    g = torch.Generator().manual_seed(21)
    lens = torch.randint(1, 1500, (B,), generator=g).to(torch.int32)
    lens[0] = 16                               # the new token ends a block
    lens[1] = 17                               # ... or starts one
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 5
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    dt = torch.bfloat16
    q = torch.randn(B, Hq, D, generator=g).to(dt)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(dt)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(dt)
    kn = torch.randn(B, Hkv, D, generator=g).to(dt)
    vn = torch.randn(B, Hkv, D, generator=g).to(dt)
    last = lens.to(torch.int64) - 1
    slots = tables[torch.arange(B), last // 16].to(torch.int64) * 16 + last % 16
    k_ref, v_ref = to_np16(kp).copy(), to_np16(vp).copy()
    oracle.cache_append(to_np16(kn), to_np16(vn), k_ref, v_ref, slots.numpy(), 16)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.decode(to_np16(q), k_ref, v_ref, tables.numpy(), lens.numpy(), scale, bf16=True)
    kd, vd = kp.cuda(), vp.cuda()
    step = DecodeStep(k_cache=kd, v_cache=vd, block_tables=tables.cuda(),
                      context_lens=lens.cuda(), max_context_len=int(lens.max()), scale=scale,
                      num_q_heads=Hq, split_ctas=7, early_prologue=True)
    out = torch.empty_like(q, device="cuda")
    step.fused(q.cuda(), kn.cuda(), vn.cuda(), slots.cuda(), out)
    assert _abi.pa_get_status() == (0, 0)
    assert np.array_equal(to_np16(kd).view(np.uint16), k_ref.view(np.uint16))
    assert np.array_equal(to_np16(vd).view(np.uint16), v_ref.view(np.uint16))
    assert max_err(out, ref) <= TOL["bf16"]


def _sync(words, ready_value, done_value):
    sy = _abi.StepSync()
    sy.ready = words[0].data_ptr()
    sy.done = words[8].data_ptr()
    sy.done_count = words[16].data_ptr()
    sy.ready_value = ready_value
    sy.done_value = done_value
    return sy


def _mqa_step(lens, seed, splits=0):
    w = to_cuda(W.make_workload("mqa_32x1", seed=seed, lens_override=lens))
    step = DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, split_ctas=splits)
    return w, step


def test_synced_step_equals_plain_step():
    w, step = _mqa_step([1, 17, 300, 2000, 5000, 64, 129, 900], 4)
    k2, v2 = w.k_cache.clone(), w.v_cache.clone()
    ref_step = DecodeStep(k_cache=k2, v_cache=v2, block_tables=w.block_tables,
                          context_lens=w.context_lens, max_context_len=w.max_context_len,
                          scale=w.scale, num_q_heads=w.Hq)
    words = torch.zeros(32, dtype=torch.int32, device="cuda")
    out, ref = torch.empty_like(w.q), torch.empty_like(w.q)
    _abi.pa_stream_write_value(words[:1], 3)             # the inputs are already in place
    step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, out, sync=_sync(words, 3, 9))
    ref_step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, ref)
    assert _abi.pa_get_status() == (0, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(w.k_cache.view(torch.int16), k2.view(torch.int16))
    assert int(words[8]) == 9 and int(words[16]) == 0    # done signalled, count reset


def test_step_without_upload_times_out_and_still_signals_done():
    w, step = _mqa_step([1, 17, 100, 256, 700], 2, splits=6)
    words = torch.zeros(32, dtype=torch.int32, device="cuda")
    out = torch.full_like(w.q, 7.0)
    k0 = w.k_cache.clone()
    back = torch.cuda.Stream()
    t = time.perf_counter()
    step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, out, sync=_sync(words, 1, 5))
    _abi.pa_stream_wait_value(words[8:9], 5, back)       # the read-back stream's wait
    back.synchronize()
    dt = time.perf_counter() - t
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_TIMEOUT and bits & _abi.PA_STATUS_TIMEOUT, (rc, bits)
    assert dt < 10.0, dt
    assert int(words[8]) == 5 and int(words[16]) == 0
    assert bool(torch.all(out == 7.0))                   # nothing attended, nothing written
    assert torch.equal(w.k_cache.view(torch.int16), k0.view(torch.int16))   # nothing appended
    step.workspace.zero_()
    out2 = torch.empty_like(w.q)
    step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, out2)
    assert _abi.pa_get_status() == (0, 0)
    assert bool(torch.isfinite(out2.float()).all())


def test_empty_and_single_token_contexts():
    B, Hq, Hkv, D = 4, 32, 1, 128
    g = torch.Generator().manual_seed(60)
    lens = torch.tensor([0, 1, 17, 300], dtype=torch.int32)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 2
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    q = torch.randn(B, Hq, D, generator=g).half()
    kp = torch.randn(NB, Hkv, 16, D, generator=g).half()
    vp = torch.randn(NB, Hkv, 16, D, generator=g).half()
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, 5, "cuda", query_rows=Hq)
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(), 300, scale,
                   5, ws)
    assert _abi.pa_get_status() == (0, 0)
    got = out.float().cpu().numpy()
    assert np.all(got[0] == 0)                                   # L = 0: zeros
    v0 = vp[int(tables[1, 0]), 0, 0].float().numpy()             # L = 1: V[0], rounded once
    assert np.array_equal(got[1], np.broadcast_to(v0, got[1].shape))
    assert np.abs(got - ref).max() <= TOL["f16"]


def test_bad_block_id_is_reported_not_read():
    w, step = _mqa_step([40, 300, 1000, 77], 8, splits=3)
    bt = w.block_tables.clone()
    bt[2, 5] = w.num_blocks + 1000           # outside the pool
    out = torch.empty_like(w.q)
    _abi.pa_decode(out, w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.max_context_len,
                   w.scale, 3, step.workspace)
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_BOUNDS and bits & _abi.PA_STATUS_BAD_BLOCK
    assert bool(torch.isfinite(out.float()).all())
    # the other sequences are exact, and the context stays usable
    lens = w.context_lens.cpu().numpy()
    ref = oracle.decode(to_np16(w.q), to_np16(w.k_cache), to_np16(w.v_cache),
                        w.block_tables.cpu().numpy(), lens, w.scale)
    assert max_err(out, ref, rows=[0, 1, 3]) <= TOL["f16"]
    step.workspace.zero_()
    step.decode(w.q, out)
    assert _abi.pa_get_status() == (0, 0)
    assert max_err(out, ref) <= TOL["f16"]


def test_results_are_deterministic():
    w, step = _mqa_step(None, 9)             # the full 128-sequence batch: many split segments
    outs = []
    for _ in range(3):
        out = torch.empty_like(w.q)
        step.decode(w.q, out)
        outs.append(out)
    assert _abi.pa_get_status() == (0, 0)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))


def _rows_case(seed, B, nq, G, D, max_len, dtype):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(max(1, nq), max_len + 1, (B,), generator=g).to(torch.int32)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 3
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    Hkv = 2
    shape = (B, G * Hkv, D) if nq == 1 else (B, nq, G * Hkv, D)
    q = torch.randn(*shape, generator=g).to(dtype)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    # rows past each context's end hold NaN: they must not reach any output
    for b in range(B):
        L = int(lens[b])
        if L % 16:
            blk = int(tables[b, L // 16])
            kp[blk, :, L % 16:] = float("nan")
            vp[blk, :, L % 16:] = float("nan")
    return q, kp, vp, tables, lens


# (n_q, G): 17 to 32 rows per kv head, odd groups, dead columns, several
# tokens (causal among them), windows shorter than a block and than a chunk
@pytest.mark.parametrize("seed,nq,G,window,splits,dtype", [
    (80, 1, 17, 0, 0, torch.float16), (81, 1, 23, 0, 5, torch.bfloat16),
    (82, 1, 31, 0, 2, torch.float16), (83, 3, 6, 0, 0, torch.float16),
    (84, 2, 9, 0, 11, torch.bfloat16), (85, 5, 5, 0, 0, torch.float16),
    (86, 8, 4, 0, 3, torch.float16), (87, 4, 8, 7, 0, torch.bfloat16),
    (88, 2, 13, 130, 9, torch.float16), (89, 3, 9, 300, 0, torch.float16),
    (90, 32, 1, 0, 0, torch.float16), (91, 16, 2, 50, 6, torch.bfloat16)])
def test_row_counts_17_to_32_match_oracle(seed, nq, G, window, splits, dtype):
    B, D = 5, 128
    q, kp, vp, tables, lens = _rows_case(seed, B, nq, G, D, 900, dtype)
    Hq = G * 2
    scale = float(np.float32(1 / math.sqrt(D)))
    bf16 = dtype == torch.bfloat16
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale,
                        bf16=bf16, window=window)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda", query_rows=nq * G)
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(),
                   int(lens.max()), scale, splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    assert max_err(out, ref) <= TOL["bf16" if bf16 else "f16"]
    assert int(ws.count_nonzero()) == 0     # the merge left the workspace zero-filled


def test_contexts_shorter_than_the_query_tokens():
    # 8 query tokens x a group of 4 = 32 rows; queries before position 0 see
    # nothing and return zeros, the rest attend causally what exists
    B, nq, G, Hkv, D = 6, 8, 4, 2, 128
    lens = [1, 3, 7, 8, 9, 200]
    g = torch.Generator().manual_seed(95)
    lt = torch.tensor(lens, dtype=torch.int32)
    nblk = (lt + 15) // 16
    NB = int(nblk.sum()) + 2
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    q = torch.randn(B, nq, G * Hkv, D, generator=g).half()
    kp = torch.randn(NB, Hkv, 16, D, generator=g).half()
    vp = torch.randn(NB, Hkv, 16, D, generator=g).half()
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lt.numpy(), scale)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, G * Hkv, D, 3, "cuda", query_rows=nq * G)
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lt.cuda(), 200, scale, 3, ws)
    assert _abi.pa_get_status() == (0, 0)
    got = out.float().cpu().numpy()
    for b, L in enumerate(lens):
        if L < nq:
            assert np.all(got[b, :nq - L] == 0)     # the queries before position 0
    assert np.abs(got - ref).max() <= TOL["f16"]
