"""More than 8 query rows per (sequence, kv head) in one pass over the K/V.

A warp holds one, two or four tiles of the MMA's 8 query columns, so a launch
serves up to 32 query rows per (sequence, kv head): multi-query attention
(one kv head for 16 or 32 q heads), query groups of 9 to 32, and several
query tokens per sequence (n_q * G <= 32: speculative verification of 4
draft tokens with G = 7 is 28 rows).  Every case is compared element by
element with the fp64 oracle: 16-bit pools (fp16, bf16), E4M3 pools (fp16
and bf16 q), the fused append + decode step, windows, split invariance,
empty and one-token contexts, and NaN in unfilled pool rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi

from _helpers import TOL, to_np16

pytestmark = pytest.mark.gpu


def _case(seed, B, nq, Hq, Hkv, D, max_len, dtype, *, lens=None, nan_fill=False, q_mul=1.0):
    g = torch.Generator().manual_seed(seed)
    if lens is None:
        lens = torch.randint(max(1, nq), max_len + 1, (B,), generator=g)
    lens = torch.as_tensor(lens, dtype=torch.int32)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 3
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, max(1, int(nblk.max()))), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    shape = (B, Hq, D) if nq == 1 else (B, nq, Hq, D)
    # "e4m3": fp16 source pools (quantised by each side), q left in fp32 for the caller
    q = (torch.randn(*shape, generator=g) * q_mul).to(torch.float32 if dtype == "e4m3" else dtype)
    pool_dtype = torch.float16 if dtype == "e4m3" else dtype
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(pool_dtype)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(pool_dtype)
    if nan_fill:
        # rows past each sequence's end hold NaN: they must not reach any output
        for b in range(B):
            L = int(lens[b])
            if L % 16:
                blk = int(tables[b, L // 16])
                kp[blk, :, L % 16:] = float("nan")
                vp[blk, :, L % 16:] = float("nan")
    return q, kp, vp, tables, lens


def _rows(nq, Hq, Hkv):
    return nq * (Hq // Hkv)


@pytest.mark.parametrize("seed,B,nq,Hq,Hkv,D,max_len,window,splits,dtype", [
    (0, 5, 1, 16, 1, 128, 700, 0, 0, torch.float16),      # MQA, 16 heads: two tiles
    (1, 4, 1, 32, 1, 128, 900, 0, 0, torch.float16),      # MQA, 32 heads: four tiles
    (2, 6, 1, 32, 1, 64, 500, 0, 13, torch.bfloat16),
    (3, 5, 1, 16, 1, 64, 300, 0, 3, torch.bfloat16),
    (4, 3, 1, 24, 2, 128, 1200, 0, 304, torch.float16),   # group 12: two tiles, 4 dead columns
    (5, 4, 1, 40, 2, 128, 600, 0, 7, torch.float16),      # group 20: four tiles, 12 dead
    (6, 5, 4, 28, 4, 128, 800, 0, 0, torch.float16),      # 4 tokens x group 7 = 28 rows
    (7, 5, 4, 28, 4, 128, 800, 96, 9, torch.bfloat16),    # ... within a window
    (8, 6, 2, 16, 2, 64, 400, 0, 1, torch.float16),       # 16 rows, one CTA
    (9, 4, 3, 32, 4, 128, 650, 40, 0, torch.float16),     # 24 rows, windowed
    (10, 3, 2, 16, 1, 128, 500, 0, 0, torch.float16),     # MQA with 2 tokens: 32 rows
    (11, 3, 3, 16, 1, 128, 500, 0, 5, torch.float16)])    # 48 rows: passes of 2 and 1 tokens
def test_query_tiles_match_oracle(seed, B, nq, Hq, Hkv, D, max_len, window, splits, dtype):
    q, kp, vp, tables, lens = _case(seed, B, nq, Hq, Hkv, D, max_len, dtype, nan_fill=True)
    scale = float(np.float32(1 / math.sqrt(D)))
    bf16 = dtype == torch.bfloat16
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale,
                        bf16=bf16, window=window)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda", query_rows=_rows(nq, Hq, Hkv))
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(),
                   int(lens.max()), scale, splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= TOL["bf16" if bf16 else "f16"], err
    assert int(ws.count_nonzero()) == 0     # the merge left the workspace zero-filled


@pytest.mark.parametrize("seed,B,nq,Hq,Hkv,D,window,splits,act", [
    (20, 5, 1, 32, 1, 128, 0, 0, torch.float16),
    (21, 4, 1, 16, 1, 64, 0, 11, torch.bfloat16),
    (22, 5, 4, 28, 4, 128, 0, 0, torch.float16),
    (23, 4, 4, 28, 4, 128, 64, 5, torch.bfloat16),
    (24, 3, 1, 24, 2, 128, 0, 2, torch.float16)])
def test_query_tiles_fp8_match_oracle(seed, B, nq, Hq, Hkv, D, window, splits, act):
    # a bf16 q spans a wider range than fp16 holds: scale it up to exercise that
    qm = 1e6 if act == torch.bfloat16 else 1.0
    q, kp, vp, tables, lens = _case(seed, B, nq, Hq, Hkv, D, 900, "e4m3", q_mul=qm)
    q = q.to(act) if act == torch.bfloat16 else q.to(torch.float16)
    kc, ks = oracle.quantize_fp8(to_np16(kp))
    vc, vs = oracle.quantize_fp8(to_np16(vp))
    scale = float(np.float32(1 / math.sqrt(D) / qm))
    bf16 = act == torch.bfloat16
    ref = oracle.decode_fp8(to_np16(q), kc, vc, ks, vs, tables.numpy(), lens.numpy(), scale,
                            bf16=bf16, window=window)
    dev = [torch.from_numpy(x).cuda() for x in (kc, vc, ks, vs)]
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda", query_rows=_rows(nq, Hq, Hkv))
    _abi.pa_decode_fp8(out, q.cuda(), *dev, tables.cuda(), lens.cuda(), int(lens.max()), scale,
                       splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["fp8"]


def _step_inputs(seed, B, Hkv, D, tables, lens, dtype):
    g = torch.Generator().manual_seed(seed + 100)
    kn = torch.randn(B, Hkv, D, generator=g).to(dtype)
    vn = torch.randn(B, Hkv, D, generator=g).to(dtype)
    last = lens.to(torch.int64) - 1
    slots = tables[torch.arange(B), last // 16].to(torch.int64) * 16 + last % 16
    return kn, vn, slots


@pytest.mark.parametrize("seed,Hq,Hkv,D,splits,dtype", [
    (30, 16, 1, 128, 0, torch.float16), (31, 32, 1, 64, 9, torch.bfloat16),
    (32, 40, 2, 128, 3, torch.float16)])
def test_fused_step_query_tiles(seed, Hq, Hkv, D, splits, dtype):
    B = 5
    q, kp, vp, tables, lens = _case(seed, B, 1, Hq, Hkv, D, 700, dtype)
    kn, vn, slots = _step_inputs(seed, B, Hkv, D, tables, lens, dtype)
    k_ref, v_ref = to_np16(kp).copy(), to_np16(vp).copy()
    oracle.cache_append(to_np16(kn), to_np16(vn), k_ref, v_ref, slots.numpy(), 16)
    scale = float(np.float32(1 / math.sqrt(D)))
    bf16 = dtype == torch.bfloat16
    ref = oracle.decode(to_np16(q), k_ref, v_ref, tables.numpy(), lens.numpy(), scale, bf16=bf16)
    kd, vd = kp.cuda(), vp.cuda()
    out = torch.empty_like(q, device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda", query_rows=Hq // Hkv)
    _abi.pa_decode_step(out, q.cuda(), kn.cuda(), vn.cuda(), kd, vd, slots.cuda(), tables.cuda(),
                        lens.cuda(), int(lens.max()), scale, splits, ws)
    assert _abi.pa_get_status() == (0, 0)
    assert np.array_equal(to_np16(kd).view(np.uint16), k_ref.view(np.uint16))
    assert np.array_equal(to_np16(vd).view(np.uint16), v_ref.view(np.uint16))
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["bf16" if bf16 else "f16"]


@pytest.mark.parametrize("seed,Hq,Hkv,D,splits,act", [
    (40, 32, 1, 128, 0, torch.float16), (41, 16, 1, 64, 4, torch.bfloat16)])
def test_fused_step_fp8_query_tiles(seed, Hq, Hkv, D, splits, act):
    B = 4
    q, kp, vp, tables, lens = _case(seed, B, 1, Hq, Hkv, D, 600, "e4m3")
    q = q.to(act)
    kn, vn, slots = _step_inputs(seed, B, Hkv, D, tables, lens, act)
    kc, ks = oracle.quantize_fp8(to_np16(kp))
    vc, vs = oracle.quantize_fp8(to_np16(vp))
    dev = [torch.from_numpy(x.copy()).cuda() for x in (kc, vc, ks, vs)]
    bf16 = act == torch.bfloat16
    oracle.cache_append_fp8(to_np16(kn), to_np16(vn), kc, vc, ks, vs, slots.numpy(), 16, bf16=bf16)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.decode_fp8(to_np16(q), kc, vc, ks, vs, tables.numpy(), lens.numpy(), scale,
                            bf16=bf16)
    out = torch.empty_like(q, device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda", query_rows=Hq // Hkv)
    _abi.pa_decode_step_fp8(out, q.cuda(), kn.cuda(), vn.cuda(), *dev, slots.cuda(),
                            tables.cuda(), lens.cuda(), int(lens.max()), scale, splits, ws)
    assert _abi.pa_get_status() == (0, 0)
    for got, want in zip(dev, (kc, vc, ks, vs)):
        assert np.array_equal(got.cpu().numpy().view(np.uint8), want.view(np.uint8))
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["fp8"]


def test_query_tiles_split_invariance():
    B, Hq, Hkv, D = 6, 32, 1, 128
    q, kp, vp, tables, lens = _case(50, B, 1, Hq, Hkv, D, 1500, torch.float16)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale)
    qd, kd, vd, td, ld = q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda()
    for splits in (1, 2, 7, 64, 304, 999, 5000):   # the last: more warps than blocks
        ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda", query_rows=Hq)
        out = torch.empty_like(qd)
        _abi.pa_decode(out, qd, kd, vd, td, ld, int(lens.max()), scale, splits, ws)
        assert _abi.pa_get_status() == (0, 0)
        assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["f16"], splits


def test_query_tiles_empty_and_single_token_contexts():
    B, Hq, Hkv, D = 4, 32, 1, 64
    q, kp, vp, tables, lens = _case(60, B, 1, Hq, Hkv, D, 0, torch.float16,
                                    lens=[0, 1, 17, 300])
    scale = 0.125
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, 5, "cuda", query_rows=Hq)
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(), 300, scale,
                   5, ws)
    assert _abi.pa_get_status() == (0, 0)
    got = out.float().cpu().numpy()
    assert np.all(got[0] == 0)                                   # L = 0: zeros
    # L = 1: every head returns V[0] of its sequence's first block, rounded once
    v0 = vp[int(tables[1, 0]), 0, 0].float().numpy()
    assert np.array_equal(got[1], np.broadcast_to(v0, got[1].shape))
    assert np.abs(got - ref).max() <= TOL["f16"]


def test_workspace_too_small_for_the_rows_is_refused():
    q, kp, vp, tables, lens = _case(70, 3, 1, 16, 1, 64, 100, torch.float16)
    ws = _abi.alloc_workspace(3, 16, 64, 4, "cuda")           # sized for 8 rows
    with pytest.raises(_abi.PAError) as e:
        _abi.pa_decode(torch.empty_like(q, device="cuda"), q.cuda(), kp.cuda(), vp.cuda(),
                       tables.cuda(), lens.cuda(), int(lens.max()), 0.125, 4, ws)
    assert e.value.code == _abi.PA_ERR_WORKSPACE
