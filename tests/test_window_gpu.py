"""Sliding-window decode (window_size > 0) against the oracle's windowed
decode: 16-bit and E4M3 pools, windows shorter than, inside and longer than
a block and than the context, several CTA splits, the fused step, and the
full Qwen2.5-7B batch on sampled sequences."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import TOL, max_err, to_cuda, to_np16

pytestmark = pytest.mark.gpu


def _case(seed, B, Hq, Hkv, D, max_len, dtype):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, max_len + 1, (B,), generator=g).to(torch.int32)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 3
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    q = torch.randn(B, Hq, D, generator=g).to(dtype)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    return q, kp, vp, tables, lens


@pytest.mark.parametrize("seed,B,Hq,Hkv,D,max_len,window,splits,dtype", [
    (0, 6, 8, 2, 64, 400, 1, 0, torch.float16),
    (1, 5, 28, 4, 128, 700, 15, 7, torch.float16),
    (2, 5, 28, 4, 128, 700, 16, 0, torch.float16),
    (3, 4, 12, 2, 128, 2000, 17, 304, torch.float16),
    (4, 6, 15, 5, 64, 900, 100, 3, torch.bfloat16),
    (5, 3, 8, 2, 128, 300, 1000, 0, torch.float16)])      # wider than every context
def test_window_decode_matches_oracle(seed, B, Hq, Hkv, D, max_len, window, splits, dtype):
    q, kp, vp, tables, lens = _case(seed, B, Hq, Hkv, D, max_len, dtype)
    scale = float(np.float32(1 / math.sqrt(D)))
    bf16 = dtype == torch.bfloat16
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale,
                        bf16=bf16, window=window)
    out = torch.empty(B, Hq, D, dtype=dtype, device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda")
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(),
                   int(lens.max()), scale, splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    assert max_err(out, ref) <= TOL["bf16" if bf16 else "f16"]


@pytest.mark.parametrize("window,splits", [(33, 0), (200, 11)])
def test_window_decode_fp8_matches_oracle(window, splits):
    q, kp, vp, tables, lens = _case(7, 5, 28, 4, 128, 900, torch.float16)
    kc, ks = oracle.quantize_fp8(to_np16(kp))
    vc, vs = oracle.quantize_fp8(to_np16(vp))
    scale = float(np.float32(1 / math.sqrt(128)))
    ref = oracle.decode_fp8(to_np16(q), kc, vc, ks, vs, tables.numpy(), lens.numpy(), scale,
                            window=window)
    dev = [torch.from_numpy(x).cuda() for x in (kc, vc, ks, vs)]
    out = torch.empty_like(q, device="cuda")
    ws = _abi.alloc_workspace(5, 28, 128, splits, "cuda")
    _abi.pa_decode_fp8(out, q.cuda(), *dev, tables.cuda(), lens.cuda(), int(lens.max()), scale,
                       splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["fp8"]


def test_window_fused_step_appends_and_attends():
    w = W.make_workload("qwen2_5_1_5b", seed=3, fill="random")
    window = 300
    kp, vp = to_np16(w.k_cache).copy(), to_np16(w.v_cache).copy()
    oracle.cache_append(to_np16(w.k_new), to_np16(w.v_new), kp, vp, w.slot_mapping.numpy(), 16)
    ref = oracle.decode(to_np16(w.q), kp, vp, w.block_tables.numpy(), w.context_lens.numpy(),
                        w.scale, window=window)
    to_cuda(w)
    step = DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, window=window)
    out = torch.empty_like(w.q)
    step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert _abi.pa_get_status() == (0, 0)
    assert np.array_equal(to_np16(w.k_cache).view(np.uint16), kp.view(np.uint16))
    assert max_err(out, ref) <= TOL["f16"]


def test_window_full_batch_sampled_rows():
    """The Qwen2.5-7B batch with a 1024-token window, the benchmark's launch
    configuration; 32 sampled sequences (the 8 shortest, the 8 longest and
    16 drawn at random) against the oracle on the blocks they read."""
    w = W.make_workload("qwen2_5_7b", seed=0, device="cuda")
    window = 1024
    step = DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, window=window)
    out = torch.empty_like(w.q)
    step(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert _abi.pa_get_status() == (0, 0)
    lens = w.context_lens.cpu().numpy()
    order = np.argsort(lens, kind="stable")
    picked = np.random.default_rng(6).choice(order[8:-8], size=16, replace=False)
    rows = sorted({int(x) for x in np.concatenate([order[:8], order[-8:], picked])})
    assert len(rows) == 32
    sub_t, sub_l, (kp, vp) = W.extract_rows(w.block_tables.cpu().numpy(), lens, rows,
                                            [w.k_cache, w.v_cache])
    ref = oracle.decode(to_np16(w.q[rows]), kp, vp, sub_t, sub_l, w.scale, window=window)
    assert max_err(out[rows], ref) <= TOL["f16"]
