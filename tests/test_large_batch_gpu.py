"""Batches above the 512 sequences one launch takes: the call splits them into
consecutive launch pairs that share the workspace.  Checked against the
oracle for the plain decode, a sliding window with two query tokens, the
fused step and an E4M3 pool, and for the static-scratch entry point."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi

from _helpers import TOL, to_np16

pytestmark = pytest.mark.gpu

B = 1100          # three launches: 512 + 512 + 76


def _case(seed, Hq, Hkv, D, max_len, nq=1, dtype=torch.float16):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(nq, max_len + 1, (B,), generator=g).to(torch.int32)
    lens[::97] = 0                                   # some empty sequences
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 7
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, max(1, int(nblk.max()))), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    shape = (B, Hq, D) if nq == 1 else (B, nq, Hq, D)
    q = torch.randn(*shape, generator=g).to(dtype)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    return q, kp, vp, tables, lens


@pytest.mark.parametrize("nq,window,splits", [(1, 0, 0), (2, 24, 0), (1, 0, 37)])
def test_large_batch_decode(nq, window, splits):
    Hq, Hkv, D = 8, 2, 64
    q, kp, vp, tables, lens = _case(1 + nq, Hq, Hkv, D, 90, nq)
    scale = 0.125
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale,
                        window=window)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda")
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(),
                   int(lens.max()), scale, splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["f16"]


def test_large_batch_fused_step():
    Hq, Hkv, D = 8, 2, 64
    q, kp, vp, tables, lens = _case(5, Hq, Hkv, D, 90)
    g = torch.Generator().manual_seed(6)
    kn = torch.randn(B, Hkv, D, generator=g).to(torch.float16)
    vn = torch.randn(B, Hkv, D, generator=g).to(torch.float16)
    last = lens.to(torch.int64) - 1
    rows = torch.arange(B)
    slots = torch.where(lens > 0, tables[rows, (last.clamp(min=0) // 16)].to(torch.int64) * 16
                        + last.clamp(min=0) % 16, torch.full_like(last, -1))
    k_ref, v_ref = to_np16(kp).copy(), to_np16(vp).copy()
    oracle.cache_append(to_np16(kn), to_np16(vn), k_ref, v_ref, slots.numpy(), 16)
    ref = oracle.decode(to_np16(q), k_ref, v_ref, tables.numpy(), lens.numpy(), 0.125)
    kd, vd = kp.cuda(), vp.cuda()
    out = torch.empty_like(q, device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, 0, "cuda")
    _abi.pa_decode_step(out, q.cuda(), kn.cuda(), vn.cuda(), kd, vd, slots.cuda(), tables.cuda(),
                        lens.cuda(), int(lens.max()), 0.125, 0, ws)
    assert _abi.pa_get_status() == (0, 0)
    assert np.array_equal(to_np16(kd).view(np.uint16), k_ref.view(np.uint16))
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["f16"]


def test_large_batch_fp8_and_noalloc():
    Hq, Hkv, D = 8, 2, 128
    q, kp, vp, tables, lens = _case(8, Hq, Hkv, D, 60)
    kc, ks = oracle.quantize_fp8(to_np16(kp))
    vc, vs = oracle.quantize_fp8(to_np16(vp))
    scale = float(np.float32(1 / math.sqrt(D)))
    ref8 = oracle.decode_fp8(to_np16(q), kc, vc, ks, vs, tables.numpy(), lens.numpy(), scale)
    dev = [torch.from_numpy(x).cuda() for x in (kc, vc, ks, vs)]
    out = torch.empty_like(q, device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, 0, "cuda")
    _abi.pa_decode_fp8(out, q.cuda(), *dev, tables.cuda(), lens.cuda(), int(lens.max()), scale,
                       0, ws)
    assert _abi.pa_get_status() == (0, 0)
    assert np.abs(out.float().cpu().numpy() - ref8).max() <= TOL["fp8"]
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale)
    out2 = torch.empty_like(q, device="cuda")
    _abi.pa_decode_noalloc(out2, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(),
                           int(lens.max()), scale, 0)
    assert _abi.pa_get_status() == (0, 0)
    assert np.abs(out2.float().cpu().numpy() - ref).max() <= TOL["f16"]
