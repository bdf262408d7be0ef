"""Several query tokens per sequence (queries_per_seq > 1): each query
attends causally up to its own position, optionally within a sliding window,
against the oracle's multi-query decode; 16-bit and E4M3 pools, several
CTA splits, sequences shorter than the query count."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi

from _helpers import TOL, to_np16

pytestmark = pytest.mark.gpu


def _case(seed, B, nq, Hq, Hkv, D, max_len, dtype, short=False):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(nq, max_len + 1, (B,), generator=g).to(torch.int32)
    if short:
        lens[0] = 1                      # queries before the cache start
        lens[1] = max(1, nq - 1)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 3
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    q = torch.randn(B, nq, Hq, D, generator=g).to(dtype)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)
    return q, kp, vp, tables, lens


@pytest.mark.parametrize("seed,B,nq,Hq,Hkv,D,max_len,window,splits,dtype,short", [
    (0, 5, 2, 8, 2, 128, 500, 0, 0, torch.float16, False),
    (1, 6, 4, 8, 4, 64, 300, 0, 9, torch.float16, True),
    (2, 4, 8, 4, 4, 128, 700, 0, 304, torch.float16, True),
    (3, 5, 3, 4, 2, 128, 900, 40, 0, torch.bfloat16, False),
    (4, 7, 2, 16, 4, 64, 250, 17, 2, torch.bfloat16, True),
    (5, 3, 4, 2, 1, 128, 2000, 0, 1, torch.float16, False)])
def test_multiquery_matches_oracle(seed, B, nq, Hq, Hkv, D, max_len, window, splits, dtype, short):
    q, kp, vp, tables, lens = _case(seed, B, nq, Hq, Hkv, D, max_len, dtype, short)
    scale = float(np.float32(1 / math.sqrt(D)))
    bf16 = dtype == torch.bfloat16
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale,
                        bf16=bf16, window=window)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda")
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(),
                   int(lens.max()), scale, splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= TOL["bf16" if bf16 else "f16"], err


@pytest.mark.parametrize("nq,window,splits", [(2, 0, 0), (2, 64, 13)])
def test_multiquery_fp8_matches_oracle(nq, window, splits):
    q, kp, vp, tables, lens = _case(9, 5, nq, 16, 4, 128, 800, torch.float16, True)
    kc, ks = oracle.quantize_fp8(to_np16(kp))
    vc, vs = oracle.quantize_fp8(to_np16(vp))
    scale = float(np.float32(1 / math.sqrt(128)))
    ref = oracle.decode_fp8(to_np16(q), kc, vc, ks, vs, tables.numpy(), lens.numpy(), scale,
                            window=window)
    dev = [torch.from_numpy(x).cuda() for x in (kc, vc, ks, vs)]
    out = torch.empty_like(q, device="cuda")
    ws = _abi.alloc_workspace(5, 16, 128, splits, "cuda")
    _abi.pa_decode_fp8(out, q.cuda(), *dev, tables.cuda(), lens.cuda(), int(lens.max()), scale,
                       splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["fp8"]


@pytest.mark.parametrize("seed,nq,Hq,Hkv,window,splits", [
    (10, 3, 28, 4, 0, 0),      # group 7: 21 rows, one pass of four column tiles
    (11, 5, 16, 4, 0, 9),      # group 4: 20 rows, one pass
    (12, 4, 28, 4, 50, 0),     # 28 rows with a sliding window
    (13, 6, 28, 4, 0, 0),      # 42 rows: passes of 4 and 2 tokens
    (14, 9, 16, 4, 30, 5)])    # 36 rows: passes of 8 and 1 tokens, windowed
def test_multiquery_beyond_eight_rows(seed, nq, Hq, Hkv, window, splits):
    q, kp, vp, tables, lens = _case(seed, 5, nq, Hq, Hkv, 128, 600, torch.float16, True)
    scale = float(np.float32(1 / math.sqrt(128)))
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale,
                        window=window)
    out = torch.full_like(q, float("nan"), device="cuda")
    ws = _abi.alloc_workspace(5, Hq, 128, splits, "cuda", query_rows=nq * (Hq // Hkv))
    _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), tables.cuda(), lens.cuda(),
                   int(lens.max()), scale, splits, ws, window=window)
    assert _abi.pa_get_status() == (0, 0)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["f16"]


def test_multiquery_noalloc_rejects_more_than_eight_rows():
    q = torch.zeros(2, 3, 8, 64, dtype=torch.float16, device="cuda")   # 3 tokens x group 4
    k = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    t = torch.zeros(2, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(_abi.PAError) as e:
        _abi.pa_decode_noalloc(torch.empty_like(q), q, k, k, t,
                               torch.ones(2, dtype=torch.int32, device="cuda"), 16, 0.125, 0)
    assert e.value.code == _abi.PA_ERR_UNSUPPORTED
