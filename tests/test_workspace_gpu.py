"""The decode workspace: one zero-filled workspace serves calls of different
sizes, split counts, windows, query counts and pool types, each call
leaving it zero-filled for the next (the merge launch zeroes every partial
it reads); a workspace that was not zero-filled is reported
(PA_STATUS_WS_DIRTY) where it matters, and zero-filling it again restores
exact results."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi

from _helpers import TOL, max_err, to_np16

pytestmark = pytest.mark.gpu


def _case(seed, B, Hq, Hkv, D, max_len, nq=1):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(nq, max_len + 1, (B,), generator=g).to(torch.int32)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 5
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    shape = (B, Hq, D) if nq == 1 else (B, nq, Hq, D)
    q = torch.randn(*shape, generator=g).to(torch.float16)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(torch.float16)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(torch.float16)
    return q, kp, vp, tables, lens


# (seed, B, Hq, Hkv, D, max_len, nq, window, splits, fp8): a mix of sizes whose
# partial rows land where earlier calls' flags or partials were
CALLS = [
    (0, 5, 28, 4, 128, 900, 1, 0, 0, False),
    (1, 9, 8, 2, 64, 500, 1, 0, 37, False),
    (2, 3, 12, 2, 128, 2000, 1, 100, 600, False),
    (3, 4, 8, 2, 64, 300, 2, 0, 13, False),
    (4, 6, 28, 4, 128, 700, 1, 0, 0, True),
    (5, 2, 8, 8, 128, 4000, 1, 0, 1, False),
    (6, 7, 16, 2, 64, 800, 1, 0, 4096, False),
]


def _run(ws, seed, B, Hq, Hkv, D, max_len, nq, window, splits, fp8):
    q, kp, vp, tables, lens = _case(seed, B, Hq, Hkv, D, max_len, nq)
    scale = float(np.float32(1 / math.sqrt(D)))
    out = torch.full_like(q, float("nan"), device="cuda")
    args = (tables.cuda(), lens.cuda(), int(lens.max()), scale, splits, ws)
    if fp8:
        kc, ks = oracle.quantize_fp8(to_np16(kp))
        vc, vs = oracle.quantize_fp8(to_np16(vp))
        ref = oracle.decode_fp8(to_np16(q), kc, vc, ks, vs, tables.numpy(), lens.numpy(), scale,
                                window=window)
        dev = [torch.from_numpy(x).cuda() for x in (kc, vc, ks, vs)]
        _abi.pa_decode_fp8(out, q.cuda(), *dev, *args, window=window)
        tol = TOL["fp8"]
    else:
        ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(),
                            scale, window=window)
        _abi.pa_decode(out, q.cuda(), kp.cuda(), vp.cuda(), *args, window=window)
        tol = TOL["f16"]
    return out, ref, tol


def test_one_workspace_serves_calls_of_every_size():
    need = max(_abi.pa_decode_workspace_size(c[1], c[2], c[4], c[8]) for c in CALLS)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(2):                 # and again, in the state the first pass left
        for c in CALLS:
            out, ref, tol = _run(ws, *c)
            assert _abi.pa_get_status() == (0, 0), c
            assert max_err(out, ref) <= tol, c
            assert int(ws.count_nonzero()) == 0, c


def test_dirty_workspace_is_reported_and_zeroing_restores_it():
    """A workspace filled with 0xFF bytes holds what reads as written partials
    (zero maxima and sums).  A partial the merge reads before its piece
    overwrites it is reported (PA_STATUS_WS_DIRTY); one overwritten first does
    no harm; which happens depends on timing.  So the call either reports the
    bit or is exact, and after zero-filling, calls are exact and clean."""
    c = CALLS[0]
    ws = torch.full((_abi.pa_decode_workspace_size(c[1], c[2], c[4], c[8]),), 0xFF,
                    dtype=torch.uint8, device="cuda")
    out, ref, tol = _run(ws, *c)
    rc, bits = _abi.pa_get_status()
    if rc == 0:
        assert max_err(out, ref) <= tol
    else:
        assert rc == _abi.PA_ERR_WORKSPACE and bits == _abi.PA_STATUS_WS_DIRTY, (rc, bits)
    ws.zero_()
    for _ in range(2):
        out, ref, tol = _run(ws, *c)
        assert _abi.pa_get_status() == (0, 0)
        assert max_err(out, ref) <= tol
