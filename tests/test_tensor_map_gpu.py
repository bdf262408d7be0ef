"""16-bit pools reach the attention launch through TMA tensor maps that the
library encodes per (pool address, tile count, head_dim) and keeps per host
thread.  Each call must read its own pool's tiles: one address seen through
a short view and then the whole pool, one address seen with head_dim 64 and
then 128, and more pools in turn than the maps kept."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi

from _helpers import TOL, max_err, to_np16

pytestmark = pytest.mark.gpu

HQ, HKV = 8, 2


def _tables(g, lens, blocks):
    """Block tables drawing each sequence's blocks from `blocks` (distinct ids)."""
    nblk = (lens + 15) // 16
    perm = blocks[torch.randperm(len(blocks), generator=g)]
    tables = torch.full((len(lens), int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(len(lens)):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    return tables


def _check(kp, vp, tables, lens, seed):
    """Decode over pools kp / vp (device views) and compare with the oracle."""
    B, D = len(lens), kp.shape[-1]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, HQ, D, generator=g).to(torch.float16)
    scale = float(np.float32(1 / math.sqrt(D)))
    out = torch.full((B, HQ, D), float("nan"), dtype=torch.float16, device="cuda")
    ws = _abi.alloc_workspace(B, HQ, D, 0, "cuda")
    _abi.pa_decode(out, q.cuda(), kp, vp, tables.cuda(), lens.cuda(), int(lens.max()), scale, 0,
                   ws)
    assert _abi.pa_get_status() == (0, 0)
    ref = oracle.decode(to_np16(q), to_np16(kp), to_np16(vp), tables.numpy(), lens.numpy(), scale)
    assert max_err(out, ref) <= TOL["f16"]


def test_short_view_then_whole_pool():
    """The first call sees only the first 8 blocks; the second reads blocks
    past them through the same address (a map kept from the first call
    would cover too few tiles)."""
    g = torch.Generator().manual_seed(3)
    NB, D = 64, 128
    kp = torch.randn(NB, HKV, 16, D, generator=g).to(torch.float16).cuda()
    vp = torch.randn(NB, HKV, 16, D, generator=g).to(torch.float16).cuda()
    lens = torch.tensor([60, 40], dtype=torch.int32)       # 4 + 3 of 8 blocks
    _check(kp[:8], vp[:8], _tables(g, lens, torch.arange(8, dtype=torch.int32)), lens, 1)
    lens = torch.tensor([500, 300], dtype=torch.int32)     # 32 + 19 of 56
    _check(kp, vp, _tables(g, lens, torch.arange(8, NB, dtype=torch.int32)), lens, 2)


def test_same_address_two_head_dims():
    """One allocation read as a head_dim-64 pool, then as a head_dim-128 pool
    with the same number of tiles."""
    g = torch.Generator().manual_seed(4)
    NB = 32
    kraw = torch.randn(NB * HKV * 16 * 128, generator=g).to(torch.float16).cuda()
    vraw = torch.randn(NB * HKV * 16 * 128, generator=g).to(torch.float16).cuda()
    lens = torch.tensor([200, 90, 150], dtype=torch.int32)   # 13 + 6 + 10 of 32
    for D in (64, 128, 64):
        n = NB * HKV * 16 * D
        kp, vp = kraw[:n].view(NB, HKV, 16, D), vraw[:n].view(NB, HKV, 16, D)
        _check(kp, vp, _tables(g, lens, torch.arange(NB, dtype=torch.int32)), lens, 5 + D)


def test_more_pools_than_maps_kept():
    """48 pools in turn, twice over (more than the library keeps, so maps are
    replaced and encoded again)."""
    g = torch.Generator().manual_seed(6)
    NB, D = 12, 64
    pools = [(torch.randn(NB, HKV, 16, D, generator=g).to(torch.float16).cuda(),
              torch.randn(NB, HKV, 16, D, generator=g).to(torch.float16).cuda())
             for _ in range(48)]
    lens = torch.tensor([120, 33], dtype=torch.int32)      # 8 + 3 of 12
    tables = _tables(g, lens, torch.arange(NB, dtype=torch.int32))
    for rep in range(2):
        for i, (kp, vp) in enumerate(pools):
            _check(kp, vp, tables, lens, 100 * rep + i)
