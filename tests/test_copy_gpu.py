"""pa_copy_blocks against the oracle's block copy: bit-exact pools (and E4M3
scales) after the copy, for 16-bit and E4M3 pools, with the edge cases:
no pairs, self-copies, pairs outside the pool (skipped and reported)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi

pytestmark = pytest.mark.gpu


def _pool(g, NB, Hkv, D, dtype):
    if dtype == torch.uint8:
        return torch.randint(0, 256, (NB, Hkv, 16, D), generator=g, dtype=torch.uint8)
    return torch.randn(NB, Hkv, 16, D, generator=g).to(dtype)


def _pairs(g, NB, n):
    """n pairs with distinct destinations, none of them a source."""
    perm = torch.randperm(NB, generator=g)
    dst = perm[:n]
    src = perm[n:][torch.randint(0, NB - n, (n,), generator=g)]
    return torch.stack([src, dst], dim=1).to(torch.int64)


def _np(t):
    t = t.cpu()
    return t.view(torch.int16).numpy() if t.dtype in (torch.float16, torch.bfloat16) else t.numpy()


@pytest.mark.parametrize("NB,Hkv,D,dtype,n", [(64, 2, 64, torch.float16, 9),
                                              (300, 4, 128, torch.bfloat16, 100),
                                              (300, 4, 128, torch.uint8, 77),
                                              (16384, 2, 128, torch.float16, 4096)])
def test_copy_blocks_matches_oracle(NB, Hkv, D, dtype, n):
    g = torch.Generator().manual_seed(NB + n)
    k, v = _pool(g, NB, Hkv, D, dtype), _pool(g, NB, Hkv, D, dtype)
    pairs = _pairs(g, NB, n)
    fp8 = dtype == torch.uint8
    ks = torch.rand(NB, Hkv, generator=g) if fp8 else None
    vs = torch.rand(NB, Hkv, generator=g) if fp8 else None
    dev = [t.cuda() if t is not None else None for t in (k, v, ks, vs)]
    _abi.pa_copy_blocks(dev[0], dev[1], pairs.cuda(), dev[2], dev[3])
    ref = [_np(t).copy() if t is not None else None for t in (k, v, ks, vs)]
    oracle.copy_blocks(ref[0], ref[1], pairs.numpy(), ref[2], ref[3])
    assert _abi.pa_get_status() == (0, 0)
    for got, want in zip(dev, ref):
        if got is not None:
            assert np.array_equal(_np(got), want)


def test_copy_blocks_edge_cases():
    g = torch.Generator().manual_seed(1)
    NB, Hkv, D = 32, 2, 64
    k, v = _pool(g, NB, Hkv, D, torch.float16), _pool(g, NB, Hkv, D, torch.float16)
    kd, vd = k.cuda(), v.cuda()
    _abi.pa_copy_blocks(kd, vd, torch.empty(0, 2, dtype=torch.int64, device="cuda"))
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
    pairs = torch.tensor([[3, 3], [5, 40], [-2, 7], [6, 8]], dtype=torch.int64)
    _abi.pa_copy_blocks(kd, vd, pairs.cuda())
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_BOUNDS and bits == _abi.PA_STATUS_BAD_BLOCK
    ref_k, ref_v = _np(k).copy(), _np(v).copy()
    oracle.copy_blocks(ref_k, ref_v, pairs.numpy())
    assert np.array_equal(_np(kd), ref_k) and np.array_equal(_np(vd), ref_v)
    assert not np.array_equal(ref_k[8], _np(k)[8])      # the valid pair did copy
