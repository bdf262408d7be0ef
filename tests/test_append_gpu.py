"""pa_cache_append on the GPU against the oracle: bit-exact, whole pools."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W

from _helpers import to_cuda, to_np16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "smollm2_360m", "qwen2_5_1_5b", "qwen2_5_7b"])
def test_append_bit_exact_whole_pool(name):
    w = W.make_workload(name, seed=1, fill="random")
    kp, vp = to_np16(w.k_cache).copy(), to_np16(w.v_cache).copy()
    oracle.cache_append(to_np16(w.k_new), to_np16(w.v_new), kp, vp, w.slot_mapping.numpy(), 16)
    to_cuda(w)
    _abi.pa_cache_append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    assert _abi.pa_get_status() == (0, 0)
    assert np.array_equal(to_np16(w.k_cache).view(np.uint16), kp.view(np.uint16))
    assert np.array_equal(to_np16(w.v_cache).view(np.uint16), vp.view(np.uint16))


@pytest.mark.parametrize("dtype,D", [(torch.float16, 128), (torch.bfloat16, 64), (torch.float16, 8)])
def test_append_sentinel_padding_and_ragged(dtype, D):
    g = torch.Generator().manual_seed(5)
    NB, Hkv, T = 37, 3, 53                         # T not a multiple of anything
    k = torch.full((NB, Hkv, 16, D), -23131, dtype=torch.int16).view(dtype)   # 0xA5A5
    v = k.clone()
    kn = torch.randn(T, Hkv, D, generator=g).to(dtype)
    vn = torch.randn(T, Hkv, D, generator=g).to(dtype)
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
    slots[::7] = -1                                # padding tokens
    kr, vr = to_np16(k).copy(), to_np16(v).copy()
    oracle.cache_append(to_np16(kn), to_np16(vn), kr, vr, slots.numpy(), 16)
    kd, vd = k.cuda(), v.cuda()
    _abi.pa_cache_append(kn.cuda(), vn.cuda(), kd, vd, slots.cuda())
    assert _abi.pa_get_status() == (0, 0)
    assert np.array_equal(to_np16(kd).view(np.uint16), kr.view(np.uint16))
    assert np.array_equal(to_np16(vd).view(np.uint16), vr.view(np.uint16))


def test_append_empty_batch_is_noop():
    k = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    e = torch.zeros(0, 2, 64, dtype=torch.float16, device="cuda")
    _abi.pa_cache_append(e, e, k, k.clone(), torch.zeros(0, dtype=torch.int64, device="cuda"))
    assert not k.any()


def test_append_out_of_range_slot_is_skipped_and_reported():
    k = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    v = torch.zeros_like(k)
    kn = torch.ones(2, 2, 64, dtype=torch.float16, device="cuda")
    slots = torch.tensor([4 * 16, 3], dtype=torch.int64, device="cuda")   # first is one past the pool
    _abi.pa_cache_append(kn, kn, k, v, slots)
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_BOUNDS and bits == _abi.PA_STATUS_BAD_SLOT
    assert k[0, :, 3].eq(1).all() and k.sum().item() == 2 * 64
    assert _abi.pa_get_status() == (0, 0)         # reading clears the word
