"""E4M3 path on the GPU against the oracle: the encoder over every fp32 bit
pattern, bulk page quantisation and FP8 append bit-exact, and pa_decode_fp8
within 3e-2 of the oracle on the dequantised pool (small shapes whole, the
256-sequence 4k-32k batch on sampled sequences)."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import TOL, to_np16

pytestmark = pytest.mark.gpu


def test_encoder_every_fp32_bit_pattern():
    chunk = 1 << 28
    x = torch.empty(chunk, dtype=torch.int32, device="cuda")
    codes = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    base = torch.arange(chunk, dtype=torch.int64, device="cuda")
    for start in range(0, 1 << 32, chunk):
        v = base + start
        x.copy_(torch.where(v >= (1 << 31), v - (1 << 32), v).to(torch.int32))
        xf = x.view(torch.float32)
        _abi.pa_e4m3_encode(xf, codes)
        got = codes.cpu().numpy()
        want = oracle.e4m3_encode(xf.cpu().numpy())
        nan = np.isnan(xf.cpu().numpy())
        # NaN inputs: any NaN code (S.1111.111) is right; everything else bit-exact
        assert np.all((got[nan] & 0x7F) == 0x7F), start
        bad = np.flatnonzero(got[~nan] != want[~nan])
        assert bad.size == 0, (start, bad[:5])


def _fp16_pool(NB, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(NB, Hkv, 16, D, generator=g) * 3).to(torch.float16)
    x[0, 0] = 0                                        # all-zero tile -> scale 1
    x[1, 0, 5, 3] = 65504.0                            # fp16 max
    x[2, 1] = (torch.randn(16, D, generator=g) * 1e-6).to(torch.float16)   # subnormal tile
    x[3, 0, 0, 0] = -0.0
    return x


@pytest.mark.parametrize("D", [64, 128])
def test_quantize_bit_exact(D):
    src_k, src_v = _fp16_pool(301, 3, D, 0), _fp16_pool(301, 3, D, 1)
    kc_o, ks_o = oracle.quantize_fp8(to_np16(src_k))
    vc_o, vs_o = oracle.quantize_fp8(to_np16(src_v))
    kd, vd = src_k.cuda(), src_v.cuda()
    kc = torch.empty(kd.shape, dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    ks = torch.empty(301, 3, dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    _abi.pa_quantize_fp8(kd, vd, kc, vc, ks, vs)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), ks_o.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), vs_o.view(np.uint32))
    assert np.array_equal(kc.cpu().numpy(), kc_o)
    assert np.array_equal(vc.cpu().numpy(), vc_o)


@pytest.mark.parametrize("D,dtype", [(64, torch.float16), (128, torch.float16),
                                     (128, torch.bfloat16)])
def test_append_fp8_bit_exact(D, dtype):
    g = torch.Generator().manual_seed(2)
    NB, Hkv = 9, 2
    kc = torch.randint(0, 256, (NB, Hkv, 16, D), generator=g, dtype=torch.uint8)
    vc = kc.clone()
    ks = torch.rand(NB, Hkv, generator=g) + 0.01
    vs = ks.clone()
    # call 1: first tokens of pages 2 and 5, and a later token of page 7 (existing scale)
    # call 2: the second token of page 2 and a padding token
    calls = [torch.tensor([2 * 16, 5 * 16, 7 * 16 + 9]), torch.tensor([2 * 16 + 1, -1])]
    ref = [a.numpy().copy() for a in (kc, vc, ks, vs)]
    dev = [a.cuda() for a in (kc, vc, ks, vs)]
    for i, slots in enumerate(calls):
        T = slots.numel()
        kn = (torch.randn(T, Hkv, D, generator=g) * (1 + 3 * i)).to(dtype)
        vn = (torch.randn(T, Hkv, D, generator=g) * (1 + 3 * i)).to(dtype)
        oracle.cache_append_fp8(to_np16(kn), to_np16(vn), *ref, slots.numpy(), 16,
                                bf16=dtype == torch.bfloat16)
        _abi.pa_cache_append_fp8(kn.cuda(), vn.cuda(), *dev, slots.cuda())
    assert _abi.pa_get_status() == (0, 0)
    for r, d in zip(ref, dev):
        assert np.array_equal(d.cpu().numpy().view(np.uint8), r.view(np.uint8))


@pytest.mark.parametrize("D,dtype", [(128, torch.float16), (64, torch.bfloat16)])
def test_append_fp8_rescales_a_page_token_by_token(D, dtype):
    """A page filled one token per call, magnitudes rising and falling, so that
    some tokens fit the page's scale and others re-scale its earlier rows."""
    g = torch.Generator().manual_seed(5)
    NB, Hkv = 3, 2
    kc = torch.zeros(NB, Hkv, 16, D, dtype=torch.uint8)
    vc = kc.clone()
    ks = torch.ones(NB, Hkv)
    vs = ks.clone()
    ref = [a.numpy().copy() for a in (kc, vc, ks, vs)]
    dev = [a.cuda() for a in (kc, vc, ks, vs)]
    mags = [1, 0.5, 3, 2, 40, 1, 0.01, 500, 7, 1e3, 1e3, 0, 2e3, 1, 5e4, 1]
    rescaled = 0
    for row, m in enumerate(mags):
        m = m if dtype == torch.bfloat16 else min(m, 2e3)   # fp16 rows stay finite
        kn = (torch.randn(1, Hkv, D, generator=g) * m).to(dtype)
        vn = (torch.randn(1, Hkv, D, generator=g) * m * 0.5).to(dtype)
        before = ref[2].copy()
        slots = torch.tensor([1 * 16 + row])
        oracle.cache_append_fp8(to_np16(kn), to_np16(vn), *ref, slots.numpy(), 16,
                                bf16=dtype == torch.bfloat16)
        _abi.pa_cache_append_fp8(kn.cuda(), vn.cuda(), *dev, slots.cuda())
        rescaled += int(row > 0 and not np.array_equal(before[1], ref[2][1]))
        for r_, d_ in zip(ref, dev):
            assert np.array_equal(d_.cpu().numpy().view(np.uint8), r_.view(np.uint8)), row
    assert _abi.pa_get_status() == (0, 0)
    assert rescaled >= 4


def _fp8_step(w, kc, vc, ks, vs, splits=0):
    return DecodeStep(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, split_ctas=splits)


def _quantized_on_gpu(w):
    kc = torch.empty(w.k_cache.shape, dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    ks = torch.empty(w.num_blocks, w.Hkv, dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    _abi.pa_quantize_fp8(w.k_cache, w.v_cache, kc, vc, ks, vs)
    return kc, vc, ks, vs


@pytest.mark.parametrize("seed,B,Hq,Hkv,D,max_len,splits,dtype", [
    (0, 4, 28, 4, 128, 700, 13, torch.float16), (1, 3, 8, 2, 64, 300, 40, torch.float16),
    (2, 5, 12, 2, 128, 2000, 304, torch.float16), (3, 2, 7, 7, 128, 50, 1, torch.float16),
    (4, 4, 28, 4, 128, 900, 0, torch.bfloat16), (5, 3, 8, 2, 64, 300, 7, torch.bfloat16)])
def test_decode_fp8_small_matches_oracle(seed, B, Hq, Hkv, D, max_len, splits, dtype):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, max_len + 1, (B,), generator=g).to(torch.int32)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 2
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    # a bf16 q spans a wider range than fp16 holds: scale it up to exercise that
    q = (torch.randn(B, Hq, D, generator=g) * (1e6 if dtype == torch.bfloat16 else 1)).to(dtype)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(torch.float16)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(torch.float16)
    scale = float(np.float32(1 / math.sqrt(D) / (1e6 if dtype == torch.bfloat16 else 1)))
    kc_o, ks_o = oracle.quantize_fp8(to_np16(kp))
    vc_o, vs_o = oracle.quantize_fp8(to_np16(vp))
    ref = oracle.decode_fp8(to_np16(q), kc_o, vc_o, ks_o, vs_o, tables.numpy(), lens.numpy(), scale,
                            bf16=dtype == torch.bfloat16)
    kc, vc = torch.from_numpy(kc_o).cuda(), torch.from_numpy(vc_o).cuda()
    ks, vs = torch.from_numpy(ks_o).cuda(), torch.from_numpy(vs_o).cuda()
    out = torch.empty(B, Hq, D, dtype=dtype, device="cuda")
    mcl = int(lens.max())
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda")
    _abi.pa_decode_fp8(out, q.cuda(), kc, vc, ks, vs, tables.cuda(), lens.cuda(), mcl, scale,
                       splits, ws)
    assert _abi.pa_get_status() == (0, 0)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= TOL["fp8"], err


def test_fp8_full_batch_sampled_rows():
    """The 256-sequence E4M3 batch at full size, in the benchmark's launch
    configuration: quantise on the GPU (checked bit-exact on the sampled
    sequences' pages), append + decode, and compare 32 sampled sequences --
    the 8 longest (32k-token contexts split across many warps), the 8
    shortest and 16 drawn at random -- with the oracle run from the fp16
    source of those pages."""
    w = W.make_workload("qwen2_5_7b_fp8", seed=0, device="cuda")
    lens = w.context_lens.cpu().numpy()
    kc, vc, ks, vs = _quantized_on_gpu(w)
    step = _fp8_step(w, kc, vc, ks, vs)
    out = torch.empty_like(w.q)
    step(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert _abi.pa_get_status() == (0, 0)
    order = np.argsort(lens, kind="stable")
    rest = order[8:-8]
    picked = np.random.default_rng(5).choice(rest, size=16, replace=False)
    rows = sorted({int(x) for x in np.concatenate([order[:8], order[-8:], picked])})
    assert len(rows) == 32
    tables = w.block_tables.cpu().numpy()
    sub_t, sub_l, (kp, vp) = W.extract_rows(tables, lens, rows, [w.k_cache, w.v_cache])
    # oracle side: quantise the fp16 source pages, then append the new tokens
    kc_o, ks_o = oracle.quantize_fp8(kp)
    vc_o, vs_o = oracle.quantize_fp8(vp)
    # the GPU's codes for those pages must be the oracle's (bit-exact quantiser)
    seen = {}
    for b in rows:
        for pid in tables[b, :(int(lens[b]) + 15) // 16].tolist():
            seen.setdefault(int(pid), len(seen))
    order_ids = list(seen)
    ids = torch.tensor(order_ids, device="cuda")
    slot_rows = w.slot_mapping.cpu().numpy()[rows]
    # the new token rewrites one row of each sampled page: compare all other pages
    last_pages = {int(s) // 16 for s in slot_rows}
    keep = [i for i, pid in enumerate(order_ids) if pid not in last_pages]
    kc_g = kc.index_select(0, ids).cpu().numpy()
    assert np.array_equal(kc_g[keep], kc_o[keep])
    # oracle append of the new tokens into the compact pool
    remap = {pid: i for i, pid in enumerate(order_ids)}
    sub_slots = np.array([remap[int(s) // 16] * 16 + int(s) % 16 for s in slot_rows], np.int64)
    oracle.cache_append_fp8(to_np16(w.k_new[rows]), to_np16(w.v_new[rows]), kc_o, vc_o, ks_o,
                            vs_o, sub_slots, 16)
    ref = oracle.decode_fp8(to_np16(w.q[rows]), kc_o, vc_o, ks_o, vs_o, sub_t, sub_l, w.scale)
    err = np.abs(out[rows].float().cpu().numpy() - ref).max()
    assert err <= TOL["fp8"], err


def test_fp8_full_pool_quantiser_bit_exact():
    """pa_quantize_fp8 over the whole E4M3 batch's pools (about 325k pages of
    each of K and V), compared code for code and scale for scale with the
    oracle's quantiser, in chunks of 32768 pages."""
    w = W.make_workload("qwen2_5_7b_fp8", seed=1, device="cuda")
    kc, vc, ks, vs = _quantized_on_gpu(w)
    assert _abi.pa_get_status() == (0, 0)
    chunk = 32768
    for src, codes, scales in ((w.k_cache, kc, ks), (w.v_cache, vc, vs)):
        for p0 in range(0, w.num_blocks, chunk):
            p1 = min(w.num_blocks, p0 + chunk)
            c_o, s_o = oracle.quantize_fp8(to_np16(src[p0:p1]))
            assert np.array_equal(codes[p0:p1].cpu().numpy(), c_o), p0
            assert np.array_equal(scales[p0:p1].cpu().numpy().view(np.uint32),
                                  s_o.view(np.uint32)), p0
