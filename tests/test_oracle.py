"""Pins for the oracle, against things other than itself (CPU only).

* E4M3 codec: the OFP8 definition's special values (tests/golden), hand-worked
  ties, torch's float8_e4m3fn conversion (a library routine) over every fp16
  input and a random sample of fp32 bit patterns, and a brute-force nearest-
  value search with ties to even.
* Quantise: torch's E4M3 cast of the fp32 quotient, the amax -> +-448
  invariant, and the half-quantum error bound.
* Append: read-back of every written row and untouched sentinel bytes.
* Decode: a dense materialised softmax(Q K^T * scale) V built from numpy and
  scipy routines (gather, repeat, matmul, softmax) on small shapes, plus the
  invariants context_len=1 -> V[0], constant V -> V, q=0 -> mean of V,
  block relabelling and prefix sharing leave the result unchanged, softmax
  weights sum to 1.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_cache_179_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split()[:2])
    return rows


# ----------------------------------------------------------------- E4M3 codec
def test_e4m3_special_values_from_ofp8():
    rows = _read_golden("e4m3_values.txt")
    assert len(rows) >= 10
    for code, val in rows:
        got = oracle.e4m3_value(np.array([int(code, 16)], dtype=np.uint8))[0]
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e4m3_decode_table_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert nan.sum() == 2   # S.1111.111 only


def test_e4m3_rounding_cases():
    for val, code in _read_golden("e4m3_rounding.txt"):
        got = oracle.e4m3_encode(np.array([float(val)], dtype=np.float32))[0]
        assert got == int(code, 16), (val, hex(got), code)


def _torch_rne(x32: np.ndarray) -> np.ndarray:
    """torch's RNE cast (non-saturating), valid for |x| <= 464 and NaN."""
    return torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _check_against_torch(x32):
    ours = oracle.e4m3_encode(x32)
    with np.errstate(invalid="ignore"):    # signalling-NaN patterns widen with a warning
        a = np.abs(x32.astype(np.float64))
    nan = np.isnan(x32)
    inr = (~nan) & (a <= 448.0)
    ref = _torch_rne(x32)
    assert np.array_equal(ours[inr], ref[inr])
    big = (~nan) & (a > 448.0)
    want_big = np.where(np.signbit(x32[big]), 0xFE, 0x7E).astype(np.uint8)
    assert np.array_equal(ours[big], want_big)
    assert np.all(ours[nan] == 0x7F)


def test_e4m3_encode_every_fp16_input():
    x16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    _check_against_torch(x16.astype(np.float32))


def test_e4m3_encode_random_fp32_bit_patterns():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    _check_against_torch(x)
    # and a dense sample of the interesting range (|x| < 512), where almost all
    # random bit patterns above fall outside
    y = (rng.standard_normal(1 << 21) * 40).astype(np.float32)
    _check_against_torch(y)


def test_e4m3_encode_brute_force_nearest_even():
    """Nearest finite E4M3 value by exhaustive search, ties to the even code."""
    codes = np.arange(0, 0x7F, dtype=np.uint8)          # +0 .. 448, finite, ascending
    vals = oracle.e4m3_value(codes)
    assert np.all(np.diff(vals) > 0)
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(0, 460, 20000), rng.uniform(0, 0.02, 20000),
        (vals[:-1] + vals[1:]) / 2,                        # every exact midpoint
    ]).astype(np.float32)
    ours = oracle.e4m3_encode(x)
    xd = x.astype(np.float64)
    for i in range(x.size):
        d = np.abs(vals - xd[i])
        best = np.flatnonzero(d == d.min())
        want = best[0] if best.size == 1 else best[(codes[best] & 1) == 0][0]
        if xd[i] > 448:
            want = 0x7E
        assert ours[i] == codes[want], (xd[i], ours[i], codes[want])


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


# ------------------------------------------------------------------ quantise
def _pool(NB, Hkv, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((NB, Hkv, 16, D)) * scale).astype(np.float16)


def test_quantize_matches_torch_cast_and_invariants():
    src = _pool(37, 3, 64, 0, scale=2.5)
    src[5, 1] = 0                                  # an all-zero tile
    src[6, 0, 3, 7] = np.float16(60000.0)           # a large outlier
    codes, scales = oracle.quantize_fp8(src)
    x = src.astype(np.float32)
    amax = np.abs(x).max(axis=(2, 3))
    want_s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(scales, want_s)
    assert scales[5, 1] == 1.0 and np.all(codes[5, 1] == 0)
    quot = (x / scales[:, :, None, None]).astype(np.float32)
    assert np.abs(quot).max() <= 448.0 * (1 + 2 ** -20)
    assert np.array_equal(codes, _torch_rne(np.clip(quot, -448, 448)))
    # the amax element of every non-zero tile maps to +-448
    for b in range(src.shape[0]):
        for h in range(src.shape[1]):
            if amax[b, h] == 0:
                continue
            i = np.unravel_index(np.abs(x[b, h]).argmax(), x[b, h].shape)
            assert codes[b, h][i] & 0x7F == 0x7E
    # |dequant - x| <= half a quantum of the code grid, times the scale
    deq = oracle.e4m3_value(codes) * scales[:, :, None, None]
    qa = np.abs(quot.astype(np.float64))
    quantum = np.where(qa < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(qa, 1e-300))) - 3))
    bound = 0.5 * quantum * scales[:, :, None, None] * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)


# -------------------------------------------------------------------- append
def test_append_writes_rows_and_leaves_other_bytes():
    rng = np.random.default_rng(3)
    NB, Hkv, D, T = 12, 3, 64, 9
    k = np.full((NB, Hkv, 16, D), 0xA5A5, dtype=np.uint16).view(np.float16)
    v = k.copy()
    k0, v0 = k.copy(), v.copy()
    kn = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    vn = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    slots = rng.choice(NB * 16, size=T, replace=False).astype(np.int64)
    slots[2] = -1                                   # padding token
    oracle.cache_append(kn, vn, k, v, slots, 16)
    touched = np.zeros((NB, 16), dtype=bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(k[s // 16, :, s % 16].view(np.uint16), kn[i].view(np.uint16))
        assert np.array_equal(v[s // 16, :, s % 16].view(np.uint16), vn[i].view(np.uint16))
        touched[s // 16, s % 16] = True
    untouched = ~touched[:, None, :, None].repeat(Hkv, 1).repeat(D, 3)
    assert np.array_equal(k.view(np.uint16)[untouched], k0.view(np.uint16)[untouched])
    assert np.array_equal(v.view(np.uint16)[untouched], v0.view(np.uint16)[untouched])


def _torch_value(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes -> their fp32 values, by torch's float8_e4m3fn."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).float().numpy()


def test_append_fp8_first_token_sets_scale_reuses_it_then_rescales():
    rng = np.random.default_rng(4)
    Hkv, D, NB = 2, 64, 4
    kc = np.zeros((NB, Hkv, 16, D), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.full((NB, Hkv), -1.0, np.float32)
    vs = ks.copy()
    t0 = rng.standard_normal((1, Hkv, D)).astype(np.float16)
    oracle.cache_append_fp8(t0, t0, kc, vc, ks, vs, np.array([2 * 16]), 16)
    amax = np.abs(t0[0].astype(np.float32)).max(axis=1)
    s0 = amax / np.float32(448)
    assert np.array_equal(ks[2], s0)
    assert np.all(ks[[0, 1, 3]] == -1.0)
    assert np.array_equal(kc[2, :, 0], _torch_rne((t0[0].astype(np.float32) / ks[2][:, None])))
    # second token within the page's range: the scale is reused
    t1 = (t0 * 0.5).astype(np.float16)
    oracle.cache_append_fp8(t1, t1, kc, vc, ks, vs, np.array([2 * 16 + 1]), 16)
    assert np.array_equal(ks[2], s0)
    assert np.array_equal(kc[2, :, 1], _torch_rne(t1[0].astype(np.float32) / s0[:, None]))
    # third token 3x larger: the page is re-scaled to it and its rows re-encoded
    before = kc[2].copy()
    t2 = (t0 * 3).astype(np.float16)
    oracle.cache_append_fp8(t2, t2, kc, vc, ks, vs, np.array([2 * 16 + 2]), 16)
    s1 = np.abs(t2[0].astype(np.float32)).max(axis=1) / np.float32(448)
    assert np.array_equal(ks[2], s1) and np.array_equal(vs[2], s1)
    for h in range(Hkv):
        old = (_torch_value(before[h, :2]) * s0[h]).astype(np.float32)
        assert np.array_equal(kc[2, h, :2], _torch_rne((old / s1[h]).astype(np.float32)))
        x = t2[0, h].astype(np.float32)
        assert np.array_equal(kc[2, h, 2], _torch_rne(x / s1[h]))
        assert np.abs(_torch_value(kc[2, h, 2])).max() == 448.0     # the row's amax, unsaturated
    assert np.array_equal(kc[2, :, 3:], before[:, 3:])             # rows past the new one
    # after two roundings every stored value stays within twice E4M3's bound of its token
    for row, t in ((0, t0), (1, t1), (2, t2)):
        x = t[0].astype(np.float64)
        got = _torch_value(kc[2, :, row]).astype(np.float64) * s1[:, None]
        bound = 2 * (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s1[:, None])
        assert np.all(np.abs(got - x) <= bound + 1e-12)


def test_append_fp8_bf16_rows():
    rng = np.random.default_rng(6)
    Hkv, D, NB = 2, 128, 2
    x = rng.standard_normal((2, Hkv, D)).astype(np.float32) * 5
    bits = (torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()).view(np.uint16)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    kc = np.zeros((NB, Hkv, 16, D), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((NB, Hkv), np.float32)
    vs = ks.copy()
    oracle.cache_append_fp8(bits, bits, kc, vc, ks, vs, np.array([16, 17]), 16, bf16=True)
    s = np.maximum(np.abs(xb[0]).max(axis=1), np.abs(xb[1]).max(axis=1)) / np.float32(448)
    assert np.array_equal(ks[1], s)
    assert np.array_equal(kc[1, :, 1], _torch_rne(xb[1] / s[:, None]))


# -------------------------------------------------------------------- decode
def _dense(q, k_pool, v_pool, tables, lens, scale):
    """Materialised softmax(q K^T * scale) V, per sequence, from numpy/scipy routines."""
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        phys = tables[b, t // 16]
        K = k_pool[phys, :, t % 16, :]                      # [L][Hkv][D]
        V = v_pool[phys, :, t % 16, :]
        K = np.repeat(K, Hq // Hkv, axis=1).transpose(1, 0, 2)   # [Hq][L][D]
        V = np.repeat(V, Hq // Hkv, axis=1).transpose(1, 0, 2)
        S = np.einsum("hd,hld->hl", q[b], K) * scale
        P = scipy.special.softmax(S, axis=1)
        out[b] = np.einsum("hl,hld->hd", P, V)
    return out


def _f64(a):
    if a.dtype == np.uint16:                                   # bf16 bits
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _random_case(rng, B, Hq, Hkv, D, max_len, bf16=False, NB=None):
    lens = rng.integers(1, max_len + 1, size=B).astype(np.int32)
    nblk = (lens + 15) // 16
    NB = NB or int(nblk.sum() + 5)
    perm = rng.permutation(NB).astype(np.int32)
    mbs = int(nblk.max())
    tables = np.full((B, mbs), -1, np.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += nblk[b]

    def draw(shape):
        x = rng.standard_normal(shape).astype(np.float32)
        if bf16:
            return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return x.astype(np.float16)
    return draw((B, Hq, D)), draw((NB, Hkv, 16, D)), draw((NB, Hkv, 16, D)), tables, lens


@pytest.mark.parametrize("B,Hq,Hkv,D,bf16", [
    (3, 8, 2, 64, False), (2, 7, 1, 128, False), (4, 15, 5, 64, True), (2, 28, 4, 128, False),
    (2, 12, 2, 128, False), (2, 4, 4, 64, True),
    # multi-query and groups above 8 (one kv head for 16 or 32 q heads; groups of 12 and 20)
    (2, 16, 1, 128, False), (2, 32, 1, 64, True), (3, 24, 2, 128, False), (2, 40, 2, 64, False)])
def test_decode_matches_dense_softmax(B, Hq, Hkv, D, bf16):
    rng = np.random.default_rng(B * 100 + Hq)
    q, kp, vp, tables, lens = _random_case(rng, B, Hq, Hkv, D, 300, bf16)
    scale = float(np.float32(1 / math.sqrt(D)))
    got, wsum = oracle.decode(q, kp, vp, tables, lens, scale, bf16=bf16, return_wsum=True)
    want = _dense(_f64(q), _f64(kp), _f64(vp), tables, lens, scale)
    assert np.abs(got - want).max() < 1e-12
    assert wsum.max() < 1e-12


def test_dense_pin_discriminates_head_mapping():
    """The dense statement distinguishes consecutive grouping from a modulo mapping."""
    rng = np.random.default_rng(11)
    q, kp, vp, tables, lens = _random_case(rng, 2, 8, 2, 64, 100)
    got = oracle.decode(q, kp, vp, tables, lens, 0.125)
    kp2 = kp[:, ::-1].copy()       # swapping the two kv heads = the other mapping of 8 q heads
    vp2 = vp[:, ::-1].copy()
    other = _dense(_f64(q), _f64(kp2), _f64(vp2), tables, lens, 0.125)
    assert np.abs(got - other).max() > 1e-2


def test_decode_invariants():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D = 4, 8, 2, 64
    q, kp, vp, tables, lens = _random_case(rng, B, Hq, Hkv, D, 200)
    scale = 0.125
    # context_len = 1 returns V[0] of the right kv head
    l1 = np.ones(B, np.int32)
    out = oracle.decode(q, kp, vp, tables, l1, scale)
    for b in range(B):
        for hq in range(Hq):
            assert np.array_equal(out[b, hq], vp[tables[b, 0], hq // (Hq // Hkv), 0].astype(np.float64))
    # constant V returns that constant
    vc = np.full_like(vp, np.float16(0.37))
    out = oracle.decode(q, kp, vc, tables, lens, scale)
    assert np.abs(out - np.float64(np.float16(0.37))).max() < 1e-14
    # q = 0 gives the mean of V over the context
    out = oracle.decode(np.zeros_like(q), kp, vp, tables, lens, scale)
    for b in range(B):
        t = np.arange(lens[b])
        V = vp[tables[b, t // 16], :, t % 16, :].astype(np.float64)
        for hq in range(Hq):
            assert np.abs(out[b, hq] - V[:, hq // (Hq // Hkv)].mean(axis=0)).max() < 1e-13
    # context_len = 0 gives zeros
    out = oracle.decode(q, kp, vp, tables, np.zeros(B, np.int32), scale)
    assert not out.any()
    # relabelling physical blocks (permute the pool, rewrite the tables) changes nothing
    base = oracle.decode(q, kp, vp, tables, lens, scale)
    NB = kp.shape[0]
    perm = rng.permutation(NB)
    inv = np.argsort(perm)
    t2 = np.where(tables >= 0, inv[np.maximum(tables, 0)], -1).astype(np.int32)
    out = oracle.decode(q, kp[perm], vp[perm], t2, lens, scale)
    assert np.array_equal(out, base)


def test_shared_prefix_equals_copied_blocks():
    w = W.make_workload("smollm2_360m", seed=2)
    tables = w.block_tables.numpy()
    lens = w.context_lens.numpy()
    rows = [0, 1, 17]
    sub_t, sub_l, (kp, vp) = W.extract_rows(tables, lens, rows, [w.k_cache, w.v_cache])
    q = W.to_numpy16(w.q)[rows]
    shared = oracle.decode(q, kp, vp, sub_t, sub_l, w.scale, bf16=True)
    # give sequence 1 private copies of the 32 shared blocks
    n_sh = len(w.shared_blocks)
    assert n_sh == 32 and np.array_equal(sub_t[0, :n_sh], sub_t[1, :n_sh])
    extra = np.arange(kp.shape[0], kp.shape[0] + n_sh, dtype=np.int32)
    kp2 = np.concatenate([kp, kp[sub_t[1, :n_sh]]])
    vp2 = np.concatenate([vp, vp[sub_t[1, :n_sh]]])
    t2 = sub_t.copy()
    t2[1, :n_sh] = extra
    copied = oracle.decode(q, kp2, vp2, t2, sub_l, w.scale, bf16=True)
    assert np.array_equal(shared, copied)


def test_copy_blocks_invariants():
    rng = np.random.default_rng(8)
    NB, Hkv, D = 10, 2, 64
    k = rng.standard_normal((NB, Hkv, 16, D)).astype(np.float16)
    v = rng.standard_normal((NB, Hkv, 16, D)).astype(np.float16)
    ks = rng.random((NB, Hkv)).astype(np.float32)
    vs = rng.random((NB, Hkv)).astype(np.float32)
    k0, v0, ks0, vs0 = k.copy(), v.copy(), ks.copy(), vs.copy()
    pairs = np.array([[1, 7], [4, 4], [2, 9], [12, 3], [0, -1]], dtype=np.int64)
    oracle.copy_blocks(k, v, pairs, ks, vs)
    for src, dst in ((1, 7), (2, 9)):                # applied pairs
        assert np.array_equal(k[dst].view(np.uint16), k0[src].view(np.uint16))
        assert np.array_equal(v[dst].view(np.uint16), v0[src].view(np.uint16))
        assert np.array_equal(ks[dst], ks0[src]) and np.array_equal(vs[dst], vs0[src])
    rest = [b for b in range(NB) if b not in (7, 9)]  # self-copy and out-of-range pairs: no-ops
    for a, a0 in ((k, k0), (v, v0)):
        assert np.array_equal(a[rest].view(np.uint16), a0[rest].view(np.uint16))
    assert np.array_equal(ks[rest], ks0[rest]) and np.array_equal(vs[rest], vs0[rest])
    # pairs apply in order: a chain carries the first source along
    c = np.arange(4 * 16 * 8, dtype=np.uint8).reshape(4, 1, 16, 8)
    c0 = c.copy()
    d = c.copy()
    oracle.copy_blocks(c, d, np.array([[0, 1], [1, 2]]))
    assert np.array_equal(c[2], c0[0]) and np.array_equal(d[2], c0[0])


def test_copy_on_write_fork_keeps_attention():
    """Forking a sequence's shared prefix into fresh blocks (the block
    manager's copy-on-write) leaves its attention output unchanged."""
    w = W.make_workload("smollm2_360m", seed=4)
    tables = w.block_tables.numpy()
    lens = w.context_lens.numpy()
    rows = [0, 1]
    sub_t, sub_l, (kp, vp) = W.extract_rows(tables, lens, rows, [w.k_cache, w.v_cache])
    q = W.to_numpy16(w.q)[rows]
    before = oracle.decode(q, kp, vp, sub_t, sub_l, w.scale, bf16=True)
    n_sh = len(w.shared_blocks)
    fresh = np.arange(kp.shape[0], kp.shape[0] + n_sh, dtype=np.int64)
    kp2 = np.concatenate([kp, np.zeros_like(kp[:n_sh])])
    vp2 = np.concatenate([vp, np.zeros_like(vp[:n_sh])])
    oracle.copy_blocks(kp2, vp2, np.stack([sub_t[1, :n_sh].astype(np.int64), fresh], axis=1))
    t2 = sub_t.copy()
    t2[1, :n_sh] = fresh
    assert np.array_equal(oracle.decode(q, kp2, vp2, t2, sub_l, w.scale, bf16=True), before)


def test_decode_fp8_matches_dense_on_dequantised_pool():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, D = 3, 28, 4, 128
    q, kp, vp, tables, lens = _random_case(rng, B, Hq, Hkv, D, 250)
    kc, ks = oracle.quantize_fp8(kp)
    vc, vs = oracle.quantize_fp8(vp)
    scale = float(np.float32(1 / math.sqrt(D)))
    got, wsum = oracle.decode_fp8(q, kc, vc, ks, vs, tables, lens, scale, return_wsum=True)
    kd = oracle.e4m3_value(kc) * ks[:, :, None, None].astype(np.float64)
    vd = oracle.e4m3_value(vc) * vs[:, :, None, None].astype(np.float64)
    want = _dense(q.astype(np.float64), kd, vd, tables, lens, scale)
    assert np.abs(got - want).max() < 1e-12
    assert wsum.max() < 1e-12
    # quantisation error against the unquantised pool is small but not zero
    ref = oracle.decode(q, kp, vp, tables, lens, scale)
    err = np.abs(got - ref)
    assert 1e-5 < err.mean() < 2e-2


def test_decode_fp8_bf16_query_matches_dense():
    rng = np.random.default_rng(10)
    B, Hq, Hkv, D = 2, 12, 2, 128
    q, kp, vp, tables, lens = _random_case(rng, B, Hq, Hkv, D, 90)
    kc, ks = oracle.quantize_fp8(kp)
    vc, vs = oracle.quantize_fp8(vp)
    qb = torch.from_numpy(q.astype(np.float32) * 3).to(torch.bfloat16)
    qbits = qb.view(torch.int16).numpy().view(np.uint16)
    scale = float(np.float32(1 / math.sqrt(D)))
    got = oracle.decode_fp8(qbits, kc, vc, ks, vs, tables, lens, scale, bf16=True)
    kd = oracle.e4m3_value(kc) * ks[:, :, None, None].astype(np.float64)
    vd = oracle.e4m3_value(vc) * vs[:, :, None, None].astype(np.float64)
    want = _dense(qb.float().numpy().astype(np.float64), kd, vd, tables, lens, scale)
    assert np.abs(got - want).max() < 1e-12


def _last_tokens_relaid(kp, vp, tables, lens, b, W):
    """Sequence b's last W tokens copied, in order, to fresh blocks starting at
    position 0 (pure data movement): (k pool, v pool, table row, length)."""
    L = int(lens[b])
    lo = max(0, L - W)
    n = L - lo
    nb = (n + 15) // 16
    k2 = np.zeros((nb,) + kp.shape[1:], kp.dtype)
    v2 = np.zeros_like(k2)
    for j in range(n):
        t = lo + j
        k2[j // 16, :, j % 16] = kp[tables[b, t // 16], :, t % 16]
        v2[j // 16, :, j % 16] = vp[tables[b, t // 16], :, t % 16]
    return k2, v2, np.arange(nb, dtype=np.int32)[None, :], np.array([n], np.int32)


@pytest.mark.parametrize("W", [1, 5, 16, 33, 100, 1000])
def test_window_equals_global_decode_of_the_last_tokens(W):
    rng = np.random.default_rng(20 + W)
    B, Hq, Hkv, D = 4, 8, 2, 64
    q, kp, vp, tables, lens = _random_case(rng, B, Hq, Hkv, D, 300)
    got = oracle.decode(q, kp, vp, tables, lens, 0.125, window=W)
    for b in range(B):
        k2, v2, t2, l2 = _last_tokens_relaid(kp, vp, tables, lens, b, W)
        want = oracle.decode(q[b:b + 1], k2, v2, t2, l2, 0.125)
        assert np.array_equal(got[b], want[0]), (W, b)
    if W >= lens.max():
        assert np.array_equal(got, oracle.decode(q, kp, vp, tables, lens, 0.125))


def test_window_of_one_token_returns_its_value():
    rng = np.random.default_rng(31)
    q, kp, vp, tables, lens = _random_case(rng, 3, 4, 2, 64, 200)
    got = oracle.decode(q, kp, vp, tables, lens, 0.125, window=1)
    for b in range(3):
        t = int(lens[b]) - 1
        v = vp[tables[b, t // 16], :, t % 16].astype(np.float64)
        assert np.array_equal(got[b], np.repeat(v, 2, axis=0))


@pytest.mark.parametrize("nq,W,fp8", [(2, 0, False), (4, 0, False), (3, 20, False),
                                      (4, 0, True), (2, 9, True)])
def test_query_tokens_equal_single_queries_at_their_positions(nq, W, fp8):
    """Query i of a sequence with L tokens is the single-query decode of the
    same cache with length L - nq + i + 1 (its position plus one)."""
    rng = np.random.default_rng(40 + nq + W)
    B, Hq, Hkv, D = 3, 8, 2, 128
    _, kp, vp, tables, lens = _random_case(rng, B, Hq, Hkv, D, 150)
    lens = np.maximum(lens, nq).astype(np.int32)
    q = rng.standard_normal((B, nq, Hq, D)).astype(np.float16)
    if fp8:
        kc, ks = oracle.quantize_fp8(kp)
        vc, vs = oracle.quantize_fp8(vp)
        run = lambda qq, ll: oracle.decode_fp8(qq, kc, vc, ks, vs, tables, ll, 0.125, window=W)
    else:
        run = lambda qq, ll: oracle.decode(qq, kp, vp, tables, ll, 0.125, window=W)
    got = run(q, lens)
    assert got.shape == q.shape
    for i in range(nq):
        want = run(np.ascontiguousarray(q[:, i]), (lens - nq + i + 1).astype(np.int32))
        assert np.array_equal(got[:, i], want), i
    # a query whose position precedes the cache gets zeros
    short = np.array([1, 2, 3], np.int32)
    z = run(q, short)
    for b in range(B):
        assert np.all(z[b, :max(0, nq - int(short[b]))] == 0)


def test_rows_subset_matches_full():
    rng = np.random.default_rng(12)
    q, kp, vp, tables, lens = _random_case(rng, 5, 8, 2, 64, 120)
    full = oracle.decode(q, kp, vp, tables, lens, 0.125)
    part = oracle.decode(q, kp, vp, tables, lens, 0.125, rows=[3, 1])
    assert np.array_equal(part[[1, 3]], full[[1, 3]])
    assert not part[[0, 2, 4]].any()
