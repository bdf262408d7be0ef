"""pa_decode_step / pa_decode_step_fp8: append and decode in one launch,
against the oracle's append followed by its decode.  Pools must come out
bit-identical to the oracle's append; outputs within the decode tolerances."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import TOL, max_err, oracle_step, to_cuda, to_np16

pytestmark = pytest.mark.gpu


def _step(w, splits=0, **pools):
    pools = pools or dict(k_cache=w.k_cache, v_cache=w.v_cache)
    return DecodeStep(**pools, block_tables=w.block_tables, context_lens=w.context_lens,
                      max_context_len=w.max_context_len, scale=w.scale, num_q_heads=w.Hq,
                      split_ctas=splits)


@pytest.mark.parametrize("name,seed,splits", [("tiny", 0, 0), ("tiny", 1, 7),
                                              ("smollm2_360m", 0, 0), ("qwen2_5_1_5b", 1, 0),
                                              ("qwen2_5_7b", 0, 0), ("qwen2_5_7b", 2, 1000)])
def test_fused_step_matches_oracle(name, seed, splits):
    w = W.make_workload(name, seed=seed, fill="random")
    kp, vp = to_np16(w.k_cache).copy(), to_np16(w.v_cache).copy()
    oracle.cache_append(to_np16(w.k_new), to_np16(w.v_new), kp, vp, w.slot_mapping.numpy(), 16)
    ref = oracle.decode(to_np16(w.q), kp, vp, w.block_tables.numpy(), w.context_lens.numpy(),
                        w.scale, bf16=(w.dtype == "bf16"))
    to_cuda(w)
    out = torch.empty_like(w.q)
    _step(w, splits).fused(w.q, w.k_new, w.v_new, w.slot_mapping, out)
    assert _abi.pa_get_status() == (0, 0)
    assert np.array_equal(to_np16(w.k_cache).view(np.uint16), kp.view(np.uint16))
    assert np.array_equal(to_np16(w.v_cache).view(np.uint16), vp.view(np.uint16))
    assert max_err(out, ref) <= TOL[w.dtype]


def test_fused_equals_append_then_decode():
    w = to_cuda(W.make_workload("qwen2_5_1_5b", seed=3))
    k0, v0 = w.k_cache.clone(), w.v_cache.clone()
    a = torch.empty_like(w.q)
    _step(w)(w.q, w.k_new, w.v_new, w.slot_mapping, a, fused=False)
    w.k_cache.copy_(k0)
    w.v_cache.copy_(v0)
    b = torch.empty_like(w.q)
    _step(w)(w.q, w.k_new, w.v_new, w.slot_mapping, b, fused=True)
    assert (a.float() - b.float()).abs().max().item() <= TOL["f16"]


def test_padding_and_mismatched_slots():
    w = to_cuda(W.make_workload("tiny", seed=4))
    slots = w.slot_mapping.clone()
    slots[1] = -1                        # padding: nothing appended for sequence 1
    slots[2] = slots[2] + 1              # not position L-1: reported, not written
    k0 = w.k_cache.clone()
    out = torch.empty_like(w.q)
    _step(w).fused(w.q, w.k_new, w.v_new, slots, out)
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_BOUNDS and bits == _abi.PA_STATUS_BAD_SLOT
    changed = (w.k_cache != k0).flatten(1).any(dim=1).nonzero().flatten().tolist()
    s0, s3 = int(w.slot_mapping[0]), int(w.slot_mapping[3])
    assert set(changed) <= {s0 // 16, s3 // 16}
    assert torch.equal(w.k_cache[s0 // 16, :, s0 % 16], w.k_new[0])
    assert torch.equal(w.k_cache[s3 // 16, :, s3 % 16], w.k_new[3])


def _fp8_case(seed, B, Hq, Hkv, D, lens, dtype=torch.float16):
    g = torch.Generator().manual_seed(seed)
    lens = torch.tensor(lens, dtype=torch.int32)
    nblk = (lens + 15) // 16
    NB = int(nblk.sum()) + 3
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    tables = torch.full((B, int(nblk.max())), -1, dtype=torch.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += int(nblk[b])
    last = lens.to(torch.int64) - 1
    slots = tables[torch.arange(B), last // 16].to(torch.int64) * 16 + last % 16
    q = torch.randn(B, Hq, D, generator=g).to(dtype)
    kp = torch.randn(NB, Hkv, 16, D, generator=g).to(torch.float16)
    vp = torch.randn(NB, Hkv, 16, D, generator=g).to(torch.float16)
    # rows at and after each sequence's new position hold no token yet
    for b in range(B):
        for j in range(int(nblk[b])):
            r0 = max(0, int(lens[b]) - 1 - 16 * j)
            if r0 < 16:
                kp[tables[b, j], :, r0:] = 0
                vp[tables[b, j], :, r0:] = 0
    # new rows larger than the pool's: most later rows re-scale their page
    kn = (torch.randn(B, Hkv, D, generator=g) * 2).to(dtype)
    vn = (torch.randn(B, Hkv, D, generator=g) * 2).to(dtype)
    return q, kp, vp, kn, vn, tables, lens, slots


@pytest.mark.parametrize("seed,B,Hq,Hkv,D,lens,splits,dtype", [
    (0, 5, 28, 4, 128, [17, 33, 300, 1, 129], 0, torch.float16),  # new rows opening pages
    (1, 4, 8, 2, 64, [20, 50, 77, 200], 9, torch.float16),        # new rows inside pages
    (2, 6, 12, 2, 128, [1, 16, 17, 32, 48, 1000], 2, torch.float16),
    (3, 5, 28, 4, 128, [18, 35, 300, 2, 130], 0, torch.bfloat16),
    (4, 4, 8, 2, 64, [21, 50, 76, 200], 5, torch.bfloat16)])
def test_fused_step_fp8_matches_oracle(seed, B, Hq, Hkv, D, lens, splits, dtype):
    q, kp, vp, kn, vn, tables, L, slots = _fp8_case(seed, B, Hq, Hkv, D, lens, dtype)
    kc, ks = oracle.quantize_fp8(to_np16(kp))
    vc, vs = oracle.quantize_fp8(to_np16(vp))
    dev = [torch.from_numpy(x.copy()).cuda() for x in (kc, vc, ks, vs)]
    bf16 = dtype == torch.bfloat16
    oracle.cache_append_fp8(to_np16(kn), to_np16(vn), kc, vc, ks, vs, slots.numpy(), 16, bf16=bf16)
    scale = float(np.float32(1 / math.sqrt(D)))
    ref = oracle.decode_fp8(to_np16(q), kc, vc, ks, vs, tables.numpy(), L.numpy(), scale,
                            bf16=bf16)
    out = torch.empty(B, Hq, D, dtype=dtype, device="cuda")
    ws = _abi.alloc_workspace(B, Hq, D, splits, "cuda")
    _abi.pa_decode_step_fp8(out, q.cuda(), kn.cuda(), vn.cuda(), *dev, slots.cuda(),
                            tables.cuda(), L.cuda(), int(L.max()), scale, splits, ws)
    assert _abi.pa_get_status() == (0, 0)
    for got, want in zip(dev, (kc, vc, ks, vs)):
        assert np.array_equal(got.cpu().numpy().view(np.uint8), want.view(np.uint8))
    assert np.abs(out.float().cpu().numpy() - ref).max() <= TOL["fp8"]


def test_run_from_staging_matches_device_call():
    """The end-to-end form: inputs packed in one pinned buffer, one upload,
    the output copied back; the same bytes as the step on device inputs."""
    from paged_kv_cache_179_gb300.step import StepStaging
    w = W.make_workload("qwen2_5_1_5b", seed=7)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    staging = StepStaging({k: (getattr(w, k).shape, getattr(w, k).dtype) for k in names}, "cuda")
    for k in names:
        staging.host[k].copy_(getattr(w, k))
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    k2, v2 = kc.clone(), vc.clone()
    step = DecodeStep(k_cache=kc, v_cache=vc, block_tables=staging.dev["block_tables"],
                      context_lens=staging.dev["context_lens"], max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq)
    host_out = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    h2d, d2h = step.run_from_staging(staging, host_out, torch.empty_like(w.q, device="cuda"))
    torch.cuda.synchronize()
    assert h2d >= sum(getattr(w, k).numel() * getattr(w, k).element_size() for k in names)
    assert d2h == w.q.numel() * 2
    to_cuda(w)
    ref_step = DecodeStep(k_cache=k2, v_cache=v2, block_tables=w.block_tables,
                          context_lens=w.context_lens, max_context_len=w.max_context_len,
                          scale=w.scale, num_q_heads=w.Hq)
    ref = torch.empty_like(w.q)
    ref_step(w.q, w.k_new, w.v_new, w.slot_mapping, ref)
    assert _abi.pa_get_status() == (0, 0)
    assert torch.equal(host_out.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(kc.view(torch.int16), k2.view(torch.int16))


@pytest.mark.parametrize("handshake", ["events", "device"])
def test_step_pipeline_overlapped_copies_match_direct_calls(handshake):
    """StepPipeline: two slots with different queries, five steps submitted
    back to back; every read-back equals the step called directly on the
    same inputs (the appended rows are the same each step)."""
    from paged_kv_cache_179_gb300.step import StepPipeline
    w = W.make_workload("qwen2_5_1_5b", seed=8)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    specs = {k: (getattr(w, k).shape, getattr(w, k).dtype) for k in names}
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    k2, v2 = kc.clone(), vc.clone()

    def make_step(st):
        return DecodeStep(k_cache=kc, v_cache=vc, block_tables=st.dev["block_tables"],
                          context_lens=st.dev["context_lens"], max_context_len=w.max_context_len,
                          scale=w.scale, num_q_heads=w.Hq)
    pipe = StepPipeline(make_step, specs, w.q.shape, w.q.dtype, "cuda", handshake=handshake)
    assert pipe.uses_device_handshake() == (handshake == "device")
    g = torch.Generator().manual_seed(1)
    qs = [torch.randn(w.q.shape, generator=g).to(w.q.dtype) for _ in range(2)]
    for k, st in enumerate(pipe.stagings):
        for n in names:
            st.host[n].copy_(qs[k] if n == "q" else getattr(w, n))
    got = []
    for _ in range(5):
        k, _, _ = pipe.submit()
        pipe.read_back[k].synchronize()
        got.append((k, pipe.host_out[k].clone()))
    pipe.finish()
    torch.cuda.synchronize()
    to_cuda(w)
    ref_step = DecodeStep(k_cache=k2, v_cache=v2, block_tables=w.block_tables,
                          context_lens=w.context_lens, max_context_len=w.max_context_len,
                          scale=w.scale, num_q_heads=w.Hq)
    refs = []
    for k in range(2):
        r = torch.empty_like(w.q)
        ref_step(qs[k].cuda(), w.k_new, w.v_new, w.slot_mapping, r)
        refs.append(r.cpu())
    assert _abi.pa_get_status() == (0, 0)
    assert [k for k, _ in got] == [0, 1, 0, 1, 0]
    for k, out in got:
        assert torch.equal(out.view(torch.int16), refs[k].view(torch.int16))
    assert torch.equal(kc.view(torch.int16), k2.view(torch.int16))


def test_bound_step_records_once_and_matches_direct_calls():
    """DecodeStep.bind: recording launches nothing; each call of the bound
    step equals a direct step on the same inputs, pools included."""
    w = to_cuda(W.make_workload("qwen2_5_1_5b", seed=11))
    k2, v2 = w.k_cache.clone(), w.v_cache.clone()
    step = DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq)
    ref_step = DecodeStep(k_cache=k2, v_cache=v2, block_tables=w.block_tables,
                          context_lens=w.context_lens, max_context_len=w.max_context_len,
                          scale=w.scale, num_q_heads=w.Hq)
    for fused in (True, False):
        out = torch.full_like(w.q, float("nan"))
        call = step.bind(w.q, w.k_new, w.v_new, w.slot_mapping, out, fused=fused)
        torch.cuda.synchronize()
        assert torch.isnan(out).all()              # nothing ran while recording
        ref = torch.empty_like(w.q)
        for _ in range(2):
            call()
            ref_step(w.q, w.k_new, w.v_new, w.slot_mapping, ref, fused=fused)
            assert _abi.pa_get_status() == (0, 0)
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(w.k_cache.view(torch.int16), k2.view(torch.int16))
        assert torch.equal(w.v_cache.view(torch.int16), v2.view(torch.int16))


@pytest.mark.parametrize("handshake,shared", [("events", False), ("device", False),
                                              ("events", True), ("device", True)])
def test_step_pipeline_early_prologue_new_lengths_each_step(handshake, shared):
    """StepPipeline with the early prologue: every step uploads new context
    lengths and slots (one token more each step), so a prologue that read
    its slot's lengths before that upload had landed would attend the wrong
    contexts.  The uploads are ordered before the step by events, which the
    early prologue does not relax: the outputs and pools must equal plain
    direct steps on the same inputs, step by step.  With the device-side
    handshake the attention launch itself waits for the upload's word.
    ``shared``: both slots' steps use one split-K workspace."""
    from paged_kv_cache_179_gb300.step import StepPipeline
    STEPS = 6
    name = "qwen2_5_1_5b"
    B = W.CONFIGS[name]["B"]
    g = torch.Generator().manual_seed(3)
    lens0 = (torch.randint(2, 100, (B,), generator=g) * 16
             + torch.randint(1, 16 - STEPS + 1, (B,), generator=g))
    w = W.make_workload(name, seed=9, lens_override=lens0.tolist(), fill="random")
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    specs = {k: (getattr(w, k).shape, getattr(w, k).dtype) for k in names}
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    k2, v2 = kc.clone(), vc.clone()
    max_ctx = int(lens0.max()) + STEPS
    tables = w.block_tables
    inputs = []
    for n in range(STEPS):
        lens = (lens0 + n).to(torch.int32)
        last = lens.to(torch.int64) - 1
        slots = tables[torch.arange(B), last // 16].to(torch.int64) * 16 + last % 16
        inputs.append(dict(q=torch.randn(w.q.shape, generator=g).to(w.q.dtype),
                           k_new=torch.randn(w.k_new.shape, generator=g).to(w.q.dtype),
                           v_new=torch.randn(w.k_new.shape, generator=g).to(w.q.dtype),
                           slot_mapping=slots, block_tables=tables, context_lens=lens))

    made = []

    def make_step(st):
        s = DecodeStep(k_cache=kc, v_cache=vc, block_tables=st.dev["block_tables"],
                       context_lens=st.dev["context_lens"], max_context_len=max_ctx,
                       scale=w.scale, num_q_heads=w.Hq, early_prologue=True,
                       workspace=made[0].workspace if shared and made else None)
        made.append(s)
        return s
    pipe = StepPipeline(make_step, specs, w.q.shape, w.q.dtype, "cuda", handshake=handshake)
    assert pipe.uses_device_handshake() == (handshake == "device")
    assert (made[0].workspace.data_ptr() == made[1].workspace.data_ptr()) == shared
    got = [None] * STEPS
    pending = None
    for n in range(STEPS):
        pipe.wait_slot_free()
        if pending is not None and pending[1] == pipe.slot():
            pipe.read_back[pending[1]].synchronize()
            got[pending[0]] = pipe.host_out[pending[1]].clone()
            pending = None
        for k in names:
            pipe.stagings[pipe.slot()].host[k].copy_(inputs[n][k])
        slot, _, _ = pipe.submit()
        if pending is not None:
            pipe.read_back[pending[1]].synchronize()
            got[pending[0]] = pipe.host_out[pending[1]].clone()
        pending = (n, slot)
    pipe.finish()
    torch.cuda.synchronize()
    got[pending[0]] = pipe.host_out[pending[1]].clone()
    assert _abi.pa_get_status() == (0, 0)

    lens_d = torch.empty(B, dtype=torch.int32, device="cuda")
    ref_step = DecodeStep(k_cache=k2, v_cache=v2, block_tables=tables.cuda(), context_lens=lens_d,
                          max_context_len=max_ctx, scale=w.scale, num_q_heads=w.Hq)
    for n in range(STEPS):
        lens_d.copy_(inputs[n]["context_lens"])
        r = torch.empty_like(w.q, device="cuda")
        d = {k: inputs[n][k].cuda() for k in ("q", "k_new", "v_new", "slot_mapping")}
        ref_step(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], r)
        assert torch.equal(got[n].view(torch.int16), r.cpu().view(torch.int16)), n
    assert torch.equal(kc.view(torch.int16), k2.view(torch.int16))


def test_step_rejects_a_workspace_too_small():
    """DecodeStep(workspace=...): a buffer smaller than the launch's split-K
    workspace is refused before anything runs."""
    w = to_cuda(W.make_workload("qwen2_5_1_5b", seed=12))
    kw = dict(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
              context_lens=w.context_lens, max_context_len=w.max_context_len,
              scale=w.scale, num_q_heads=w.Hq)
    full = DecodeStep(**kw)
    n = full.workspace.numel() * full.workspace.element_size()
    assert n > 4096
    with pytest.raises(ValueError):
        DecodeStep(**kw, workspace=torch.zeros(n - 16, dtype=torch.uint8, device="cuda"))
    ok = DecodeStep(**kw, workspace=full.workspace)
    assert ok.workspace.data_ptr() == full.workspace.data_ptr()
