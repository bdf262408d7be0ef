"""The device-side handshake of a decode step with copies on other streams.

pa_decode_step_synced waits on the device for a word that the upload's
stream writes after the step's inputs, and signals a second word once its
output is complete, so that a serving loop's compute stream holds only the
steps' kernels.  The pipelined end-to-end tests (test_step_gpu.py) check its
results step by step; these check the pieces: stream-ordered word writes and
waits, the done signal of a step with nothing to attend, a step whose upload
never arrives (its attention launch gives up after the 2 s limit, reports a
timeout, and the step still signals done, so a stream waiting on it never
waits forever), the one-call pipelined step over E4M3 pools, and a
pipelined call whose step is refused (it queues no wait for a done word).
"""
import ctypes
import time

import pytest
import torch

from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import to_cuda

pytestmark = pytest.mark.gpu


def _sync(words, ready_value, done_value):
    sy = _abi.StepSync()
    sy.ready = words[0].data_ptr()
    sy.done = words[8].data_ptr()
    sy.done_count = words[16].data_ptr()
    sy.ready_value = ready_value
    sy.done_value = done_value
    return sy


def test_stream_value_write_and_wait_keep_their_order():
    words = torch.zeros(8, dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(a):
        torch.cuda._sleep(20_000_000)                    # about 10 ms of GPU time first
    _abi.pa_stream_write_value(words[:1], 5, a)
    _abi.pa_stream_wait_value(words[:1], 5, b)
    with torch.cuda.stream(b):
        out.copy_(words[:1])                             # only after the write
    b.synchronize()
    assert int(out.item()) == 5
    # the wait compares cyclically: a later value satisfies an earlier wait
    _abi.pa_stream_write_value(words[:1], 7, a)
    _abi.pa_stream_wait_value(words[:1], 6, b)
    b.synchronize()


def test_synced_step_equals_plain_step():
    w = to_cuda(W.make_workload("qwen2_5_1_5b", seed=4))
    k2, v2 = w.k_cache.clone(), w.v_cache.clone()
    step = DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq)
    ref_step = DecodeStep(k_cache=k2, v_cache=v2, block_tables=w.block_tables,
                          context_lens=w.context_lens, max_context_len=w.max_context_len,
                          scale=w.scale, num_q_heads=w.Hq)
    words = torch.zeros(32, dtype=torch.int32, device="cuda")
    out, ref = torch.empty_like(w.q), torch.empty_like(w.q)
    _abi.pa_stream_write_value(words[:1], 3)             # the inputs are already in place
    step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, out, sync=_sync(words, 3, 9))
    ref_step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, ref)
    assert _abi.pa_get_status() == (0, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(w.k_cache.view(torch.int16), k2.view(torch.int16))
    assert int(words[8]) == 9 and int(words[16]) == 0    # done signalled, count reset


def test_synced_empty_batch_signals_done():
    words = torch.zeros(32, dtype=torch.int32, device="cuda")
    z3 = torch.empty(0, 8, 64, dtype=torch.float16, device="cuda")
    pool = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    _abi.pa_decode_step(z3, z3, torch.empty(0, 2, 64, dtype=torch.float16, device="cuda"),
                        torch.empty(0, 2, 64, dtype=torch.float16, device="cuda"), pool, pool,
                        torch.empty(0, dtype=torch.int64, device="cuda"),
                        torch.empty(0, 1, dtype=torch.int32, device="cuda"),
                        torch.empty(0, dtype=torch.int32, device="cuda"), 16, 0.125, 4,
                        torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"),
                        sync=_sync(words, 1, 12))
    torch.cuda.synchronize()
    assert int(words[8]) == 12


def test_synced_step_without_upload_times_out_and_still_signals_done():
    w = to_cuda(W.make_workload("tiny", seed=2))
    step = DecodeStep(k_cache=w.k_cache, v_cache=w.v_cache, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, split_ctas=6)
    words = torch.zeros(32, dtype=torch.int32, device="cuda")
    out = torch.full_like(w.q, 7.0)
    k0 = w.k_cache.clone()
    back = torch.cuda.Stream()
    t = time.perf_counter()
    step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, out, sync=_sync(words, 1, 5))
    _abi.pa_stream_wait_value(words[8:9], 5, back)       # the read-back stream's wait
    back.synchronize()
    dt = time.perf_counter() - t
    rc, bits = _abi.pa_get_status()
    assert rc == _abi.PA_ERR_TIMEOUT and bits & _abi.PA_STATUS_TIMEOUT, (rc, bits)
    assert dt < 10.0, dt
    assert int(words[8]) == 5 and int(words[16]) == 0
    assert bool(torch.all(out == 7.0))                   # nothing attended, nothing written
    assert torch.equal(w.k_cache.view(torch.int16), k0.view(torch.int16))   # nothing appended
    # the context still works and a plain step afterwards is exact
    step.workspace.zero_()
    out2 = torch.empty_like(w.q)
    step.fused(w.q, w.k_new, w.v_new, w.slot_mapping, out2)
    assert _abi.pa_get_status() == (0, 0)
    assert bool(torch.isfinite(out2.float()).all())


def test_synced_call_argument_checks():
    w = to_cuda(W.make_workload("tiny", seed=0))
    ws = _abi.alloc_workspace(w.B, w.Hq, w.D, 4, "cuda")
    words = torch.zeros(32, dtype=torch.int32, device="cuda")
    bad = _sync(words, 1, 1)
    bad.done_count = None
    with pytest.raises(_abi.PAError) as e:
        _abi.pa_decode_step(torch.empty_like(w.q), w.q, w.k_new, w.v_new, w.k_cache, w.v_cache,
                            w.slot_mapping, w.block_tables, w.context_lens, w.max_context_len,
                            w.scale, 4, ws, sync=bad)
    assert e.value.code == _abi.PA_ERR_INVALID_ARG


def test_pipelined_fp8_steps_match_direct_calls():
    """StepPipeline over E4M3 pools with fused steps, each step one library
    call (pa_decode_step_fp8_pipelined): every step uploads new lengths,
    slots, rows and queries; outputs, codes and page scales must equal the
    same fused steps called directly, step by step."""
    from paged_kv_cache_179_gb300.step import StepPipeline
    STEPS = 5
    name = "qwen2_5_1_5b"
    B = W.CONFIGS[name]["B"]
    g = torch.Generator().manual_seed(21)
    lens0 = (torch.randint(2, 60, (B,), generator=g) * 16
             + torch.randint(1, 16 - STEPS + 1, (B,), generator=g))
    w = W.make_workload(name, seed=5, lens_override=lens0.tolist())
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    specs = {k: (getattr(w, k).shape, getattr(w, k).dtype) for k in names}
    kp, vp = w.k_cache.cuda(), w.v_cache.cuda()
    kc = torch.empty(kp.shape, dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    ks = torch.empty(w.num_blocks, w.Hkv, dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    _abi.pa_quantize_fp8(kp, vp, kc, vc, ks, vs)
    ref_pools = [t.clone() for t in (kc, vc, ks, vs)]
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

    def make_step(st):
        return DecodeStep(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs,
                          block_tables=st.dev["block_tables"],
                          context_lens=st.dev["context_lens"], max_context_len=max_ctx,
                          scale=w.scale, num_q_heads=w.Hq, early_prologue=True)
    pipe = StepPipeline(make_step, specs, w.q.shape, w.q.dtype, "cuda")
    assert pipe.uses_device_handshake(fused=True)
    got = []
    for n in range(STEPS):
        pipe.wait_slot_free()
        for k in names:
            pipe.stagings[pipe.slot()].host[k].copy_(inputs[n][k])
        slot, _, _ = pipe.submit(fused=True)
        pipe.read_back[slot].synchronize()
        got.append(pipe.host_out[slot].clone())
    pipe.finish()
    torch.cuda.synchronize()
    assert _abi.pa_get_status() == (0, 0)

    rk, rv, rks, rvs = ref_pools
    lens_d = torch.empty(B, dtype=torch.int32, device="cuda")
    ref_step = DecodeStep(k_cache=rk, v_cache=rv, k_scale=rks, v_scale=rvs,
                          block_tables=tables.cuda(), context_lens=lens_d,
                          max_context_len=max_ctx, scale=w.scale, num_q_heads=w.Hq)
    for n in range(STEPS):
        lens_d.copy_(inputs[n]["context_lens"])
        r = torch.empty_like(w.q, device="cuda")
        d = {k: inputs[n][k].cuda() for k in ("q", "k_new", "v_new", "slot_mapping")}
        ref_step.fused(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], r)
        assert torch.equal(got[n].view(torch.int16), r.cpu().view(torch.int16)), n
    for a, b in zip((kc, vc, ks, vs), (rk, rv, rks, rvs)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_pipelined_step_refused_launch_queues_no_wait():
    """A pipelined call whose step cannot be launched (here: q heads not a
    multiple of kv heads) returns the error after its upload and before it
    queues the wait for a done word that would never come: the read-back
    stream stays free."""
    w = to_cuda(W.make_workload("tiny", seed=1))
    words = torch.zeros(32, dtype=torch.int32, device="cuda")
    sy = _sync(words, 1, 1)
    host_in = torch.zeros(4096, dtype=torch.uint8).pin_memory()
    dev_in = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(w.q)
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    copy, back = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    ev.record(back)
    io = _abi.StepCopies(host_in.data_ptr(), dev_in.data_ptr(), 4096, out.data_ptr(),
                         host_out.data_ptr(), out.numel() * out.element_size(),
                         copy.cuda_stream, back.cuda_stream, ev.cuda_event, 0)
    ws = _abi.alloc_workspace(w.B, w.Hq, w.D, 4, "cuda")
    lib = _abi.load()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.pa_decode_step_pipelined(
        P(out), P(w.q), P(w.k_new), P(w.v_new), P(w.k_cache), P(w.v_cache), P(w.slot_mapping),
        P(w.block_tables), w.block_tables.shape[1], P(w.context_lens), w.max_context_len, w.B,
        w.Hq - 1, w.Hkv, w.D, 16, w.num_blocks, w.scale, 0, 0, 4, P(ws),
        ws.numel(), 0, ctypes.c_void_p(ctypes.addressof(sy)),
        ctypes.c_void_p(ctypes.addressof(io)), None)
    assert rc == _abi.PA_ERR_INVALID_ARG
    back.synchronize()                     # nothing waits on the done word
    copy.synchronize()
    assert int(words[0]) == 1              # the upload's ready word was written
    assert int(words[8]) == 0              # no step, no done signal
