"""PA_DECODE_EARLY_PROLOGUE: the attention launch is a programmatic dependent
launch whose prologue may overlap the kernel before it on the stream.  That
kernel here writes what the decode reads after its wait (the appended rows
of the pools, q), so a read made too early would show.  With
PA_DECODE_EARLY_COPIES as well, the first K/V copies of blocks before each
sequence's last two start before the wait; the kernels before write the
pools only in the last block (the appends, E4M3 page re-scales included),
as the flag requires.  Results must equal those of the plain launch bit for
bit, step after step."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import TOL, max_err, to_cuda, to_np16

pytestmark = pytest.mark.gpu


# (early_prologue, early_copies)
MODES = {"plain": (False, False), "prologue": (True, False), "copies": (True, True)}


def _steps(w, kc, vc, mode, **kw):
    early, copies = MODES[mode]
    return DecodeStep(k_cache=kc, v_cache=vc, block_tables=w.block_tables,
                      context_lens=w.context_lens, max_context_len=w.max_context_len,
                      scale=w.scale, num_q_heads=w.Hq, early_prologue=early,
                      early_copies=copies, **kw)


@pytest.mark.parametrize("config,window", [("qwen2_5_1_5b", 0), ("smollm2_360m", 0),
                                           ("qwen2_5_1_5b", 200)])
def test_early_prologue_matches_plain_launch(config, window):
    w = to_cuda(W.make_workload(config, seed=21, fill="random"))
    g = torch.Generator(device="cuda").manual_seed(5)
    n = 4
    qs = [torch.randn(w.q.shape, generator=g, device="cuda").to(w.q.dtype) for _ in range(n)]
    kns = [torch.randn(w.k_new.shape, generator=g, device="cuda").to(w.q.dtype) for _ in range(n)]
    vns = [torch.randn(w.k_new.shape, generator=g, device="cuda").to(w.q.dtype) for _ in range(n)]
    outs = {}
    for mode in MODES:
        kc, vc = w.k_cache.clone(), w.v_cache.clone()
        st = _steps(w, kc, vc, mode, window=window)
        q_buf = torch.empty_like(w.q)
        got = []
        for i in range(n):
            # two-launch form: the append kernel writes the rows this decode reads
            o1 = torch.empty_like(w.q)
            _abi.pa_cache_append(kns[i], vns[i], kc, vc, w.slot_mapping)
            st.decode(qs[i], o1)
            # fused form after a kernel that writes q
            o2 = torch.empty_like(w.q)
            q_buf.copy_(qs[(i + 1) % n])
            st.fused(q_buf, kns[i], vns[i], w.slot_mapping, o2)
            got += [o1, o2]
        torch.cuda.synchronize()
        assert _abi.pa_get_status() == (0, 0)
        outs[mode] = ([o.clone() for o in got], kc.clone(), vc.clone())
    plain = outs["plain"]
    for mode in ("prologue", "copies"):
        early = outs[mode]
        for a, b in zip(plain[0], early[0]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), mode
        assert torch.equal(plain[1].view(torch.int16), early[1].view(torch.int16)), mode
        assert torch.equal(plain[2].view(torch.int16), early[2].view(torch.int16)), mode
    # and the last fused step against the oracle
    kp, vp = to_np16(plain[1]), to_np16(plain[2])
    ref = oracle.decode(to_np16(qs[0]), kp, vp, w.block_tables.cpu().numpy(),
                        w.context_lens.cpu().numpy(), w.scale, bf16=(w.dtype == "bf16"),
                        window=window)
    assert max_err(early[0][-1], ref) <= TOL["bf16" if w.dtype == "bf16" else "f16"]


def test_early_prologue_fp8_and_noalloc():
    w = to_cuda(W.make_workload("qwen2_5_1_5b", seed=22, fill="random"))
    kc = torch.empty(w.k_cache.shape, dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    ks = torch.empty(w.num_blocks, w.Hkv, dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    _abi.pa_quantize_fp8(w.k_cache, w.v_cache, kc, vc, ks, vs)
    res = {}
    g = torch.Generator(device="cuda").manual_seed(6)
    # new rows of growing size: later appends re-scale their (last) page
    news = [(torch.randn(w.k_new.shape, generator=g, device="cuda") * 4 ** i).to(w.q.dtype)
            for i in range(3)]
    for mode in MODES:
        early, copies = MODES[mode]
        kc2, vc2, ks2, vs2 = kc.clone(), vc.clone(), ks.clone(), vs.clone()
        st = _steps(w, kc2, vc2, mode, k_scale=ks2, v_scale=vs2)
        got = []
        for kn in news:
            o1 = torch.empty_like(w.q)
            st(w.q, kn, kn.flip(-1), w.slot_mapping, o1)       # append (E4M3), then decode
            got.append(o1)
        o2 = torch.empty_like(w.q)
        _abi.pa_decode_noalloc(o2, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                               w.max_context_len, w.scale, 0, early_prologue=early,
                               early_copies=copies)
        torch.cuda.synchronize()
        assert _abi.pa_get_status() == (0, 0)
        res[mode] = (*got, o2, kc2, ks2, vc2, vs2)
    for mode in ("prologue", "copies"):
        for a, b in zip(res["plain"], res[mode]):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), mode
