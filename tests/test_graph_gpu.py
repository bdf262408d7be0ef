"""DecodeStep.capture: the fused step recorded once into a CUDA graph and
replayed over successive decode steps must produce, step by step, the same
bytes (outputs and pools) as the same step called eagerly: one kernel, one
split, the same inputs.  Also with the captured attention launch as an
early-prologue (programmatic dependent) launch."""
import pytest
import torch

from paged_kv_cache_179_gb300 import _abi
from paged_kv_cache_179_gb300 import workloads as W
from paged_kv_cache_179_gb300.step import DecodeStep

from _helpers import to_cuda

pytestmark = pytest.mark.gpu

STEPS = 4


def _slots(tables, lens):
    """Slot of each sequence's newest token (position len - 1)."""
    last = lens.to(torch.int64) - 1
    rows = torch.arange(lens.numel(), device=lens.device)
    return tables[rows, last // 16].to(torch.int64) * 16 + last % 16


@pytest.mark.parametrize("name,fp8,early", [("qwen2_5_1_5b", False, False),
                                            ("smollm2_360m", False, False),
                                            ("qwen2_5_1_5b", True, False),
                                            ("qwen2_5_1_5b", False, True),
                                            ("qwen2_5_1_5b", True, True)])
def test_graph_replay_matches_eager_over_steps(name, fp8, early):
    g = torch.Generator().manual_seed(11)
    cfg = W.CONFIGS[name]
    B = cfg["B"]
    # every sequence's last block keeps room for STEPS - 1 more tokens
    lens0 = (torch.randint(2, 120, (B,), generator=g) * 16
             + torch.randint(1, 16 - STEPS + 1, (B,), generator=g))
    w = to_cuda(W.make_workload(name, seed=5, lens_override=lens0.tolist(), fill="random"))
    if fp8:
        kc = torch.empty(w.k_cache.shape, dtype=torch.uint8, device="cuda")
        vc = torch.empty_like(kc)
        ks = torch.empty(w.num_blocks, w.Hkv, device="cuda")
        vs = torch.empty_like(ks)
        _abi.pa_quantize_fp8(w.k_cache, w.v_cache, kc, vc, ks, vs)
        pools = [kc, vc, ks, vs]
    else:
        pools = [w.k_cache, w.v_cache]
    eager_pools = [p.clone() for p in pools]
    names = ["k_cache", "v_cache", "k_scale", "v_scale"]
    tables = w.block_tables
    max_ctx = int(lens0.max()) + STEPS
    act = w.q.dtype

    def make_step(pl, lens, early_prologue=False):
        return DecodeStep(**dict(zip(names, pl)), block_tables=tables, context_lens=lens,
                          max_context_len=max_ctx, scale=w.scale, num_q_heads=w.Hq,
                          early_prologue=early_prologue)

    lens_g = w.context_lens.clone()       # the graph's lengths, grown in place
    lens_e = w.context_lens.clone()
    step_g = make_step(pools, lens_g, early)     # the graph's kernels may start early
    step_e = make_step(eager_pools, lens_e)
    q = torch.empty_like(w.q)
    kn = torch.empty_like(w.k_new)
    vn = torch.empty_like(w.v_new)
    slots = torch.empty_like(w.slot_mapping)
    out_g = torch.empty_like(w.q)
    graph = None
    for step in range(STEPS):
        if step:
            lens_g += 1
            lens_e += 1
        q.copy_(torch.randn(q.shape, generator=g).to(act))
        kn.copy_(torch.randn(kn.shape, generator=g).to(kn.dtype))
        vn.copy_(torch.randn(vn.shape, generator=g).to(vn.dtype))
        slots.copy_(_slots(tables, lens_g))
        if graph is None:
            graph = step_g.capture(q, kn, vn, slots, out_g)
        else:
            graph.replay()
        out_e = torch.empty_like(q)
        step_e(q.clone(), kn.clone(), vn.clone(), slots.clone(), out_e)
        torch.cuda.synchronize()
        assert _abi.pa_get_status() == (0, 0)
        assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16)), step
        for a, b in zip(pools, eager_pools):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), step
