"""The seeded input generators: shapes, determinism, slot mappings, shared
prefixes and the length distributions the workloads name (CPU only)."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_179_gb300 import workloads as W


@pytest.mark.parametrize("name", ["tiny", "smollm2_360m", "qwen2_5_1_5b", "qwen2_5_7b",
                                  "mqa_32x1"])
def test_shapes_tables_and_slots(name):
    w = W.make_workload(name, seed=0)
    cfg = W.CONFIGS[name]
    assert (w.B, w.Hq, w.Hkv, w.D) == (cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"])
    assert w.q.shape == (w.B, w.Hq, w.D) and w.k_new.shape == (w.B, w.Hkv, w.D)
    assert w.k_cache.shape == (w.num_blocks, w.Hkv, 16, w.D)
    lens = w.context_lens.numpy()
    tables = w.block_tables.numpy()
    assert lens.max() <= w.max_context_len <= tables.shape[1] * 16
    used = []
    for b in range(w.B):
        n = (lens[b] + 15) // 16
        assert np.all(tables[b, :n] >= 0) and np.all(tables[b, n:] == -1)
        used += tables[b, :n].tolist()
        # the new token goes to position L-1 of the sequence
        s = int(w.slot_mapping[b])
        assert s // 16 == tables[b, (lens[b] - 1) // 16] and s % 16 == (lens[b] - 1) % 16
    assert max(used) < w.num_blocks
    assert w.scale == float(np.float32(1 / math.sqrt(w.D)))


def test_private_blocks_are_distinct_and_prefix_is_shared():
    w = W.make_workload("smollm2_360m", seed=1)
    lens = w.context_lens.numpy()
    tables = w.block_tables.numpy()
    sh = w.shared_blocks
    assert len(sh) == 32
    for b in range(16):
        assert tables[b, :32].tolist() == sh and lens[b] >= 513
    private = [p for b in range(w.B) for p in tables[b, :(lens[b] + 15) // 16].tolist()
               if p not in sh]
    assert len(private) == len(set(private))
    # nothing appends into a shared block
    assert not set((w.slot_mapping // 16).tolist()) & set(sh)


def test_unfilled_rows_are_zero_and_filled_rows_random():
    w = W.make_workload("tiny", seed=2)
    lens = w.context_lens.numpy()
    tables = w.block_tables.numpy()
    k = w.k_cache.float().numpy()
    for b in range(w.B):
        L = lens[b]
        last = tables[b, (L - 1) // 16]
        row = (L - 1) % 16
        assert not k[last, :, row:].any()          # position L-1 and beyond: empty before append
        if row > 0:
            assert np.abs(k[last, :, :row]).sum() > 0


def test_deterministic_and_seed_dependent():
    a, b, c = (W.make_workload("qwen2_5_1_5b", seed=s) for s in (4, 4, 5))
    assert torch.equal(a.q, b.q) and torch.equal(a.block_tables, b.block_tables)
    assert not torch.equal(a.q, c.q)


def test_length_distributions():
    w = W.make_workload("qwen2_5_7b", seed=0)
    L = w.context_lens.numpy()
    assert L.min() >= 1 and L.max() <= 8192
    assert 700 < np.median(L) < 1500               # lognormal with median 1024
    u = W.make_workload("qwen2_5_1_5b", seed=0).context_lens.numpy()
    assert u.min() >= 512 and u.max() <= 4096
    assert W.make_workload("tiny").context_lens.tolist() == [1, 17, 100, 256]
