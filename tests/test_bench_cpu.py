"""Host-side accounting of bench.py, checked on the CPU: the algorithmic
bytes its roofline divides by (against counts worked out by hand for the
4-sequence workload and the shared prefix of the SmolLM2-360M one), and the
use of the committed ncu traffic figures only for the kernel sources they
were taken from."""
import json
import os

import numpy as np

import bench
from paged_kv_cache_179_gb300 import workloads as W


def test_attended_tokens_with_and_without_window():
    lens = np.array([0, 5, 100, 4096])
    assert bench.attended(lens).tolist() == [0, 5, 100, 4096]
    assert bench.attended(lens, 16).tolist() == [0, 5, 16, 16]


def test_algorithmic_bytes_of_the_small_workload():
    # lengths 1, 17, 100, 256; 2 kv heads, head_dim 64, fp16 pools and q
    w = W.make_workload("tiny", seed=0)
    lens = w.context_lens.numpy()
    assert lens.tolist() == [1, 17, 100, 256]
    ab = bench.algorithmic_bytes(w, lens)
    per_token = 2 * 2 * 64 * 2            # kv heads x (K, V) x head_dim x 2 bytes
    assert ab["kv"] == 374 * per_token
    assert ab["q_out"] == 2 * 4 * 8 * 64 * 2
    assert ab["meta"] == (1 + 2 + 7 + 16) * 4 + 4 * 4   # table entries read, lengths
    assert ab["scales"] == 0
    assert ab["total"] == ab["kv"] + ab["q_out"] + ab["meta"]
    assert ab["kv_unique"] == ab["kv"]    # no block is shared
    # a 16-token window: 1 + 16 + 16 + 16 tokens; blocks from the window's first
    win = bench.algorithmic_bytes(w, lens, window=16)
    assert win["kv"] == 49 * per_token
    assert win["meta"] == (1 + 2 + 2 + 1) * 4 + 4 * 4
    assert win["kv_unique"] == win["kv"]


def test_shared_prefix_counted_once_in_unique_bytes():
    # 16 sequences share a 512-token prefix, each longer than it
    w = W.make_workload("smollm2_360m", seed=0)
    lens = w.context_lens.numpy()
    ab = bench.algorithmic_bytes(w, lens)
    per_token = w.Hkv * 2 * w.D * 2
    assert ab["kv"] == int(lens.sum()) * per_token
    assert ab["kv"] - ab["kv_unique"] == (16 - 1) * 512 * per_token


def test_traffic_used_only_for_its_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    entry = {"split_ctas": 304, "kernel_sha": "abc", "bytes_per_launch": 123}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"cfg": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sha", lambda tc=False: "abc")
    assert bench.load_traffic("cfg", 304) == 123
    assert bench.load_traffic("cfg", 456) is None         # another CTA split
    assert bench.load_traffic("other", 304) is None
    monkeypatch.setattr(bench, "kernel_sha", lambda tc=False: "def")
    assert bench.load_traffic("cfg", 304) is None         # the kernel changed since


def test_committed_traffic_figures_are_consistent():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for name, e in t.items():
        if name.startswith("_"):
            continue
        # "config" (the decode step) or "config:qN" (N query tokens per sequence)
        config, _, queries = name.partition(":")
        assert config in W.CONFIGS
        assert queries == "" or (queries.startswith("q") and int(queries[1:]) >= 2)
        assert e["bytes_per_launch"] == e["read"] + e["write"]
        assert len(e["kernel_sha"]) == 16
