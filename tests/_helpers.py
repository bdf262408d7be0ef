"""Shared test plumbing: run the oracle side and the CUDA side on one workload."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_179_gb300 import workloads as W

# Attention-output tolerances (max abs error against the fp64 oracle), as the
# decode path states them: fp16 output 2e-3, bf16 output 8e-3, E4M3 pool 3e-2.
TOL = {"f16": 2e-3, "bf16": 8e-3, "fp8": 3e-2}


def to_np16(t):
    return W.to_numpy16(t)


def oracle_step(w: W.Workload, rows=None):
    """Oracle append (on host copies of the pools) then oracle decode; float64 [B][Hq][D]."""
    kp = to_np16(w.k_cache).copy()
    vp = to_np16(w.v_cache).copy()
    oracle.cache_append(to_np16(w.k_new), to_np16(w.v_new), kp, vp,
                        w.slot_mapping.cpu().numpy(), w.block_size)
    return oracle.decode(to_np16(w.q), kp, vp, w.block_tables.cpu().numpy(),
                         w.context_lens.cpu().numpy(), w.scale, bf16=(w.dtype == "bf16"),
                         rows=rows)


def to_cuda(w: W.Workload) -> W.Workload:
    for f in ("context_lens", "block_tables", "slot_mapping", "q", "k_cache", "v_cache", "k_new",
              "v_new"):
        setattr(w, f, getattr(w, f).cuda())
    return w


def max_err(gpu_out: torch.Tensor, ref: np.ndarray, rows=None) -> float:
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g, ref = g[rows], ref[rows]
    return float(np.abs(g - ref).max())
