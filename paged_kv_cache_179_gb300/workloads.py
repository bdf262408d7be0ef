"""Seeded synthetic inputs for the paged-KV decode step.

This module is the only code that both the CUDA path and the oracle use.  It
holds none of the method's arithmetic: it draws context lengths, block tables,
slot mappings and random Q/K/V values, and moves data around; it never appends,
quantises or attends.

Shapes follow the workloads the pages describe (model names are shapes only:
no weights, no datasets):

=================  ====  ========  ====  =====  ==============================
name               B     Hq/Hkv    D     dtype  context lengths / pool
=================  ====  ========  ====  =====  ==============================
tiny               4     8/2       64    f16    {1,17,100,256}; pool of 64 blocks
smollm2_360m       32    15/5      64    bf16   U[128,2048]; seqs 0-15 share a
                                                512-token prefix, draw U[513,2048]
qwen2_5_1_5b       48    12/2      128   f16    U[512,4096]; 16384-block pool
qwen2_5_7b         128   28/4      128   f16    lognormal(median 1024, sigma 1)
                                                clipped to [1,8192]
qwen2_5_7b_fp8     256   28/4      128   fp8    U[4096,32768]; K/V drawn fp16,
                                                then quantised to E4M3 per page
mqa_32x1           128   32/1      128   f16    as qwen2_5_7b (multi-query)
=================  ====  ========  ====  =====  ==============================

Generation order is fixed: context lengths, block tables, Q, the K/V pool,
then the new token's K/V.  ``context_lens`` count the token appended this
step: the pool holds positions ``0 .. L-2`` on entry, the append writes
position ``L-1`` and decode attends over ``0 .. L-1``.  Pool rows that hold no
token (the tail of each sequence's last block, unused blocks) are zero unless
``fill`` asks for something else.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16

CONFIGS = {
    "tiny": dict(B=4, Hq=8, Hkv=2, D=64, dtype="f16", kv="f16", lens="fixed",
                 fixed_lens=(1, 17, 100, 256), pool_blocks=64),
    "smollm2_360m": dict(B=32, Hq=15, Hkv=5, D=64, dtype="bf16", kv="bf16", lens="uniform",
                         lo=128, hi=2048, shared_prefix_seqs=16, shared_prefix_tokens=512),
    "qwen2_5_1_5b": dict(B=48, Hq=12, Hkv=2, D=128, dtype="f16", kv="f16", lens="uniform",
                         lo=512, hi=4096, pool_blocks=16384),
    "qwen2_5_7b": dict(B=128, Hq=28, Hkv=4, D=128, dtype="f16", kv="f16", lens="lognormal",
                       median=1024, sigma=1.0, lo=1, hi=8192),
    "qwen2_5_7b_fp8": dict(B=256, Hq=28, Hkv=4, D=128, dtype="f16", kv="fp8", lens="uniform",
                           lo=4096, hi=32768),
    # multi-query attention: one kv head serves all 32 q heads (the pages'
    # "GQA/MQA"), with the Qwen2.5-7B batch's lengths
    "mqa_32x1": dict(B=128, Hq=32, Hkv=1, D=128, dtype="f16", kv="f16", lens="lognormal",
                     median=1024, sigma=1.0, lo=1, hi=8192),
}

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    """One decode step's inputs.  Tensors live on ``device``."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str                      # activation dtype of q / out / new K,V: "f16" | "bf16"
    kv: str                         # pool storage: "f16" | "bf16" | "fp8" (fp8: pool below is the fp16 source)
    block_size: int
    num_blocks: int
    max_context_len: int            # the host-side bound the scheduler knows
    context_lens: torch.Tensor      # int32 [B], includes the token appended this step
    block_tables: torch.Tensor      # int32 [B][MBS], -1 past each sequence's blocks
    slot_mapping: torch.Tensor      # int64 [B], slot of position L-1
    q: torch.Tensor                 # [B][Hq][D]
    k_cache: torch.Tensor           # [NB][Hkv][bs][D], positions 0..L-2 filled
    v_cache: torch.Tensor
    k_new: torch.Tensor             # [B][Hkv][D]
    v_new: torch.Tensor
    scale: float                    # 1/sqrt(D) rounded to fp32
    shared_blocks: list = field(default_factory=list)   # physical ids shared by several tables
    seed: int = 0

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def total_tokens(self) -> int:
        return int(self.context_lens.sum().item())


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(g, shape, dev, dtype, chunk=1 << 26):
    """N(0,1) drawn in fp32 and rounded to ``dtype``, in chunks to bound the fp32 temporary."""
    out = torch.empty(shape, device=dev, dtype=dtype)
    flat = out.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=g, device=dev, dtype=torch.float32).to(dtype)
    return out


def _draw_lens(cfg, B, g):
    kind = cfg["lens"]
    if kind == "fixed":
        return torch.tensor(cfg["fixed_lens"], dtype=torch.int64)
    if kind == "uniform":
        lens = torch.randint(cfg["lo"], cfg["hi"] + 1, (B,), generator=g)
        n_sh = cfg.get("shared_prefix_seqs", 0)
        if n_sh:
            # Sequences that share the prefix must extend past it, so their
            # next token lands in a private block (nothing appends into a
            # shared block).
            lo_sh = cfg["shared_prefix_tokens"] + 1
            lens[:n_sh] = torch.randint(lo_sh, cfg["hi"] + 1, (n_sh,), generator=g)
        return lens
    if kind == "lognormal":
        z = torch.randn(B, generator=g, dtype=torch.float64)
        lens = torch.exp(math.log(cfg["median"]) + cfg["sigma"] * z).round().to(torch.int64)
        return lens.clamp(cfg["lo"], cfg["hi"])
    raise ValueError(kind)


def make_workload(name: str, seed: int = 0, device="cpu", fill: str = "zero",
                  lens_override=None) -> Workload:
    """Draw the named workload.  ``fill`` sets pool rows that hold no token:
    "zero", "random" (N(0,1) garbage) or "nan" (16-bit NaN patterns)."""
    cfg = CONFIGS[name]
    B, Hq, Hkv, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"]
    bs = BLOCK_SIZE
    act = TORCH_DTYPE[cfg["dtype"]]
    pool_dtype = torch.float16 if cfg["kv"] == "fp8" else TORCH_DTYPE[cfg["kv"]]
    dev = torch.device(device)
    gc = _gen("cpu", seed)

    # 1. context lengths (post-append)
    lens = (torch.as_tensor(lens_override, dtype=torch.int64) if lens_override is not None
            else _draw_lens(cfg, B, gc))
    B = int(lens.numel())
    nblk = (lens + bs - 1) // bs
    max_ctx = int(cfg.get("hi", int(lens.max())))
    max_ctx = max(max_ctx, int(lens.max()))
    mbs = (max_ctx + bs - 1) // bs

    # 2. block tables: a seeded shuffle of the pool, with an optional shared prefix
    n_sh = cfg.get("shared_prefix_seqs", 0) if lens_override is None else 0
    sh_blocks = cfg.get("shared_prefix_tokens", 0) // bs if n_sh else 0
    private = [int(nblk[b]) - (sh_blocks if b < n_sh else 0) for b in range(B)]
    needed = sum(private) + sh_blocks
    NB = cfg.get("pool_blocks") or int(math.ceil(needed * 1.1))
    if needed > NB:
        raise ValueError(f"{name}: {needed} blocks needed, pool has {NB}")
    perm = torch.randperm(NB, generator=gc)
    shared = perm[:sh_blocks].tolist()
    tables = torch.full((B, mbs), -1, dtype=torch.int32)
    cursor = sh_blocks
    for b in range(B):
        row = []
        if b < n_sh:
            row += shared
        row += perm[cursor:cursor + private[b]].tolist()
        cursor += private[b]
        tables[b, :len(row)] = torch.tensor(row, dtype=torch.int32)

    # rows of each physical block that hold a token before this step's append
    rows_filled = np.zeros(NB, dtype=np.int64)
    tnp = tables.numpy()
    for b in range(B):
        n = int(nblk[b])
        filled = np.clip(int(lens[b]) - 1 - np.arange(n) * bs, 0, bs)
        np.maximum.at(rows_filled, tnp[b, :n], filled)
    rows_filled = torch.from_numpy(rows_filled)
    last_pos = lens - 1
    slots = tables[torch.arange(B), (last_pos // bs)].to(torch.int64) * bs + last_pos % bs

    # 3-5. values: Q, the pool, the new token (on the target device)
    gd = _gen(dev, seed + 1)
    q = _randn(gd, (B, Hq, D), dev, act)
    k_cache = _randn(gd, (NB, Hkv, bs, D), dev, pool_dtype)
    v_cache = _randn(gd, (NB, Hkv, bs, D), dev, pool_dtype)
    k_new = _randn(gd, (B, Hkv, D), dev, pool_dtype)
    v_new = _randn(gd, (B, Hkv, D), dev, pool_dtype)
    empty = (torch.arange(bs)[None, :] >= rows_filled[:, None]).to(dev)[:, None, :, None]
    if fill == "zero":
        k_cache.masked_fill_(empty, 0)
        v_cache.masked_fill_(empty, 0)
    elif fill == "nan":
        k_cache.masked_fill_(empty, float("nan"))
        v_cache.masked_fill_(empty, float("nan"))
    elif fill != "random":
        raise ValueError(fill)

    scale = float(np.float32(1.0 / math.sqrt(D)))
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=cfg["dtype"], kv=cfg["kv"],
                    block_size=bs, num_blocks=NB, max_context_len=max_ctx,
                    context_lens=lens.to(torch.int32).to(dev), block_tables=tables.to(dev),
                    slot_mapping=slots.to(dev), q=q, k_cache=k_cache, v_cache=v_cache,
                    k_new=k_new, v_new=v_new, scale=scale, shared_blocks=shared, seed=seed)


def to_numpy16(t: torch.Tensor) -> np.ndarray:
    """A 16-bit tensor as a numpy array the oracle takes (float16, or bf16 bits as uint16)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def extract_rows(tables: np.ndarray, lens: np.ndarray, rows, pool_tensors):
    """Copy only the blocks that the sequences ``rows`` read into a compact pool.

    Returns (tables', lens', pools') where tables' relabels the physical ids
    0..n-1 in first-seen order and pools' are host numpy arrays.  Used to hand
    a sample of a large batch to the oracle.  Pure data movement.
    """
    rows = list(rows)
    sub_t = np.full((len(rows), tables.shape[1]), -1, dtype=np.int32)
    ids = {}
    for i, b in enumerate(rows):
        n = (int(lens[b]) + BLOCK_SIZE - 1) // BLOCK_SIZE
        for j in range(n):
            pb = int(tables[b, j])
            if pb not in ids:
                ids[pb] = len(ids)
            sub_t[i, j] = ids[pb]
    order = torch.tensor(list(ids.keys()), dtype=torch.int64)
    pools = []
    for p in pool_tensors:
        sel = p.index_select(0, order.to(p.device)).cpu()
        pools.append(to_numpy16(sel) if sel.element_size() == 2 else sel.numpy())
    return sub_t, np.asarray([lens[b] for b in rows], dtype=np.int32), pools
