"""Thin ctypes binding of libpa (include/pa.h): argument marshalling only.

Every function takes torch tensors, checks that they are CUDA, contiguous and
of the expected dtype and shape, passes their device pointers and the current
torch stream to the C entry point of the same name, and raises ``PAError`` on a
non-zero return code.  All arithmetic happens in the CUDA kernels; if
libpa.so is missing this module raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

PA_F16, PA_BF16, PA_E4M3 = 0, 1, 2
PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_BOUNDS, \
    PA_ERR_TIMEOUT, PA_ERR_SCRATCH_LIMIT = range(8)
PA_NOALLOC_SCRATCH_BYTES = 16 << 20
PA_STATUS_BAD_BLOCK, PA_STATUS_BAD_LEN, PA_STATUS_BAD_SLOT, PA_STATUS_TIMEOUT = 1, 2, 4, 8
PA_STATUS_NO_WORKSPACE = 16
PA_STATUS_WS_DIRTY = 32
PA_DECODE_EARLY_PROLOGUE = 1
PA_DECODE_EARLY_COPIES = 2

# (name, argtypes, restype) of every exported entry point
_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_u32 = ctypes.c_uint
SIGNATURES = {
    "pa_version": ([], _i32),
    "pa_status_string": ([_i32], ctypes.c_char_p),
    "pa_cache_append": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp], _i32),
    "pa_cache_append_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                             _vp], _i32),
    "pa_quantize_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp], _i32),
    "pa_e4m3_encode": ([_vp, _vp, _i64, _vp], _i32),
    "pa_copy_blocks": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp], _i32),
    "pa_decode_workspace_size": ([_i32, _i32, _i32, _i32], _sz),
    "pa_decode_workspace_size_rows": ([_i32, _i32, _i32, _i32, _i32], _sz),
    "pa_decode_default_splits": ([_i32], _i32),
    "pa_decode": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                   _f32, _i32, _i32, _i32, _i32, _vp, _sz, _u32, _vp], _i32),
    "pa_decode_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                       _i32, _i32, _f32, _i32, _i32, _i32, _i32, _vp, _sz, _u32, _vp], _i32),
    "pa_decode_step": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                        _i32, _i32, _i32, _f32, _i32, _i32, _i32, _vp, _sz, _u32, _vp], _i32),
    "pa_decode_step_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                            _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _i32, _vp, _sz, _u32,
                            _vp], _i32),
    "pa_decode_noalloc": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                           _i32, _i32, _f32, _i32, _i32, _i32, _i32, _u32, _vp], _i32),
    "pa_decode_step_synced": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                               _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _i32, _vp, _sz,
                               _u32, _vp, _vp], _i32),
    "pa_decode_step_fp8_synced": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp,
                                   _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32,
                                   _i32, _vp, _sz, _u32, _vp, _vp], _i32),
    "pa_decode_step_pipelined": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32,
                                  _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _i32,
                                  _vp, _sz, _u32, _vp, _vp, _vp], _i32),
    "pa_decode_step_fp8_pipelined": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                      _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                                      _i32, _i32, _vp, _sz, _u32, _vp, _vp, _vp], _i32),
    "pa_stream_write_value": ([_vp, _vp, _u32], _i32),
    "pa_stream_wait_value": ([_vp, _vp, _u32], _i32),
    "pa_get_status": ([_vp, ctypes.POINTER(ctypes.c_uint)], _i32),
    "pa_test_wait_timeout": ([ctypes.c_uint64, _vp], _i32),
    "pa_test_merge_timeout": ([_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz,
                               ctypes.c_uint64, _vp], _i32),
}

_lock = threading.Lock()
_lib = None


class PAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})")


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libpa.so (raising if it is absent, unless asked to build it)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                if not build_if_missing:
                    raise RuntimeError(f"{_build.LIB} is not built; call __graft_entry__.build() "
                                       "or python -m paged_kv_cache_179_gb300.build")
                _build.build()
            L = ctypes.CDLL(_build.LIB)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return load().pa_status_string(code).decode()


def _check(rc: int, where: str):
    if rc != PA_OK:
        raise PAError(rc, where)


class _Recording(threading.local):
    """Per-thread state of ``prepare``: while active, entry points record
    their C calls (with marshalled arguments) instead of making them."""
    active = False
    stream = None
    calls = None


_rec = _Recording()


def _call(fn, where: str, *args):
    if _rec.active:
        conv = []
        for t, a in zip(fn.argtypes, args):
            conv.append(a if a is None or isinstance(a, t) else t(a))
        _rec.calls.append((fn, tuple(conv), where))
        return
    _check(fn(*args), where)


class Prepared:
    """C-ABI calls recorded once, with their arguments already marshalled;
    calling the object makes them again, in order, on the recorded stream.
    Checking shapes, dtypes and devices and converting arguments is done
    once, at ``prepare``; the tensors must stay alive and in place."""

    def __init__(self, calls):
        self.calls = calls

    def __call__(self):
        for fn, args, where in self.calls:
            rc = fn(*args)
            if rc != PA_OK:
                raise PAError(rc, where)


def prepare(body, stream=None) -> Prepared:
    """Run ``body()`` (which calls entry points of this module) with every C
    call recorded instead of made, launching on ``stream`` (a
    torch.cuda.Stream; default: the current stream when the calls run).
    Returns the recorded calls as one callable: a serving loop that repeats
    a step on the same tensors pays the argument checks once."""
    if _rec.active:
        raise RuntimeError("prepare() does not nest")
    _rec.active = True
    _rec.stream = None if stream is None else ctypes.c_void_p(stream.cuda_stream)
    _rec.calls = []
    try:
        body()
        return Prepared(_rec.calls)
    finally:
        _rec.active, _rec.stream, _rec.calls = False, None, None


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev) -> ctypes.c_void_p:
    if _rec.active and _rec.stream is not None:
        return _rec.stream
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(t, name, dtype=None, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, has {t.dim()}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _flags(early_prologue: bool, early_copies: bool = False) -> int:
    if early_copies and not early_prologue:
        raise ValueError("early_copies needs early_prologue")
    return ((PA_DECODE_EARLY_PROLOGUE if early_prologue else 0) |
            (PA_DECODE_EARLY_COPIES if early_copies else 0))


def _act_code(dtype) -> int:
    if dtype == torch.float16:
        return PA_F16
    if dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported activation dtype {dtype}")


# ---------------------------------------------------------------- entry points
def pa_version() -> int:
    return load().pa_version()


def pa_cache_append(k_new, v_new, k_cache, v_cache, slot_mapping) -> None:
    """Scatter k_new/v_new [T][Hkv][D] into the pools [NB][Hkv][bs][D] at slot_mapping [T]."""
    dev = k_cache.device
    act = (torch.float16, torch.bfloat16)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, act, 3, dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_new.dtype, 4, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    T, Hkv, D = k_new.shape
    NB, Hkv2, bs, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or v_new.shape != k_new.shape or v_cache.shape != k_cache.shape \
            or slot_mapping.shape[0] != T:
        raise ValueError("shape mismatch")
    _call(load().pa_cache_append, "pa_cache_append",
          _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, Hkv, D,
          bs, NB, _act_code(k_new.dtype), _stream(dev))


def pa_cache_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, slot_mapping) -> None:
    """E4M3-encode fp16/bf16 k_new/v_new into uint8 pools: a page's first token
    sets its scales, a later token that would saturate re-scales the page."""
    dev = k_cache.device
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, (torch.float16, torch.bfloat16), 3, dev)
    _need(v_new, "v_new", k_new.dtype)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8, 4, dev)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.float32, 2, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    T, Hkv, D = k_new.shape
    NB, _, bs, _ = k_cache.shape
    if k_scale.shape != (NB, Hkv) or v_scale.shape != (NB, Hkv) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    _call(load().pa_cache_append_fp8, "pa_cache_append_fp8",
          _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
          _ptr(slot_mapping), T, Hkv, D, bs, NB, _act_code(k_new.dtype), _stream(dev))


def pa_quantize_fp8(k_src, v_src, k_cache, v_cache, k_scale, v_scale) -> None:
    """Quantise fp16 pools [NB][Hkv][bs][D] into E4M3 pools and [NB][Hkv] fp32 scales."""
    ref = k_src if k_src is not None else v_src
    dev = ref.device
    NB, Hkv, bs, D = ref.shape
    for src, codes, sc, n in ((k_src, k_cache, k_scale, "k"), (v_src, v_cache, v_scale, "v")):
        if src is None:
            continue
        _need(src, n + "_src", torch.float16, 4, dev)
        _need(codes, n + "_cache", torch.uint8, 4, dev)
        _need(sc, n + "_scale", torch.float32, 2, dev)
        if src.shape != ref.shape or codes.shape != ref.shape or sc.shape != (NB, Hkv):
            raise ValueError("shape mismatch")
    _call(load().pa_quantize_fp8, "pa_quantize_fp8",
          _ptr(k_src), _ptr(v_src), _ptr(k_cache if k_src is not None else None),
          _ptr(v_cache if v_src is not None else None),
          _ptr(k_scale if k_src is not None else None),
          _ptr(v_scale if v_src is not None else None), NB, Hkv, D, bs, _stream(dev))


def pa_copy_blocks(k_cache, v_cache, block_mapping, k_scale=None, v_scale=None) -> None:
    """Copy whole physical blocks of both pools: block_mapping is int64
    [n][2] of (src, dst); E4M3 (uint8) pools also copy their [NB][Hkv] scales."""
    dev = k_cache.device
    fp8 = k_cache.dtype == torch.uint8
    _need(k_cache, "k_cache", (torch.float16, torch.bfloat16, torch.uint8), 4, dev)
    _need(v_cache, "v_cache", k_cache.dtype, 4, dev)
    _need(block_mapping, "block_mapping", torch.int64, 2, dev)
    NB, Hkv, bs, D = k_cache.shape
    if v_cache.shape != k_cache.shape or block_mapping.shape[1] != 2:
        raise ValueError("shape mismatch")
    if fp8:
        for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
            _need(t, n, torch.float32, 2, dev)
            if t.shape != (NB, Hkv):
                raise ValueError("shape mismatch")
        code = PA_E4M3
    else:
        if k_scale is not None or v_scale is not None:
            raise ValueError("scales are for E4M3 pools only")
        code = _act_code(k_cache.dtype)
    _call(load().pa_copy_blocks, "pa_copy_blocks",
          _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_mapping),
          block_mapping.shape[0], Hkv, D, bs, NB, code, _stream(dev))


def pa_e4m3_encode(x, codes) -> None:
    _need(x, "x", torch.float32, None)
    _need(codes, "codes", torch.uint8, None, x.device)
    if codes.numel() != x.numel():
        raise ValueError("size mismatch")
    _call(load().pa_e4m3_encode, "pa_e4m3_encode",
          _ptr(x), _ptr(codes), x.numel(), _stream(x.device))


def pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, split_ctas=0) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, split_ctas))


def pa_decode_workspace_size_rows(num_seqs, num_q_heads, head_dim, split_ctas=0,
                                  query_rows=8) -> int:
    """Workspace bytes for calls with up to ``query_rows`` = queries_per_seq *
    (num_q_heads / num_kv_heads) query rows per (sequence, kv head)."""
    return int(load().pa_decode_workspace_size_rows(num_seqs, num_q_heads, head_dim, split_ctas,
                                                    query_rows))


def pa_decode_default_splits(pool_dtype=torch.float16) -> int:
    """CTAs a default (split_ctas=0) decode uses over pools of this dtype
    (torch.uint8 for E4M3 pools)."""
    code = PA_E4M3 if pool_dtype == torch.uint8 else _act_code(pool_dtype)
    return int(load().pa_decode_default_splits(code))


def alloc_workspace(num_seqs, num_q_heads, head_dim, split_ctas, device, query_rows=8):
    """Caller-owned workspace for pa_decode, zero-filled as the decode needs
    it (each call leaves it zero-filled again); ``query_rows``: the most
    query rows per (sequence, kv head) of the calls it serves (queries per
    sequence times the query group)."""
    n = pa_decode_workspace_size_rows(num_seqs, num_q_heads, head_dim, split_ctas, query_rows)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def _decode_common(out, q, block_tables, context_lens, dev):
    """q/out [B][Hq][D], or [B][n_q][Hq][D] for n_q query tokens per sequence."""
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    if q.dim() == 3:
        (B, Hq, D), nq = q.shape, 1
    else:
        B, nq, Hq, D = q.shape
    if out.shape != q.shape or block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("shape mismatch")
    return B, nq, Hq, D


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
              scale: float, split_ctas: int = 0, workspace=None, *, window: int = 0,
              early_prologue: bool = False, early_copies: bool = False) -> None:
    """out[b][hq] = softmax(scale q.K) V over each sequence's blocks (16-bit pools).
    early_prologue: PA_DECODE_EARLY_PROLOGUE (the kernel before this call on
    the stream must not write context_lens or block_tables).
    early_copies: PA_DECODE_EARLY_COPIES as well (the kernels before it must
    also write nothing in the pools except in each sequence's last two
    blocks, as the previous decode step of the same batch does)."""
    dev = q.device
    act = (torch.float16, torch.bfloat16)
    _need(q, "q", act, None, dev)
    _need(out, "out", q.dtype, None, dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, q.dtype, 4, dev)
    B, nq, Hq, D = _decode_common(out, q, block_tables, context_lens, dev)
    NB, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, "workspace", None, None, dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    _call(load().pa_decode, "pa_decode",
          _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
          block_tables.shape[1], _ptr(context_lens), int(max_context_len), B, Hq, Hkv, D, bs, NB,
          float(scale), int(window), nq, _act_code(q.dtype), int(split_ctas), _ptr(workspace),
          ws_bytes, _flags(early_prologue, early_copies), _stream(dev))


def pa_decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                  max_context_len: int, scale: float, split_ctas: int = 0, workspace=None, *,
                  window: int = 0, early_prologue: bool = False, early_copies: bool = False) -> None:
    """As pa_decode over E4M3 pools with per-(block, kv head) fp32 scales; q/out
    fp16 or bf16."""
    dev = q.device
    _need(q, "q", (torch.float16, torch.bfloat16), None, dev)
    _need(out, "out", q.dtype, None, dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8, 4, dev)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.float32, 2, dev)
    B, nq, Hq, D = _decode_common(out, q, block_tables, context_lens, dev)
    NB, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, "workspace", None, None, dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    _call(load().pa_decode_fp8, "pa_decode_fp8",
          _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
          _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), int(max_context_len), B,
          Hq, Hkv, D, bs, NB, float(scale), int(window), nq, _act_code(q.dtype), int(split_ctas),
          _ptr(workspace), ws_bytes, _flags(early_prologue, early_copies), _stream(dev))


class StepSync(ctypes.Structure):
    """pa_step_sync: the device words and values of one step's handshake with
    the copies on other streams (see include/pa.h).  The entry points read
    the values when they are called, so a bound call sees updated values."""
    _fields_ = [("ready", ctypes.c_void_p), ("done", ctypes.c_void_p),
                ("done_count", ctypes.c_void_p), ("ready_value", ctypes.c_uint32),
                ("done_value", ctypes.c_uint32)]


class StepCopies(ctypes.Structure):
    """pa_step_copies: the host<->device copies of one pipelined step (see
    include/pa.h); ``slot_reused`` is read at each call."""
    _fields_ = [("host_in", ctypes.c_void_p), ("dev_in", ctypes.c_void_p),
                ("in_bytes", ctypes.c_size_t), ("dev_out", ctypes.c_void_p),
                ("host_out", ctypes.c_void_p), ("out_bytes", ctypes.c_size_t),
                ("copy_stream", ctypes.c_void_p), ("back_stream", ctypes.c_void_p),
                ("reuse_event", ctypes.c_void_p), ("slot_reused", ctypes.c_int)]


def _sync_ptr(sync):
    return ctypes.c_void_p(ctypes.addressof(sync))


def pa_stream_write_value(word, value: int, stream=None) -> None:
    """Stream-ordered store of ``value`` into the device int32 tensor element
    ``word`` (a 1-element view) on ``stream`` (default: the current stream)."""
    _need(word, "word", (torch.int32,), None)
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(word.device)
    _call(load().pa_stream_write_value, "pa_stream_write_value", s, _ptr(word),
          int(value) & 0xffffffff)


def pa_stream_wait_value(word, value: int, stream=None) -> None:
    """Hold ``stream``'s later work until the device word reaches ``value``
    (cyclic 32-bit comparison)."""
    _need(word, "word", (torch.int32,), None)
    s = ctypes.c_void_p(stream.cuda_stream) if stream is not None else _stream(word.device)
    _call(load().pa_stream_wait_value, "pa_stream_wait_value", s, _ptr(word),
          int(value) & 0xffffffff)


def _ws_bytes(workspace, dev):
    if workspace is None:
        return 0
    _need(workspace, "workspace", None, None, dev)
    return workspace.numel() * workspace.element_size()


def pa_decode_step(out, q, k_new, v_new, k_cache, v_cache, slot_mapping, block_tables,
                   context_lens, max_context_len: int, scale: float, split_ctas: int = 0,
                   workspace=None, *, window: int = 0, early_prologue: bool = False, early_copies: bool = False,
                   sync: StepSync = None, copies: StepCopies = None) -> None:
    """Append k_new/v_new at slot_mapping, then decode, in one launch (16-bit
    pools); with ``sync``, pa_decode_step_synced (device-side handshake); with
    ``copies`` too, pa_decode_step_pipelined (the step's upload and read-back
    in the same call)."""
    dev = q.device
    act = (torch.float16, torch.bfloat16)
    _need(q, "q", act, 3, dev)
    _need(out, "out", q.dtype, 3, dev)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, q.dtype, 3, dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, q.dtype, 4, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    B, nq, Hq, D = _decode_common(out, q, block_tables, context_lens, dev)
    if nq != 1:
        raise ValueError("the fused step takes one query token per sequence")
    NB, Hkv, bs, _ = k_cache.shape
    if k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape or slot_mapping.shape[0] != B:
        raise ValueError("shape mismatch")
    args = (_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
            _ptr(slot_mapping), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            int(max_context_len), B, Hq, Hkv, D, bs, NB, float(scale), int(window),
            _act_code(q.dtype), int(split_ctas), _ptr(workspace), _ws_bytes(workspace, dev),
            _flags(early_prologue, early_copies))
    if sync is None:
        _call(load().pa_decode_step, "pa_decode_step", *args, _stream(dev))
    elif copies is None:
        _call(load().pa_decode_step_synced, "pa_decode_step_synced", *args, _sync_ptr(sync),
              _stream(dev))
    else:
        _call(load().pa_decode_step_pipelined, "pa_decode_step_pipelined", *args,
              _sync_ptr(sync), _sync_ptr(copies), _stream(dev))


def pa_decode_step_fp8(out, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                       block_tables, context_lens, max_context_len: int, scale: float,
                       split_ctas: int = 0, workspace=None, *, window: int = 0,
                       early_prologue: bool = False, early_copies: bool = False, sync: StepSync = None,
                       copies: StepCopies = None) -> None:
    """Append (E4M3-encode) k_new/v_new, then decode over the E4M3 pools, in one
    attention launch; q, k_new, v_new and out share one dtype (fp16 or bf16)."""
    dev = q.device
    _need(q, "q", (torch.float16, torch.bfloat16), 3, dev)
    for t, n in ((out, "out"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, q.dtype, 3, dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8, 4, dev)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.float32, 2, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    B, nq, Hq, D = _decode_common(out, q, block_tables, context_lens, dev)
    if nq != 1:
        raise ValueError("the fused step takes one query token per sequence")
    NB, Hkv, bs, _ = k_cache.shape
    if k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape or slot_mapping.shape[0] != B:
        raise ValueError("shape mismatch")
    args = (_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
            _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), int(max_context_len), B, Hq, Hkv, D, bs, NB,
            float(scale), int(window), _act_code(q.dtype), int(split_ctas), _ptr(workspace),
            _ws_bytes(workspace, dev), _flags(early_prologue, early_copies))
    if sync is None:
        _call(load().pa_decode_step_fp8, "pa_decode_step_fp8", *args, _stream(dev))
    elif copies is None:
        _call(load().pa_decode_step_fp8_synced, "pa_decode_step_fp8_synced", *args,
              _sync_ptr(sync), _stream(dev))
    else:
        _call(load().pa_decode_step_fp8_pipelined, "pa_decode_step_fp8_pipelined", *args,
              _sync_ptr(sync), _sync_ptr(copies), _stream(dev))


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                      max_context_len: int, scale: float, split_ctas: int = 0,
                      window: int = 0, early_prologue: bool = False, early_copies: bool = False) -> None:
    """pa_decode with the library's static scratch instead of a workspace (allocates nothing)."""
    dev = q.device
    act = (torch.float16, torch.bfloat16)
    _need(q, "q", act, None, dev)
    _need(out, "out", q.dtype, None, dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, q.dtype, 4, dev)
    B, nq, Hq, D = _decode_common(out, q, block_tables, context_lens, dev)
    NB, Hkv, bs, _ = k_cache.shape
    _call(load().pa_decode_noalloc, "pa_decode_noalloc",
          _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
          block_tables.shape[1], _ptr(context_lens), int(max_context_len), B, Hq, Hkv, D, bs, NB,
          float(scale), int(window), nq, _act_code(q.dtype), int(split_ctas),
          _flags(early_prologue, early_copies), _stream(dev))


def pa_test_wait_timeout(limit_ns: int, device=None) -> None:
    """Failure-path test: one warp's bounded mbarrier wait on a barrier that
    nothing completes gives up after ``limit_ns`` and sets PA_STATUS_TIMEOUT."""
    _call(load().pa_test_wait_timeout, "pa_test_wait_timeout", int(limit_ns),
          _stream(device or torch.cuda.current_device()))


def pa_test_merge_timeout(out, context_lens, max_context_len: int, num_kv_heads: int,
                          split_ctas: int, workspace, limit_ns: int) -> None:
    """Failure-path test: pa_decode's merge launch alone (nothing writes the
    partials it polls for) gives up after ``limit_ns`` and sets
    PA_STATUS_TIMEOUT.  out [B][Hq][D] as for pa_decode."""
    dev = out.device
    _need(out, "out", (torch.float16, torch.bfloat16), 3, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = out.shape
    _call(load().pa_test_merge_timeout, "pa_test_merge_timeout",
          _ptr(out), _ptr(context_lens), int(max_context_len), B, Hq, int(num_kv_heads), D,
          _act_code(out.dtype), int(split_ctas), _ptr(workspace), _ws_bytes(workspace, dev),
          int(limit_ns), _stream(dev))


def pa_get_status(device=None) -> tuple[int, int]:
    """(return code, raw status bits) after synchronising the current stream."""
    bits = ctypes.c_uint(0)
    rc = load().pa_get_status(_stream(device or torch.cuda.current_device()), ctypes.byref(bits))
    return rc, bits.value
