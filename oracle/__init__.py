"""The oracle: plain fp64 CPU statement of the paged-KV decode-step hot path.

TEST INFRASTRUCTURE ONLY.  This package is loaded by the tests, by the smoke
check and by the benchmark's CPU-baseline leg, never by the product library.
It shares no code with the CUDA path; the two meet only in the seeded input
generators of ``paged_kv_cache_179_gb300.workloads``.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision, compiled
with gcc, no fast-math, no FMA contraction); this module only compiles it and
marshals numpy arrays.  Every function here is pinned by ``tests/test_oracle.py``
against closed forms, invariants, a dense materialised-softmax statement built
from numpy/scipy routines, and torch's E4M3 conversion.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into liboracle.so beside it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            L.oracle_e4m3_encode.argtypes = [f32]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_e4m3_encode_array.argtypes = [vp, vp, i64]
            L.oracle_e4m3_value_array.argtypes = [vp, vp, i64]
            L.oracle_cache_append.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32]
            L.oracle_quantize_fp8.argtypes = [vp, i64, i32, i32, i32, vp, vp]
            L.oracle_cache_append_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                  i32]
            L.oracle_decode.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                                        f32, i32, i32, vp, i32, vp]
            L.oracle_decode_fp8.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                            i32, i32, f32, i32, i32, vp, i32, vp]
            L.oracle_copy_blocks.argtypes = [vp, vp, vp, vp, vp, i32, ctypes.c_size_t, i32, i64]
            L.oracle_num_threads.restype = i32
            L.oracle_set_num_threads.argtypes = [i32]
            _lib = L
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use (OMP_NUM_THREADS or all cores)."""
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Run the oracle's parallel loops on ``n`` threads from now on (results
    do not depend on it: each output row is reduced by one thread)."""
    lib().oracle_set_num_threads(int(n))


def _u16(a: np.ndarray) -> np.ndarray:
    """16-bit activations (float16 or bf16 carried as uint16/int16 bits) as contiguous uint16."""
    a = np.ascontiguousarray(a)
    assert a.dtype.itemsize == 2, a.dtype
    return a.view(np.uint16)


# ------------------------------------------------------------------ E4M3 codec
def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> E4M3 codes (RNE, saturating to +-448, NaN -> 0x7F)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_p(x), _p(out), x.size)
    return out


def e4m3_value(codes) -> np.ndarray:
    """E4M3 codes -> exact values (float64); NaN codes give NaN."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_value_array(_p(c), _p(out), c.size)
    return out


# ------------------------------------------------------------------ append
def cache_append(k_new, v_new, k_cache, v_cache, slot_mapping, block_size: int) -> None:
    """In place: scatter each token's [Hkv][D] K/V rows to cache[slot//bs][h][slot%bs]."""
    T, Hkv, D = k_new.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype.itemsize == k_new.dtype.itemsize
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    lib().oracle_cache_append(_p(k_new), _p(v_new), _p(k_cache), _p(v_cache), _p(slots), T, Hkv, D,
                              block_size, k_new.dtype.itemsize)


def copy_blocks(k_cache, v_cache, pairs, k_scale=None, v_scale=None) -> None:
    """In place: for each (src, dst) row of pairs, in order, copy physical block
    src of both pools (and of the scales, when given) to block dst."""
    NB, Hkv = k_cache.shape[:2]
    for a in (k_cache, v_cache):
        assert a.flags.c_contiguous and a.shape == k_cache.shape and a.dtype == k_cache.dtype
    if k_scale is not None:
        assert k_scale.dtype == np.float32 and k_scale.shape == (NB, Hkv)
        assert v_scale.dtype == np.float32 and v_scale.shape == (NB, Hkv)
    pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    block_bytes = k_cache[0].nbytes if NB else 0
    lib().oracle_copy_blocks(_p(k_cache), _p(v_cache), _p(k_scale), _p(v_scale), _p(pairs),
                             pairs.shape[0], block_bytes, Hkv, NB)


def cache_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                     block_size: int, *, bf16: bool = False) -> None:
    """In place: E4M3-encode each token row (fp16, or bf16 bits as uint16 when
    ``bf16``) into its page: the page's first token sets the scale, a later
    token that would saturate re-scales the page first."""
    T, Hkv, D = k_new.shape
    for a in (k_cache, v_cache, k_scale, v_scale):
        assert a.flags.c_contiguous
    assert k_cache.dtype == np.uint8 and k_scale.dtype == np.float32
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    lib().oracle_cache_append_fp8(_p(_u16(k_new)), _p(_u16(v_new)), _p(k_cache), _p(v_cache),
                                  _p(k_scale), _p(v_scale), _p(slots), T, Hkv, D, block_size,
                                  int(bf16))


def quantize_fp8(src) -> tuple[np.ndarray, np.ndarray]:
    """fp16 pool [NB][Hkv][bs][D] -> (E4M3 codes same shape, fp32 scales [NB][Hkv])."""
    NB, Hkv, bs, D = src.shape
    codes = np.empty(src.shape, dtype=np.uint8)
    scales = np.empty((NB, Hkv), dtype=np.float32)
    lib().oracle_quantize_fp8(_p(_u16(src)), NB, Hkv, bs, D, _p(codes), _p(scales))
    return codes, scales


# ------------------------------------------------------------------ decode
def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int32)
    return r, int(r.size)


def _q_shape(q):
    """[B][Hq][D] (one query per sequence) or [B][n_q][Hq][D]."""
    if q.ndim == 3:
        B, Hq, D = q.shape
        return B, 1, Hq, D
    return q.shape


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, *, bf16: bool = False,
           window: int = 0, rows=None, return_wsum: bool = False):
    """GQA decode over a 16-bit paged pool, in double.

    q: [B][Hq][D], or [B][n_q][Hq][D] for n_q query tokens per sequence at
    positions L-n_q .. L-1, each attending causally (float16, or bf16 bits as
    uint16 when ``bf16``); ``window`` > 0 limits each query to its last
    ``window`` positions.  Caches [NB][Hkv][bs][D] of the same type;
    block_tables int32 [B][MBS]; context_lens int32 [B].  Returns float64 of
    q's shape (rows not selected by ``rows`` are zero) and, with
    ``return_wsum``, |sum_t w_t/Z - 1| per output row.
    """
    B, nq, Hq, D = _q_shape(q)
    NB, Hkv, bs, D2 = k_cache.shape
    assert D == D2 and Hq % Hkv == 0 and D <= 256 and window >= 0
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros(q.shape, dtype=np.float64)
    ws = np.zeros(q.shape[:-1], dtype=np.float64) if return_wsum else None
    r, nr = _rows_arg(rows)
    lib().oracle_decode(_p(out), _p(_u16(q)), _p(_u16(k_cache)), _p(_u16(v_cache)), int(bf16),
                        _p(bt), bt.shape[1], _p(cl), B, Hq, Hkv, D, bs, float(np.float32(scale)),
                        int(window), nq, _p(r), nr, _p(ws))
    return (out, ws) if return_wsum else out


def decode_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale: float, *,
               bf16: bool = False, window: int = 0, rows=None, return_wsum: bool = False):
    """GQA decode over an E4M3 pool with per-(block, kv head) fp32 scales, in
    double; q is fp16, or bf16 bits as uint16 when ``bf16``; q's shape,
    ``window`` and the result as for ``decode``."""
    B, nq, Hq, D = _q_shape(q)
    NB, Hkv, bs, D2 = k_codes.shape
    assert D == D2 and Hq % Hkv == 0 and D <= 256 and window >= 0
    assert k_codes.dtype == np.uint8 and v_codes.dtype == np.uint8
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    kc = np.ascontiguousarray(k_codes)
    vc = np.ascontiguousarray(v_codes)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros(q.shape, dtype=np.float64)
    ws = np.zeros(q.shape[:-1], dtype=np.float64) if return_wsum else None
    r, nr = _rows_arg(rows)
    lib().oracle_decode_fp8(_p(out), _p(_u16(q)), int(bf16), _p(kc), _p(vc), _p(ks), _p(vs), _p(bt),
                            bt.shape[1], _p(cl), B, Hq, Hkv, D, bs, float(np.float32(scale)),
                            int(window), nq, _p(r), nr, _p(ws))
    return (out, ws) if return_wsum else out
