"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/pa.h declares, and rejects bad arguments on the host before any
CUDA call (these calls never dereference the pointers they are given)."""
import ctypes
import os
import re

import pytest
import torch

from paged_kv_cache_179_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")

FAKE = 0x10000          # a 16-byte-aligned address that is never dereferenced
MISALIGNED = 0x10008


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    names = header_functions()
    assert len(names) == 24
    assert sorted(_abi.SIGNATURES) == names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    assert lib.pa_version() == 101
    assert lib.pa_status_string(0) == b"ok"
    assert b"workspace" in lib.pa_status_string(3)


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mbs=8, cl=FAKE, max_ctx=128, B=2, Hq=8,
             Hkv=2, D=64, bs=16, NB=32, scale=0.125, window=0, nq=1, dtype=0, splits=8,
             ws=FAKE, ws_bytes=1 << 20, flags=0)
    a.update(kw)
    return lib.pa_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mbs"], a["cl"],
                         a["max_ctx"], a["B"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"],
                         a["scale"], a["window"], a["nq"], a["dtype"], a["splits"], a["ws"],
                         a["ws_bytes"], a["flags"], None)


def test_decode_argument_errors(lib):
    assert _decode(lib, q=None) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, Hq=7) == _abi.PA_ERR_INVALID_ARG            # 7 % 2 != 0
    assert _decode(lib, splits=-1) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, flags=2) == _abi.PA_ERR_INVALID_ARG         # unknown flag bit
    assert _decode(lib, max_ctx=129) == _abi.PA_ERR_INVALID_ARG     # > mbs * 16
    assert _decode(lib, scale=float("nan")) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, dtype=3) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, window=-1) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, nq=0) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, nq=1025) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, q=MISALIGNED) == _abi.PA_ERR_INVALID_ARG
    assert _decode(lib, D=96) == _abi.PA_ERR_UNSUPPORTED
    assert _decode(lib, bs=32, mbs=4) == _abi.PA_ERR_UNSUPPORTED
    assert _decode(lib, Hq=66, Hkv=2) == _abi.PA_ERR_UNSUPPORTED    # group of 33
    assert _decode(lib, Hq=32, Hkv=1, ws_bytes=16) == _abi.PA_ERR_WORKSPACE   # 32 rows: larger
    assert _decode(lib, ws=None) == _abi.PA_ERR_WORKSPACE
    assert _decode(lib, ws_bytes=16) == _abi.PA_ERR_WORKSPACE
    assert _decode(lib, ws=FAKE + 16) == _abi.PA_ERR_WORKSPACE      # not 256-aligned
    assert _decode(lib, splits=1, ws=None) == _abi.PA_ERR_WORKSPACE # a single CTA needs one too
    assert _decode(lib, B=0) == _abi.PA_OK                          # nothing to do


def test_workspace_size_formula(lib):
    # partial rows: 2 per warp (4 warps per CTA), 8 query-head slots each, D floats +
    # (max, sum); each part rounded up to 256 bytes
    n = lib.pa_decode_workspace_size(2, 8, 64, 10)
    up = lambda x: (x + 255) // 256 * 256
    rows = 10 * 4 * 2 * 8
    acc, ml = rows * 64 * 4, rows * 2 * 4
    assert n == up(acc) + up(ml)
    assert lib.pa_decode_workspace_size(2, 8, 64, 1) > 0        # one CTA's 4 warps still split
    assert lib.pa_decode_workspace_size(2, 8, 64, -1) == 0      # invalid
    # launches holding 16 or 32 query rows per (sequence, kv head)
    f = lib.pa_decode_workspace_size_rows
    assert f(2, 8, 64, 10, 8) == n
    for qr, rows_per_piece in ((1, 8), (9, 16), (16, 16), (17, 32), (32, 32), (200, 32)):
        r = 10 * 4 * 2 * rows_per_piece
        assert f(2, 8, 64, 10, qr) == up(r * 64 * 4) + up(r * 2 * 4), qr
    assert f(2, 8, 64, 10, 0) == 0
    # the size does not grow with the batch (launches of 512 sequences share it)
    assert lib.pa_decode_workspace_size(5000, 8, 64, 10) == \
        lib.pa_decode_workspace_size(2, 8, 64, 10)


def test_append_and_quantize_argument_errors(lib):
    f = lib.pa_cache_append
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 16, 8, 0, None) == _abi.PA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 60, 16, 8, 0, None) == _abi.PA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, MISALIGNED, FAKE, FAKE, 4, 2, 64, 16, 8, 0, None) == _abi.PA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 64, 16, 8, 0, None) == _abi.PA_OK
    assert f(None, None, None, None, None, 0, 2, 64, 16, 8, 0, None) == _abi.PA_OK   # empty batch
    g = lib.pa_cache_append_fp8
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 96, 16, 8, 0, None) == _abi.PA_ERR_UNSUPPORTED
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 16, 8, 7, None) == _abi.PA_ERR_INVALID_ARG
    q = lib.pa_quantize_fp8
    assert q(None, None, FAKE, FAKE, FAKE, FAKE, 8, 2, 64, 16, None) == _abi.PA_ERR_INVALID_ARG
    assert q(FAKE, None, FAKE, None, FAKE, None, 8, 2, 64, 32, None) == _abi.PA_ERR_UNSUPPORTED
    assert lib.pa_e4m3_encode(FAKE, MISALIGNED, 10, None) == _abi.PA_ERR_INVALID_ARG


def test_handshake_argument_errors(lib):
    # the synced step needs its sync words; stream word operations a 4-aligned word
    args = [FAKE] * 8 + [8, FAKE, 128, 2, 8, 2, 64, 16, 32, 0.125, 0, 0, 8, FAKE, 1 << 20, 0]
    assert lib.pa_decode_step_synced(*args, None, None) == _abi.PA_ERR_INVALID_ARG
    # the pipelined step needs both its sync words and its copies
    sync = _abi.StepSync(FAKE, FAKE, FAKE, 1, 1)
    sp = ctypes.c_void_p(ctypes.addressof(sync))
    assert lib.pa_decode_step_pipelined(*args, sp, None, None) == _abi.PA_ERR_INVALID_ARG
    io = _abi.StepCopies(FAKE, FAKE, 0, FAKE, FAKE, 64, None, None, FAKE, 0)   # no input bytes
    iop = ctypes.c_void_p(ctypes.addressof(io))
    assert lib.pa_decode_step_pipelined(*args, sp, iop, None) == _abi.PA_ERR_INVALID_ARG
    assert lib.pa_stream_write_value(None, None, 1) == _abi.PA_ERR_INVALID_ARG
    assert lib.pa_stream_wait_value(None, FAKE + 2, 1) == _abi.PA_ERR_INVALID_ARG


def test_failure_path_hooks_check_their_limits(lib):
    # a limit of 0 or above the 2 s default is refused before any CUDA call
    assert lib.pa_test_wait_timeout(0, None) == _abi.PA_ERR_INVALID_ARG
    assert lib.pa_test_wait_timeout(3_000_000_000, None) == _abi.PA_ERR_INVALID_ARG
    m = lib.pa_test_merge_timeout
    assert m(FAKE, FAKE, 128, 2, 8, 2, 64, 0, 8, FAKE, 1 << 20, 0, None) == _abi.PA_ERR_INVALID_ARG
    assert m(FAKE, FAKE, 128, 2, 8, 2, 96, 0, 8, FAKE, 1 << 20, 1000, None) == \
        _abi.PA_ERR_UNSUPPORTED
    assert m(FAKE, FAKE, 128, 2, 8, 2, 64, 0, 8, FAKE, 16, 1000, None) == _abi.PA_ERR_WORKSPACE
    assert m(FAKE, FAKE, 128, 513, 8, 2, 64, 0, 8, FAKE, 1 << 20, 1000, None) == \
        _abi.PA_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a CUDA device")
def test_valid_call_without_device_reports_cuda_error(lib):
    assert _decode(lib) == _abi.PA_ERR_CUDA


def test_binding_refuses_cpu_tensors():
    t = torch.zeros(2, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        _abi.pa_decode(t, t, t, t, torch.zeros(2, 4, dtype=torch.int32),
                       torch.zeros(2, dtype=torch.int32), 64, 0.125, 64)


def test_early_copies_need_the_early_prologue():
    """PA_DECODE_EARLY_COPIES only together with PA_DECODE_EARLY_PROLOGUE: the
    binding refuses it alone (the library returns PA_ERR_INVALID_ARG)."""
    from paged_kv_cache_179_gb300 import _abi
    assert _abi._flags(True, True) == _abi.PA_DECODE_EARLY_PROLOGUE | _abi.PA_DECODE_EARLY_COPIES
    assert _abi._flags(True) == _abi.PA_DECODE_EARLY_PROLOGUE
    assert _abi._flags(False) == 0
    with pytest.raises(ValueError):
        _abi._flags(False, True)
