"""The C-ABI library: it builds for sm_103a, loads, exports every function
include/fa_fwd.h declares, and rejects bad arguments on the host before any
CUDA call (these calls use fake, never-dereferenced addresses)."""
import ctypes
import os
import re

import pytest

from exact_attention_forward_04_gb300 import SYMBOLS, _build, load_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_fwd.h")

FA_OK, INVALID, UNSUPPORTED, MISALIGNED = 0, -1, -2, -3


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_entry_points():
    names = _declared_functions()
    assert "fa_fwd" in names and "fa_fwd_host" in names and "fa_check_errors" in names


def test_every_declared_symbol_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa_fwd.h but not exported"
        assert name in SYMBOLS, f"{name} has no ctypes signature in the binding"


def test_binding_has_no_undeclared_symbols():
    assert set(SYMBOLS) == set(_declared_functions())


def test_version_and_status_strings(lib):
    assert lib.fa_version() >= 100
    assert lib.fa_status_string(0) == b"FA_OK"
    assert lib.fa_status_string(-5) == b"FA_ERR_TIMEOUT"
    assert lib.fa_status_string(12345) == b"FA_ERR_UNKNOWN"
    rec = (ctypes.c_uint * 4)()
    assert lib.fa_get_last_error_record(rec) == FA_OK
    assert list(rec) == [0, 0, 0, 0]
    assert lib.fa_get_last_error_record(None) == INVALID


# Fake device addresses: aligned, far apart, never dereferenced because
# validation fails before anything is enqueued.
Q, K, V, O, L = (0x10000000 * (i + 1) for i in range(5))
GOOD = dict(q=Q, k=K, v=V, o=O, lse=L, B=2, H=3, N=100, d=64, scale=0.125, causal=0)


def _call(lib, **kw):
    a = dict(GOOD, **kw)
    return lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                      a["d"], a["scale"], a["causal"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(v=0), INVALID),
    (dict(o=0), INVALID), (dict(lse=0), INVALID),
    (dict(B=0), INVALID), (dict(H=-1), INVALID), (dict(N=0), INVALID),
    (dict(causal=2), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(d=256), UNSUPPORTED), (dict(d=0), UNSUPPORTED),
    (dict(q=Q + 8), MISALIGNED), (dict(o=O + 2), MISALIGNED), (dict(lse=L + 2), MISALIGNED),
    (dict(o=Q), INVALID), (dict(lse=V + 64), INVALID), (dict(lse=O + 16), INVALID),
    (dict(B=65536, H=65536), UNSUPPORTED),
])
def test_validation_rejects(lib, kw, want):
    assert _call(lib, **kw) == want


def test_host_entry_rejects_null_host_buffers(lib):
    args = [0, K, V, O, L] + [Q + 0x1000, K + 0x1000, V + 0x1000, O + 0x1000, L + 0x1000]
    assert lib.fa_fwd_host(*args, 1, 1, 16, 64, 0.125, 0, None) == INVALID


W = 0x60000000  # fake workspace, far from the fake tensors above


def _split(lib, ws=W, ws_bytes=1 << 30, num_splits=4, **kw):
    # N = 2000: eight key tiles, so four splits are kept (a count above the
    # tiles is lowered, and one split would launch the one-pass kernel)
    a = dict(GOOD, N=2000, **kw)
    return lib.fa_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                              a["d"], a["scale"], a["causal"], num_splits, ws, ws_bytes, None)


def test_splitkv_workspace_size(lib):
    assert lib.fa_fwd_splitkv_workspace_size(2, 3, 100, 64, 4) == 4 * 2 * 3 * 100 * 65 * 4
    assert lib.fa_fwd_splitkv_workspace_size(1, 1, 7, 128, 1) == 7 * 129 * 4
    for bad in ((2, 3, 100, 96, 4), (2, 3, 100, 64, 0), (2, 3, 100, 64, 65),
                (0, 3, 100, 64, 2), (2, 3, 0, 64, 2)):
        assert lib.fa_fwd_splitkv_workspace_size(*bad) == 0, bad


@pytest.mark.parametrize("kw,want", [
    (dict(num_splits=-1), INVALID), (dict(num_splits=65), INVALID),
    (dict(ws=0), INVALID), (dict(ws_bytes=4 * 2 * 3 * 2000 * 65 * 4 - 1), INVALID),
    (dict(ws=W + 8), MISALIGNED), (dict(ws=Q), INVALID), (dict(ws=L - 4096), INVALID),
    (dict(q=0), INVALID), (dict(d=96), UNSUPPORTED), (dict(causal=3), INVALID),
])
def test_splitkv_validation_rejects(lib, kw, want):
    assert _split(lib, **kw) == want


DO, DQ, DK, DV, WS = (0x70000000 + 0x1000000 * i for i in range(5))


def _bwd(lib, dout=DO, dq=DQ, dk=DK, dv=DV, ws=WS, ws_bytes=1 << 30, **kw):
    a = dict(GOOD, **kw)
    return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], dout, dq, dk, dv, a["B"], a["H"],
                      a["N"], a["d"], a["scale"], a["causal"], ws, ws_bytes, None)


def test_bwd_workspace_size(lib):
    assert lib.fa_bwd_workspace_size(2, 3, 100, 64) == 2 * 3 * 128 * 8 + 256
    for bad in ((2, 3, 100, 96), (0, 3, 100, 64), (2, 3, 0, 128)):
        assert lib.fa_bwd_workspace_size(*bad) == 0, bad


@pytest.mark.parametrize("kw,want", [
    (dict(dout=0), INVALID), (dict(dq=0), INVALID), (dict(dk=0), INVALID), (dict(dv=0), INVALID),
    (dict(ws=0), INVALID), (dict(ws_bytes=2 * 3 * 128 * 8 + 255), INVALID),
    (dict(dq=DQ + 8), MISALIGNED), (dict(ws=WS + 4), MISALIGNED), (dict(dout=DO + 2), MISALIGNED),
    (dict(dq=Q), INVALID), (dict(dk=DO), INVALID), (dict(dv=DK), INVALID), (dict(ws=L), INVALID),
    (dict(q=0), INVALID), (dict(d=96), UNSUPPORTED), (dict(causal=2), INVALID),
    (dict(scale=-0.5), UNSUPPORTED),  # the forward takes a negative scale, the backward not
])
def test_bwd_validation_rejects(lib, kw, want):
    assert _bwd(lib, **kw) == want


def test_ptxas_report_has_no_spills(lib):
    rep = open(os.path.join(os.path.dirname(_build.LIB_PATH), "ptxas_report.txt")).read()
    assert "sm_103a" in rep
    spills = re.findall(r"(\d+) bytes spill stores", rep)
    assert spills and all(int(s) == 0 for s in spills), spills


def test_e4m3_bytes(lib):
    assert lib.fa_e4m3_bytes(2, 3, 100, 128, 0) == 2 * 3 * 100 * 128
    assert lib.fa_e4m3_bytes(2, 3, 100, 128, 1) == 2 * 3 * 112 * 128  # keys padded to 16
    assert lib.fa_e4m3_bytes(1, 1, 16, 64, 1) == 16 * 64
    for bad in ((2, 3, 100, 96, 0), (0, 3, 100, 64, 0), (2, 3, 0, 64, 1), (2, 3, 100, 64, 2)):
        assert lib.fa_e4m3_bytes(*bad) == 0, bad


X, X8, DS = 0x40000000, 0x50000000, 0x60000000


def _quant(lib, x=X, x8=X8, ds=DS, B=2, H=3, N=100, d=128, keys_last=0):
    return lib.fa_quantize_e4m3(x, x8, ds, B, H, N, d, keys_last, None)


@pytest.mark.parametrize("kw,want", [
    (dict(x=0), INVALID), (dict(x8=0), INVALID), (dict(ds=0), INVALID), (dict(B=0), INVALID),
    (dict(N=-1), INVALID), (dict(keys_last=2), INVALID), (dict(d=96), UNSUPPORTED),
    (dict(B=300, H=300), UNSUPPORTED), (dict(x=X + 8), MISALIGNED), (dict(x8=X8 + 4), MISALIGNED),
    (dict(ds=DS + 2), MISALIGNED), (dict(x8=X + 64), INVALID), (dict(ds=X8 + 16), INVALID),
    (dict(ds=X + 1024), INVALID),
])
def test_quantize_validation_rejects(lib, kw, want):
    assert _quant(lib, **kw) == want


Q8, K8, V8, DQS, DKS, DVS = (0x10000000 * (i + 1) for i in range(6))
O8, L8 = 0x70000000, 0x78000000


def _fwd8(lib, q=Q8, k=K8, v=V8, dq=DQS, dk=DKS, dv=DVS, o=O8, lse=L8, B=2, H=3, N=100, d=128,
          scale=0.088, causal=0):
    return lib.fa_fwd_e4m3(q, k, v, dq, dk, dv, o, lse, B, H, N, d, scale, causal, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), INVALID), (dict(v=0), INVALID), (dict(dq=0), INVALID), (dict(dv=0), INVALID),
    (dict(o=0), INVALID), (dict(lse=0), INVALID), (dict(B=0), INVALID), (dict(causal=2), INVALID),
    (dict(scale=float("nan")), INVALID), (dict(scale=-1.0), UNSUPPORTED),
    (dict(d=32), UNSUPPORTED), (dict(d=96), UNSUPPORTED),
    (dict(q=Q8 + 8), MISALIGNED), (dict(v=V8 + 1), MISALIGNED), (dict(o=O8 + 4), MISALIGNED),
    (dict(dk=DKS + 2), MISALIGNED), (dict(lse=L8 + 1), MISALIGNED),
    (dict(o=Q8 + 256), INVALID), (dict(lse=V8 + 64), INVALID), (dict(o=DVS), INVALID),
    (dict(lse=O8 + 1024), INVALID),
])
def test_fwd_e4m3_validation_rejects(lib, kw, want):
    assert _fwd8(lib, **kw) == want


def test_selftest_rejects_bad_timeout(lib):
    assert lib.fa_selftest_wait_timeout(0, None) == INVALID
    assert lib.fa_selftest_wait_timeout(1000001, None) == INVALID


def _quant3(lib, q=X, k=X + 0x100000, v=X + 0x200000, q8=X8, k8=X8 + 0x100000, vt8=X8 + 0x200000,
            dq=DS, dk=DS + 0x1000, dv=DS + 0x2000, B=2, H=3, N=100, d=128):
    return lib.fa_quantize_qkv_e4m3(q, k, v, q8, k8, vt8, dq, dk, dv, B, H, N, d, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), INVALID), (dict(vt8=0), INVALID), (dict(dv=0), INVALID), (dict(B=0), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(B=300, H=300), UNSUPPORTED), (dict(k=X + 8), MISALIGNED),
    (dict(vt8=X8 + 4), MISALIGNED), (dict(dk=DS + 2), MISALIGNED),
    (dict(k8=X8 + 64), INVALID),        # overlaps q8
    (dict(dv=DS), INVALID),             # overlaps descale_q
    (dict(q8=X + 0x100000), INVALID),   # overlaps k
    (dict(dq=X8 + 0x200000), INVALID),  # overlaps vt8
])
def test_quantize_qkv_validation_rejects(lib, kw, want):
    assert _quant3(lib, **kw) == want


UW = 0x7c000000  # fake unfused workspace


def _unf(lib, ws=UW, ws_bytes=1 << 30, **kw):
    a = dict(GOOD, **kw)
    return lib.fa_attn_unfused(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                               a["d"], a["scale"], a["causal"], ws, ws_bytes, None)


def test_unfused_workspace_size(lib):
    # S fp32 then P bf16, rows padded to 8 elements, S padded to 256 bytes
    cells = 2 * 3 * 100 * 104
    assert lib.fa_attn_unfused_workspace_size(2, 3, 100, 64) == (cells * 4 + 255) // 256 * 256 + cells * 2
    cells = 1 * 1 * 8 * 8
    assert lib.fa_attn_unfused_workspace_size(1, 1, 8, 128) == 256 + cells * 2
    for bad in ((2, 3, 100, 96), (0, 3, 100, 64), (2, 3, 0, 128), (1, 1, -5, 64)):
        assert lib.fa_attn_unfused_workspace_size(*bad) == 0, bad


@pytest.mark.parametrize("kw,want", [
    (dict(ws=0), INVALID), (dict(ws_bytes=2 * 3 * 100 * 104 * 6 - 1), INVALID),
    (dict(ws=UW + 8), MISALIGNED), (dict(ws=Q), INVALID), (dict(ws=L - 4096), INVALID),
    (dict(q=0), INVALID), (dict(lse=0), INVALID), (dict(d=96), UNSUPPORTED),
    (dict(causal=2), INVALID), (dict(scale=float("nan")), INVALID), (dict(N=0), INVALID),
    (dict(o=Q), INVALID), (dict(q=Q + 8), MISALIGNED),
])
def test_unfused_validation_rejects(lib, kw, want):
    assert _unf(lib, **kw) == want
