"""Exact attention forward pass for GB300 (sm_103a).

    O = softmax(scale * Q K^T [+ causal mask]) V,   L = logsumexp of each row

computed by hand-written CUDA (TMA, tcgen05 MMAs with tensor-memory
accumulators) behind the C ABI declared in ``include/fa_fwd.h``.  This module
only marshals arguments to that library through ctypes; PyTorch supplies the
device memory and the stream.  There is no fallback: if the library is not
built, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "FAError", "forward", "forward_into", "forward_host", "forward_splitkv", "fa_fwd",
    "fa_fwd_host", "fa_fwd_splitkv", "splitkv_workspace_size", "splitkv_num_splits",
    "forward_splitkv_noalloc", "backward", "bwd_workspace_size", "quantize_e4m3",
    "forward_e4m3", "e4m3_bytes", "quantize_qkv_e4m3", "attention_unfused",
    "unfused_workspace_size", "unfused_intermediates",
    "check_errors", "status_string", "library_path", "load_library", "SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libfa_fwd.so")

# Every function the C ABI exports, with its ctypes signature.
_c = ctypes
SYMBOLS = {
    "fa_fwd": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                          _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_float, _c.c_int,
                          _c.c_void_p]),
    "fa_fwd_host": (_c.c_int, [_c.c_void_p] * 10 + [_c.c_int] * 4 +
                    [_c.c_float, _c.c_int, _c.c_void_p]),
    "fa_fwd_splitkv": (_c.c_int, [_c.c_void_p] * 5 + [_c.c_int] * 4 +
                       [_c.c_float, _c.c_int, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "fa_fwd_splitkv_workspace_size": (_c.c_size_t, [_c.c_int] * 5),
    "fa_fwd_splitkv_num_splits": (_c.c_int, [_c.c_int] * 4),
    "fa_fwd_splitkv_noalloc": (_c.c_int, [_c.c_void_p] * 5 + [_c.c_int] * 4 +
                               [_c.c_float, _c.c_int, _c.c_int, _c.c_void_p]),
    "fa_fwd_splitkv_noalloc_capacity": (_c.c_size_t, []),
    "fa_bwd": (_c.c_int, [_c.c_void_p] * 9 + [_c.c_int] * 4 +
               [_c.c_float, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "fa_bwd_workspace_size": (_c.c_size_t, [_c.c_int] * 4),
    "fa_e4m3_bytes": (_c.c_size_t, [_c.c_int] * 5),
    "fa_quantize_e4m3": (_c.c_int, [_c.c_void_p] * 3 + [_c.c_int] * 5 + [_c.c_void_p]),
    "fa_quantize_qkv_e4m3": (_c.c_int, [_c.c_void_p] * 9 + [_c.c_int] * 4 + [_c.c_void_p]),
    "fa_fwd_e4m3": (_c.c_int, [_c.c_void_p] * 8 + [_c.c_int] * 4 +
                    [_c.c_float, _c.c_int, _c.c_void_p]),
    "fa_attn_unfused": (_c.c_int, [_c.c_void_p] * 5 + [_c.c_int] * 4 +
                        [_c.c_float, _c.c_int, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    "fa_attn_unfused_workspace_size": (_c.c_size_t, [_c.c_int] * 4),
    "fa_check_errors": (_c.c_int, [_c.c_void_p]),
    "fa_selftest_wait_timeout": (_c.c_int, [_c.c_uint, _c.c_void_p]),
    "fa_status_string": (_c.c_char_p, [_c.c_int]),
    "fa_get_last_cuda_error": (_c.c_int, []),
    "fa_get_last_error_record": (_c.c_int, [_c.POINTER(_c.c_uint)]),
    "fa_version": (_c.c_int, []),
}

STATUS = {0: "FA_OK", -1: "FA_ERR_INVALID_ARG", -2: "FA_ERR_UNSUPPORTED",
          -3: "FA_ERR_MISALIGNED", -4: "FA_ERR_CUDA", -5: "FA_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of libfa_fwd.so."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise FAError(-4, "load_library",
                          f"{p} is missing; build it with "
                          "`python -m exact_attention_forward_04_gb300._build`")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SYMBOLS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().fa_status_string(status).decode()


def _raise(status: int, where: str):
    lib = load_library()
    detail = ""
    if status == -4:
        detail = f"cudaError {lib.fa_get_last_cuda_error()}"
    elif status == -5:
        rec = (ctypes.c_uint * 4)()
        lib.fa_get_last_error_record(rec)
        detail = f"record code={rec[0]} site={rec[1]} block={rec[2]} tile={rec[3]}"
    raise FAError(status, where, detail)


def fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal, stream) -> int:
    """Raw C-ABI call on device pointers (ints); returns the status code."""
    return load_library().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(N),
                                 int(d), float(scale), int(bool(causal)), stream)


def fa_fwd_host(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, dq, dk, dv, do_, dlse,
                B, H, N, d, scale, causal, stream) -> int:
    """Raw C-ABI call on host buffers with device staging buffers."""
    return load_library().fa_fwd_host(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, dq, dk, dv, do_,
                                      dlse, int(B), int(H), int(N), int(d), float(scale),
                                      int(bool(causal)), stream)


def fa_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal, num_splits,
                   ws_ptr, ws_bytes, stream) -> int:
    """Raw C-ABI call of the split key/value forward; returns the status."""
    return load_library().fa_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H),
                                         int(N), int(d), float(scale), int(bool(causal)),
                                         int(num_splits), ws_ptr, int(ws_bytes), stream)


def splitkv_workspace_size(B, H, N, d, num_splits) -> int:
    """Workspace bytes fa_fwd_splitkv needs (0 for out-of-range arguments)."""
    return int(load_library().fa_fwd_splitkv_workspace_size(int(B), int(H), int(N), int(d),
                                                            int(num_splits)))


def splitkv_num_splits(B, H, N, causal=False) -> int:
    """The split count num_splits = 0 picks on the current device."""
    n = load_library().fa_fwd_splitkv_num_splits(int(B), int(H), int(N), int(bool(causal)))
    if n < 0:
        _raise(n, "fa_fwd_splitkv_num_splits")
    return n


def check_errors(stream=None) -> None:
    """Synchronise the stream and raise FAError if a device-side bounded wait
    expired since the last check."""
    st = load_library().fa_check_errors(_stream_handle(stream))
    if st != 0:
        _raise(st, "fa_check_errors")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_inputs(q, k, v):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, d], got shape {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if not (q.shape == k.shape == v.shape):
        raise ValueError(f"q, k, v shapes differ: {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")


def forward_into(q, k, v, o, lse, scale=None, causal=False, stream=None) -> None:
    """Enqueue the forward pass into caller-provided o (bf16 [B,H,N,d]) and
    lse (fp32 [B,H,N]) on `stream` (default: torch's current stream)."""
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if not q.is_cuda or not (q.device == k.device == v.device == o.device == lse.device):
        raise ValueError("q, k, v, o, lse must be CUDA tensors on one device")
    st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                B, H, N, d, scale, causal, _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_fwd")


def forward(q, k, v, scale=None, causal=False, stream=None):
    """Return (o, lse): o bf16 [B,H,N,d], lse fp32 [B,H,N] (natural log)."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    forward_into(q, k, v, o, lse, scale=scale, causal=causal, stream=stream)
    return o, lse


def forward_splitkv(q, k, v, scale=None, causal=False, num_splits=0, workspace=None, stream=None):
    """Forward with the key blocks of each query tile split into up to
    ``num_splits`` ranges (0: the library's choice), merged by logsumexp.
    ``workspace`` (a CUDA tensor of at least splitkv_workspace_size bytes)
    may be passed to reuse memory; otherwise it is allocated here by torch.
    Returns (o, lse) like ``forward``."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if not q.is_cuda or not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be CUDA tensors on one device")
    with torch.cuda.device(q.device):
        if num_splits == 0:
            num_splits = splitkv_num_splits(B, H, N, causal)
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
        need = splitkv_workspace_size(B, H, N, d, num_splits) if num_splits > 1 else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, scale, causal, num_splits, ws_ptr, ws_bytes,
                            _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_fwd_splitkv")
    return o, lse


def forward_splitkv_noalloc(q, k, v, scale=None, causal=False, num_splits=0, stream=None):
    """``forward_splitkv`` with the partials in the library's fixed device
    scratch (no workspace argument, nothing allocated for it).  Calls that
    may overlap on different streams must not share it."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if not q.is_cuda or not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be CUDA tensors on one device")
    with torch.cuda.device(q.device):
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
        st = load_library().fa_fwd_splitkv_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), int(num_splits), _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_fwd_splitkv_noalloc")
    return o, lse


def backward(q, k, v, o, lse, dout, scale=None, causal=False, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of the attention forward given dout, the
    gradient of o; q, k, v, o, lse are the forward's inputs and outputs
    (``forward``), all on one CUDA device.  ``workspace`` (a CUDA tensor of
    at least bwd_workspace_size bytes) may be passed to reuse memory;
    otherwise torch allocates it here."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for name, t in (("o", o), ("dout", dout)):
        if t.dtype != torch.bfloat16 or t.shape != q.shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    if not q.is_cuda or not all(t.device == q.device for t in (k, v, o, lse, dout)):
        raise ValueError("all tensors must be CUDA tensors on one device")
    with torch.cuda.device(q.device):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        need = bwd_workspace_size(B, H, N, d)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        st = load_library().fa_bwd(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_bwd")
    return dq, dk, dv


def bwd_workspace_size(B, H, N, d) -> int:
    """Workspace bytes fa_bwd needs (0 for invalid sizes)."""
    return int(load_library().fa_bwd_workspace_size(int(B), int(H), int(N), int(d)))


def e4m3_bytes(B, H, N, d, keys_last=False) -> int:
    """Bytes of the E4M3 codes of a [B, H, N, d] tensor (0 if out of range)."""
    return int(load_library().fa_e4m3_bytes(int(B), int(H), int(N), int(d), int(bool(keys_last))))


def quantize_e4m3(x, keys_last=False, stream=None):
    """E4M3 codes and per-(batch, head) descales of a bf16 [B, H, N, d] CUDA
    tensor.  Returns (codes, descale): codes uint8 [B, H, N, d], or with
    ``keys_last`` [B, H, d, P] (P = N rounded up to 16, columns >= N zero),
    the layout ``forward_e4m3`` takes for V; descale fp32 [B, H]."""
    import torch
    _check_inputs(x, x, x)
    B, H, N, d = x.shape
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    shape = (B, H, d, (N + 15) // 16 * 16) if keys_last else (B, H, N, d)
    with torch.cuda.device(x.device):
        codes = torch.empty(shape, dtype=torch.uint8, device=x.device)
        descale = torch.empty(B, H, dtype=torch.float32, device=x.device)
        st = load_library().fa_quantize_e4m3(x.data_ptr(), codes.data_ptr(), descale.data_ptr(),
                                             B, H, N, d, int(bool(keys_last)),
                                             _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_quantize_e4m3")
    return codes, descale


def quantize_qkv_e4m3(q, k, v, stream=None):
    """``quantize_e4m3`` of q and k (rows) and of v (keys-last) in one call
    (four launches).  Returns (q8, k8, vt8, descale_q, descale_k, descale_v),
    ready for ``forward_e4m3``."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if not q.is_cuda or not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be CUDA tensors on one device")
    with torch.cuda.device(q.device):
        q8 = torch.empty(B, H, N, d, dtype=torch.uint8, device=q.device)
        k8 = torch.empty_like(q8)
        vt8 = torch.empty(B, H, d, (N + 15) // 16 * 16, dtype=torch.uint8, device=q.device)
        ds = [torch.empty(B, H, dtype=torch.float32, device=q.device) for _ in range(3)]
        st = load_library().fa_quantize_qkv_e4m3(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(),
            ds[0].data_ptr(), ds[1].data_ptr(), ds[2].data_ptr(), B, H, N, d, _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_quantize_qkv_e4m3")
    return q8, k8, vt8, ds[0], ds[1], ds[2]


def forward_e4m3(q8, k8, vt8, descale_q, descale_k, descale_v, scale=None, causal=False,
                 stream=None):
    """The forward on E4M3 codes: q8, k8 uint8 [B, H, N, d], vt8 uint8
    keys-last [B, H, d, P] (``quantize_e4m3(v, keys_last=True)``), descales
    fp32 [B, H].  Head dim 64 or 128.  Returns (o bf16 [B, H, N, d], lse fp32
    [B, H, N])."""
    import torch
    for name, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or t.dim() != 4 \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous uint8 [B, H, ., .] tensor")
    B, H, N, d = q8.shape
    if tuple(k8.shape) != (B, H, N, d) or tuple(vt8.shape) != (B, H, d, (N + 15) // 16 * 16):
        raise ValueError(f"shapes: q8 {tuple(q8.shape)} k8 {tuple(k8.shape)} vt8 {tuple(vt8.shape)}")
    for name, t in (("descale_q", descale_q), ("descale_k", descale_k), ("descale_v", descale_v)):
        if t.dtype != torch.float32 or tuple(t.shape) != (B, H) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 [B, H] tensor")
    if not q8.is_cuda or not all(t.device == q8.device
                                 for t in (k8, vt8, descale_q, descale_k, descale_v)):
        raise ValueError("all tensors must be CUDA tensors on one device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(q8.device):
        o = torch.empty(B, H, N, d, dtype=torch.bfloat16, device=q8.device)
        lse = torch.empty(B, H, N, dtype=torch.float32, device=q8.device)
        st = load_library().fa_fwd_e4m3(
            q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), descale_q.data_ptr(),
            descale_k.data_ptr(), descale_v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_fwd_e4m3")
    return o, lse


def unfused_workspace_size(B, H, N, d) -> int:
    """Workspace bytes fa_attn_unfused needs (0 for invalid sizes)."""
    return int(load_library().fa_attn_unfused_workspace_size(int(B), int(H), int(N), int(d)))


def attention_unfused(q, k, v, scale=None, causal=False, workspace=None, stream=None):
    """Standard attention in three kernels with S (fp32) and P (bf16) in
    device memory: the computation the fused ``forward`` replaces, for
    measuring what writing S and P costs.  ``workspace`` (a CUDA tensor of at
    least unfused_workspace_size bytes) may be passed to reuse memory and to
    read S and P afterwards (``unfused_intermediates``); otherwise torch
    allocates it here.  Returns (o, lse) like ``forward``."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if not q.is_cuda or not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be CUDA tensors on one device")
    with torch.cuda.device(q.device):
        need = unfused_workspace_size(B, H, N, d)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
        st = load_library().fa_attn_unfused(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != 0:
        _raise(st, "fa_attn_unfused")
    return o, lse


def unfused_intermediates(workspace, B, H, N):
    """Views of S (fp32) and P (bf16), each [B, H, N, N], in a workspace that
    ``attention_unfused`` has filled (the layout fa_attn_unfused documents:
    rows padded to a multiple of 8 elements, S padded to 256 bytes)."""
    import torch
    np_ = (N + 7) // 8 * 8
    cells = B * H * N * np_
    s_bytes = (cells * 4 + 255) // 256 * 256
    raw = workspace.view(torch.uint8).reshape(-1)
    S = raw[:cells * 4].view(torch.float32).view(B, H, N, np_)[..., :N]
    P = raw[s_bytes:s_bytes + cells * 2].view(torch.bfloat16).view(B, H, N, np_)[..., :N]
    return S, P


def forward_host(q, k, v, scale=None, causal=False, stream=None, staging=None, out=None):
    """Forward on HOST tensors through the C ABI's host entry point: the
    host-to-device copies, the kernel and the device-to-host copies are all
    enqueued on one stream.  ``staging`` (dq, dk, dv, do, dlse) and ``out``
    (o, lse) may be passed to reuse buffers; host tensors should be pinned.
    Returns (o, lse) on the host after synchronising the stream."""
    import torch
    _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if staging is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        staging = (torch.empty_like(q, device=dev), torch.empty_like(k, device=dev),
                   torch.empty_like(v, device=dev), torch.empty_like(q, device=dev),
                   torch.empty(B, H, N, dtype=torch.float32, device=dev))
    if out is None:
        out = (torch.empty(B, H, N, d, dtype=torch.bfloat16, pin_memory=True),
               torch.empty(B, H, N, dtype=torch.float32, pin_memory=True))
    o, lse = out
    h = _stream_handle(stream)
    st = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     *(t.data_ptr() for t in staging), B, H, N, d, scale, causal, h)
    if st != 0:
        _raise(st, "fa_fwd_host")
    st = load_library().fa_check_errors(h)
    if st != 0:
        _raise(st, "fa_check_errors")
    return o, lse
