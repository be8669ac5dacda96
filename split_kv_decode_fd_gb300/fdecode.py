"""ctypes binding of libfdecode (include/fdecode.h), taking PyTorch tensors.

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
CPU fallback: calls with CPU tensors raise, and a missing library raises.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "FdError", "KvDesc", "library_path", "load_library", "workspace_bytes", "split_size", "plan_pieces",
    "Workspace", "decode", "decode_rows", "append_decode", "prefill", "attend", "attend_backend", "decode_host", "HostDecoder", "decode_static", "static_status", "split_partial", "combine", "workspace_status",
]

FD_OK, FD_ERR_INVALID_ARG, FD_ERR_UNSUPPORTED, FD_ERR_WORKSPACE_TOO_SMALL = 0, 1, 2, 3
FD_ERR_BAD_INDEX, FD_ERR_CUDA, FD_ERR_TIMEOUT = 4, 5, 6
FD_F32, FD_BF16 = 0, 1
FD_KV_CONTIGUOUS, FD_KV_PAGED = 0, 1
FD_SPLITS_AUTO = 0
FD_AUTO_MAX_BATCH = 1024

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None
_LOCK = threading.Lock()


class FdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib().fd_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


class KvDesc(ctypes.Structure):
    _fields_ = [
        ("layout", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("capacity", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
        ("max_pages_per_seq", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
    ]


def library_path() -> str:
    return os.environ.get("FDECODE_LIB", os.path.join(_HERE, "libfdecode.so"))


def load_library(path: Optional[str] = None):
    """Load libfdecode.so (built in-tree by ``split_kv_decode_fd_gb300/build.py``)."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = path or library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libfdecode.so not found at {path}; build it with "
                               "`python split_kv_decode_fd_gb300/build.py`")
        lib = ctypes.CDLL(path)
        c_i32, c_i64, c_sz, vp, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
        kvp = ctypes.POINTER(KvDesc)
        sig = {
            "fd_workspace_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
            "fd_workspace_init": (ctypes.c_int, [vp, c_sz, vp]),
            "fd_workspace_status": (ctypes.c_int, [vp, c_sz, vp]),
            "fd_split_size": (c_i32, [c_i32, c_i32]),
            "fd_decode": (ctypes.c_int, [vp, kvp, vp, vp, c_i32, c_i32, c_i32, vp, c_i32, c_i32, f32, c_i32, vp,
                                         c_sz, vp]),
            "fd_split_partial": (ctypes.c_int, [vp, kvp, c_i32, c_i32, c_i32, vp, c_i32, c_i32, f32, c_i32, vp,
                                                vp, vp, vp]),
            "fd_combine": (ctypes.c_int, [vp, vp, vp, vp, vp, c_i32, c_i32, c_i32, c_i32, vp]),
            "fd_decode_host": (ctypes.c_int, [vp, kvp, vp, vp, c_i32, c_i32, c_i32, vp, c_i32, c_i32, f32, c_i32,
                                              vp, c_sz, vp]),
            "fd_plan_pieces": (c_i64, [c_i32, c_i32, c_i32, c_i32, vp, c_i32, c_i32, c_i32, vp, c_i64]),
            "fd_decode_static": (ctypes.c_int, [vp, kvp, vp, vp, c_i32, c_i32, c_i32, vp, c_i32, c_i32, f32,
                                                c_i32, vp]),
            "fd_static_status": (ctypes.c_int, [vp]),
            "fd_decode_rows": (ctypes.c_int, [vp, c_i32, c_i32, kvp, vp, vp, c_i32, c_i32, c_i32, vp, c_i32,
                                              c_i32, f32, c_i32, vp, c_sz, vp]),
            "fd_append_decode": (ctypes.c_int, [vp, vp, vp, kvp, vp, vp, c_i32, c_i32, c_i32, vp, c_i32, c_i32, f32,
                                                c_i32, vp, c_sz, vp]),
            "fd_prefill": (ctypes.c_int, [vp, c_i32, c_i32, kvp, vp, vp, c_i32, c_i32, c_i32, vp, c_i32, c_i32, f32,
                                          vp, c_sz, vp]),
            "fd_attend": (ctypes.c_int, [vp, c_i32, c_i32, kvp, vp, vp, c_i32, c_i32, c_i32, vp, c_i32, c_i32, f32,
                                         c_i32, vp, c_sz, vp, ctypes.POINTER(c_i32)]),
            "fd_attend_backend": (c_i32, [c_i32, c_i32, c_i32, c_i32, c_i32]),
            "fd_backend_name": (ctypes.c_char_p, [c_i32]),
            "fd_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "fd_version": (c_i32, []),
            "fd_debug_stall": (None, [c_i32, c_i64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
        return lib


def _lib():
    return load_library()


def _check(status: int, where: str):
    if status != FD_OK:
        raise FdError(status, where)


# ------------------------------------------------------------------ host-only
def workspace_bytes(B, Hq, Hkv, D, n_splits=FD_SPLITS_AUTO, num_sms=0) -> int:
    n = _lib().fd_workspace_bytes(B, Hq, Hkv, D, n_splits, num_sms)
    if n == 0:
        raise FdError(FD_ERR_INVALID_ARG, "fd_workspace_bytes")
    return int(n)


def split_size(max_seq_len: int, n_splits: int) -> int:
    return int(_lib().fd_split_size(max_seq_len, n_splits))


def plan_pieces(B, Hq, Hkv, seq_lens: Optional[Sequence[int]], max_seq_len, n_splits=0, grid=152,
                kv_dtype="bf16") -> np.ndarray:
    """The pieces fd_decode runs: int32 [n, 7] of (cta, b, vkv, tok_begin, tok_end, slot, pieces_of_sequence)."""
    lib = _lib()
    dt = {"bf16": FD_BF16, "f32": FD_F32}[kv_dtype]
    lens = None if seq_lens is None else np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    lp = None if lens is None else lens.ctypes.data
    n = lib.fd_plan_pieces(B, Hq, Hkv, dt, lp, max_seq_len, n_splits, grid, None, 0)
    if n < 0:
        raise FdError(FD_ERR_INVALID_ARG, "fd_plan_pieces")
    buf = np.zeros((max(n, 1), 7), dtype=np.int32)
    lib.fd_plan_pieces(B, Hq, Hkv, dt, lp, max_seq_len, n_splits, grid, buf.ctypes.data, n)
    return buf[:n]


# ------------------------------------------------------------------ device
def _torch():
    import torch
    return torch


def _stream_handle(device, stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _need_cuda(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libfdecode has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _kv_desc(k, v, block_table):
    torch = _torch()
    _need_cuda(k, "k")
    _need_cuda(v, "v")
    if k.dtype != v.dtype or k.shape != v.shape:
        raise ValueError("k and v must have the same dtype and shape")
    dt = {torch.bfloat16: FD_BF16, torch.float32: FD_F32}.get(k.dtype)
    if dt is None:
        raise ValueError(f"unsupported KV dtype {k.dtype}")
    d = KvDesc()
    d.dtype = dt
    d.k = k.data_ptr()
    d.v = v.data_ptr()
    if block_table is None:
        d.layout = FD_KV_CONTIGUOUS
        d.capacity = k.shape[2]
    else:
        _need_cuda(block_table, "block_table", torch.int32)
        d.layout = FD_KV_PAGED
        d.block_table = block_table.data_ptr()
        d.max_pages_per_seq = block_table.shape[1]
        d.page_size = k.shape[2]
        d.num_pages = k.shape[0]
    return d


class Workspace:
    """Zero-initialised device scratch for the kernels, grown on demand.

    It holds the error word, the decode kernels' arrival counters and partial
    states, and the prefill's item queue, all left at zero between calls: calls
    that may run at the same time (on different streams) need a Workspace each.
    The default one, used when none is passed, is shared per device.
    """

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int, device):
        torch = _torch()
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self.buf


_DEFAULT_WS = {}


def _default_workspace(device) -> Workspace:
    key = (device.type, device.index)
    if key not in _DEFAULT_WS:
        _DEFAULT_WS[key] = Workspace(device)
    return _DEFAULT_WS[key]


def _geometry(q, k, block_table, seq_lens, max_seq_len):
    if q.dim() != 3:
        raise ValueError("q must be [B, Hq, D]")
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    if k.shape[3] != D:
        raise ValueError("head_dim of q and k differ")
    if max_seq_len is None:
        max_seq_len = k.shape[2] if block_table is None else block_table.shape[1] * k.shape[2]
    return B, Hq, Hkv, D, int(max_seq_len)


def decode(q, k, v, *, seq_lens=None, max_seq_len=None, block_table=None, scale=None, n_splits=FD_SPLITS_AUTO,
           out=None, lse=None, return_lse=True, workspace: Optional[Workspace] = None, stream=None):
    """Split-KV decode attention (``fd_decode``).

    q ``[B, Hq, D]`` fp32 CUDA; k, v contiguous ``[B, Hkv, T_cap, D]`` or, with
    ``block_table`` ``[B, max_pages]`` int32, paged ``[num_pages, Hkv, page, D]``
    (bf16 or fp32).  Returns ``(out [B, Hq, D], lse [B, Hq] or None)``.
    """
    torch = _torch()
    _need_cuda(q, "q", torch.float32)
    kv = _kv_desc(k, v, block_table)
    B, Hq, Hkv, D, max_seq_len = _geometry(q, k, block_table, seq_lens, max_seq_len)
    if seq_lens is not None:
        _need_cuda(seq_lens, "seq_lens", torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    _need_cuda(out, "out", torch.float32)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    ws = workspace or _default_workspace(q.device)
    nbytes = workspace_bytes(B, Hq, Hkv, D, n_splits)
    buf = ws.get(nbytes, q.device)
    st = _lib().fd_decode(q.data_ptr(), ctypes.byref(kv), out.data_ptr(), lse.data_ptr() if lse is not None else None,
                          B, Hq, Hkv, seq_lens.data_ptr() if seq_lens is not None else None, max_seq_len, D,
                          float(scale), int(n_splits), buf.data_ptr(), buf.numel(), _stream_handle(q.device, stream))
    _check(st, "fd_decode")
    return out, lse


def decode_rows(q, k, v, *, causal=True, seq_lens=None, max_seq_len=None, block_table=None, scale=None,
                n_splits=FD_SPLITS_AUTO, out=None, lse=None, return_lse=True, workspace: Optional[Workspace] = None,
                stream=None):
    """``fd_decode_rows``: q ``[B, Hq, n_q, D]`` (n_q query rows per head); returns
    ``(out [B, Hq, n_q, D], lse [B, Hq, n_q] or None)``.  With ``causal`` row i sees
    keys ``t < L_b - (n_q - 1 - i)``.
    """
    torch = _torch()
    _need_cuda(q, "q", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, Hq, n_q, D]")
    kv = _kv_desc(k, v, block_table)
    B, Hq, n_q, D = q.shape
    Hkv = k.shape[1]
    if max_seq_len is None:
        max_seq_len = k.shape[2] if block_table is None else block_table.shape[1] * k.shape[2]
    if seq_lens is not None:
        _need_cuda(seq_lens, "seq_lens", torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, n_q), dtype=torch.float32, device=q.device)
    ws = workspace or _default_workspace(q.device)
    buf = ws.get(workspace_bytes(B, Hq * n_q, Hkv, D, n_splits), q.device)
    st = _lib().fd_decode_rows(q.data_ptr(), int(n_q), int(bool(causal)), ctypes.byref(kv), out.data_ptr(),
                               lse.data_ptr() if lse is not None else None, B, Hq, Hkv,
                               seq_lens.data_ptr() if seq_lens is not None else None, int(max_seq_len), D,
                               float(scale), int(n_splits), buf.data_ptr(), buf.numel(),
                               _stream_handle(q.device, stream))
    _check(st, "fd_decode_rows")
    return out, lse


def append_decode(q, k, v, k_new, v_new, *, seq_lens=None, max_seq_len=None, block_table=None, scale=None,
                  n_splits=FD_SPLITS_AUTO, out=None, lse=None, return_lse=True,
                  workspace: Optional[Workspace] = None, stream=None):
    """``fd_append_decode``: write ``k_new``/``v_new`` (``[B, Hkv, D]``, cache dtype) at
    position ``L_b`` of every sequence, then decode over ``L_b + 1`` keys.

    ``seq_lens``/``max_seq_len`` are the lengths before the append (default
    ``max_seq_len``: the cache capacity minus one).  ``k`` and ``v`` are written.
    Returns ``(out, lse)``.
    """
    torch = _torch()
    _need_cuda(q, "q", torch.float32)
    kv = _kv_desc(k, v, block_table)
    _need_cuda(k_new, "k_new", k.dtype)
    _need_cuda(v_new, "v_new", k.dtype)
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError("k_new and v_new must be [B, Hkv, D]")
    if max_seq_len is None:
        cap = k.shape[2] if block_table is None else block_table.shape[1] * k.shape[2]
        max_seq_len = cap - 1
    if seq_lens is not None:
        _need_cuda(seq_lens, "seq_lens", torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    ws = workspace or _default_workspace(q.device)
    buf = ws.get(workspace_bytes(B, Hq, Hkv, D, n_splits), q.device)
    st = _lib().fd_append_decode(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), ctypes.byref(kv), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, B, Hq, Hkv,
                                 seq_lens.data_ptr() if seq_lens is not None else None, int(max_seq_len), D,
                                 float(scale), int(n_splits), buf.data_ptr(), buf.numel(),
                                 _stream_handle(q.device, stream))
    _check(st, "fd_append_decode")
    return out, lse


def _rows_args(q, k, v, block_table, seq_lens, max_seq_len, scale, out, lse, return_lse):
    torch = _torch()
    _need_cuda(q, "q", torch.float32)
    if q.dim() != 4:
        raise ValueError("q must be [B, Hq, n_q, D]")
    kv = _kv_desc(k, v, block_table)
    B, Hq, n_q, D = q.shape
    if max_seq_len is None:
        max_seq_len = k.shape[2] if block_table is None else block_table.shape[1] * k.shape[2]
    if seq_lens is not None:
        _need_cuda(seq_lens, "seq_lens", torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, n_q, D), dtype=torch.float32, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, n_q), dtype=torch.float32, device=q.device)
    return kv, B, Hq, n_q, D, max_seq_len, scale, out, lse


def prefill(q, k, v, *, causal=True, seq_lens=None, max_seq_len=None, block_table=None, scale=None, out=None,
            lse=None, return_lse=True, workspace: Optional[Workspace] = None, stream=None):
    """``fd_prefill``: the ``decode_rows`` operation for long windows, on tcgen05 query tiles."""
    kv, B, Hq, n_q, D, max_seq_len, scale, out, lse = _rows_args(q, k, v, block_table, seq_lens, max_seq_len,
                                                                scale, out, lse, return_lse)
    ws = workspace or _default_workspace(q.device)
    buf = ws.get(256, q.device)
    st = _lib().fd_prefill(q.data_ptr(), int(n_q), int(bool(causal)), ctypes.byref(kv), out.data_ptr(),
                           lse.data_ptr() if lse is not None else None, B, Hq, k.shape[1],
                           seq_lens.data_ptr() if seq_lens is not None else None, int(max_seq_len), D, float(scale),
                           buf.data_ptr(), buf.numel(), _stream_handle(q.device, stream))
    _check(st, "fd_prefill")
    return out, lse


def attend_backend(n_q, Hq, Hkv, D, kv_dtype="bf16") -> str:
    """Name of the backend ``attend`` would run (``fd_attend_backend``)."""
    dt = {"bf16": FD_BF16, "f32": FD_F32}[kv_dtype]
    return _lib().fd_backend_name(_lib().fd_attend_backend(int(n_q), int(Hq), int(Hkv), int(D), dt)).decode()


def attend(q, k, v, *, causal=True, seq_lens=None, max_seq_len=None, block_table=None, scale=None,
           n_splits=FD_SPLITS_AUTO, out=None, lse=None, return_lse=True, workspace: Optional[Workspace] = None,
           stream=None):
    """``fd_attend``: phase dispatch for q ``[B, Hq, n_q, D]``; returns ``(out, lse, backend name)``."""
    kv, B, Hq, n_q, D, max_seq_len, scale, out, lse = _rows_args(q, k, v, block_table, seq_lens, max_seq_len,
                                                                scale, out, lse, return_lse)
    Hkv = k.shape[1]
    lib = _lib()
    be = lib.fd_attend_backend(int(n_q), Hq, Hkv, D, kv.dtype)
    need = 256 if be == 2 else workspace_bytes(B, Hq * n_q, Hkv, D, n_splits)
    ws = workspace or _default_workspace(q.device)
    buf = ws.get(need, q.device)
    chosen = ctypes.c_int32(-1)
    st = lib.fd_attend(q.data_ptr(), int(n_q), int(bool(causal)), ctypes.byref(kv), out.data_ptr(),
                       lse.data_ptr() if lse is not None else None, B, Hq, Hkv,
                       seq_lens.data_ptr() if seq_lens is not None else None, int(max_seq_len), D, float(scale),
                       int(n_splits), buf.data_ptr(), buf.numel(), _stream_handle(q.device, stream),
                       ctypes.byref(chosen))
    _check(st, "fd_attend")
    return out, lse, lib.fd_backend_name(chosen.value).decode()


def decode_static(q, k, v, *, out, lse=None, seq_lens=None, max_seq_len=None, block_table=None, scale=None,
                  n_splits=FD_SPLITS_AUTO, stream=None):
    """``fd_decode_static``: fd_decode for callers that may not allocate device memory.

    The caller passes every buffer (``out`` is required; ``lse`` optional); the
    library's scratch is a fixed device array inside libfdecode, shared by all
    calls, so calls must not overlap on the GPU.  Nothing is allocated here.
    """
    torch = _torch()
    _need_cuda(q, "q", torch.float32)
    _need_cuda(out, "out", torch.float32)
    kv = _kv_desc(k, v, block_table)
    B, Hq, Hkv, D, max_seq_len = _geometry(q, k, block_table, seq_lens, max_seq_len)
    if seq_lens is not None:
        _need_cuda(seq_lens, "seq_lens", torch.int32)
    if lse is not None:
        _need_cuda(lse, "lse", torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = _lib().fd_decode_static(q.data_ptr(), ctypes.byref(kv), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, B, Hq, Hkv,
                                 seq_lens.data_ptr() if seq_lens is not None else None, max_seq_len, D,
                                 float(scale), int(n_splits), _stream_handle(q.device, stream))
    _check(st, "fd_decode_static")
    return out, lse


def static_status(device=None, stream=None) -> int:
    """``fd_static_status``: synchronise and return (then clear) the error word of the
    static scratch array that ``decode_static`` uses (0 = no error)."""
    torch = _torch()
    device = device or torch.device("cuda", torch.cuda.current_device())
    return int(_lib().fd_static_status(_stream_handle(device, stream)))


def decode_host(q_host, k, v, *, seq_lens_host=None, max_seq_len=None, block_table=None, scale=None,
                n_splits=FD_SPLITS_AUTO, out_host=None, lse_host=None, workspace: Optional[Workspace] = None,
                stream=None):
    """``fd_decode_host``: q, seq_lens and the outputs in (pinned) host memory; synchronous."""
    torch = _torch()
    if q_host.is_cuda or q_host.dtype != torch.float32 or not q_host.is_contiguous():
        raise ValueError("q_host must be a contiguous fp32 CPU tensor")
    kv = _kv_desc(k, v, block_table)
    B, Hq, Hkv, D, max_seq_len = _geometry(q_host, k, block_table, seq_lens_host, max_seq_len)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out_host is None:
        out_host = torch.empty((B, Hq, D), dtype=torch.float32, pin_memory=True)
    if lse_host is None:
        lse_host = torch.empty((B, Hq), dtype=torch.float32, pin_memory=True)
    if seq_lens_host is not None and (seq_lens_host.is_cuda or seq_lens_host.dtype != torch.int32):
        raise ValueError("seq_lens_host must be an int32 CPU tensor")
    ws = workspace or _default_workspace(k.device)
    nbytes = workspace_bytes(B, Hq, Hkv, D, n_splits)
    buf = ws.get(nbytes, k.device)
    st = _lib().fd_decode_host(q_host.data_ptr(), ctypes.byref(kv), out_host.data_ptr(), lse_host.data_ptr(),
                               B, Hq, Hkv, seq_lens_host.data_ptr() if seq_lens_host is not None else None,
                               max_seq_len, D, float(scale), int(n_splits), buf.data_ptr(), buf.numel(),
                               _stream_handle(k.device, stream))
    _check(st, "fd_decode_host")
    return out_host, lse_host


class HostDecoder:
    """``fd_decode_host`` with its arguments marshalled once, for a decode loop
    that passes the same host buffers and KV cache every step.

    ``q_host`` ``[B, Hq, D]`` fp32, ``out_host`` ``[B, Hq, D]`` and ``lse_host``
    ``[B, Hq]`` (optional), ``seq_lens_host`` ``[B]`` int32 (optional) are CPU
    tensors whose contents the caller rewrites between steps; pinned buffers
    (``pin_memory=True``) are read and written by the kernels in place, over the
    host link, and pageable ones are copied through the workspace.  Calling the
    object runs one synchronous step and returns ``(out_host, lse_host)``.
    """

    def __init__(self, q_host, k, v, *, out_host=None, lse_host=None, seq_lens_host=None, max_seq_len=None,
                 block_table=None, scale=None, n_splits=FD_SPLITS_AUTO, workspace: Optional[Workspace] = None,
                 stream=None):
        torch = _torch()
        if q_host.is_cuda or q_host.dtype != torch.float32 or not q_host.is_contiguous():
            raise ValueError("q_host must be a contiguous fp32 CPU tensor")
        self._kv = _kv_desc(k, v, block_table)
        B, Hq, Hkv, D, max_seq_len = _geometry(q_host, k, block_table, seq_lens_host, max_seq_len)
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        if out_host is None:
            out_host = torch.empty((B, Hq, D), dtype=torch.float32, pin_memory=True)
        for t, name, shape, dt in ((out_host, "out_host", (B, Hq, D), torch.float32),
                                   (lse_host, "lse_host", (B, Hq), torch.float32),
                                   (seq_lens_host, "seq_lens_host", (B,), torch.int32)):
            if t is not None and (t.is_cuda or t.dtype != dt or not t.is_contiguous() or tuple(t.shape) != shape):
                raise ValueError(f"{name} must be a contiguous {dt} CPU tensor of shape {shape}")
        ws = workspace or _default_workspace(k.device)
        buf = ws.get(workspace_bytes(B, Hq, Hkv, D, n_splits), k.device)
        self.q_host, self.out_host, self.lse_host, self.seq_lens_host = q_host, out_host, lse_host, seq_lens_host
        self._keep = (k, v, block_table, buf)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        self._fn = _lib().fd_decode_host
        self._args = (vp(q_host.data_ptr()), ctypes.byref(self._kv), vp(out_host.data_ptr()),
                      vp(lse_host.data_ptr() if lse_host is not None else None), i32(B), i32(Hq), i32(Hkv),
                      vp(seq_lens_host.data_ptr() if seq_lens_host is not None else None), i32(max_seq_len), i32(D),
                      ctypes.c_float(scale), i32(int(n_splits)), vp(buf.data_ptr()), ctypes.c_size_t(buf.numel()),
                      vp(_stream_handle(k.device, stream)))

    def __call__(self):
        st = self._fn(*self._args)
        if st != FD_OK:
            raise FdError(st, "fd_decode_host")
        return self.out_host, self.lse_host


def split_partial(q, k, v, n_splits: int, *, seq_lens=None, max_seq_len=None, block_table=None, scale=None,
                  stream=None):
    """``fd_split_partial``: returns ``(o_part [B,Hq,n,D], m_part [B,Hq,n], l_part [B,Hq,n])``."""
    torch = _torch()
    _need_cuda(q, "q", torch.float32)
    kv = _kv_desc(k, v, block_table)
    B, Hq, Hkv, D, max_seq_len = _geometry(q, k, block_table, seq_lens, max_seq_len)
    if seq_lens is not None:
        _need_cuda(seq_lens, "seq_lens", torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty((B, Hq, n_splits, D), dtype=torch.float32, device=q.device)
    m = torch.empty((B, Hq, n_splits), dtype=torch.float32, device=q.device)
    l = torch.empty((B, Hq, n_splits), dtype=torch.float32, device=q.device)
    st = _lib().fd_split_partial(q.data_ptr(), ctypes.byref(kv), B, Hq, Hkv,
                                 seq_lens.data_ptr() if seq_lens is not None else None, max_seq_len, D, float(scale),
                                 int(n_splits), o.data_ptr(), m.data_ptr(), l.data_ptr(),
                                 _stream_handle(q.device, stream))
    _check(st, "fd_split_partial")
    return o, m, l


def combine(o_part, m_part, l_part, *, out=None, lse=None, return_lse=True, stream=None):
    """``fd_combine`` over partials in the ``fd_split_partial`` layout."""
    torch = _torch()
    for t, n in ((o_part, "o_part"), (m_part, "m_part"), (l_part, "l_part")):
        _need_cuda(t, n, torch.float32)
    B, Hq, n_splits, D = o_part.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=o_part.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=o_part.device)
    st = _lib().fd_combine(o_part.data_ptr(), m_part.data_ptr(), l_part.data_ptr(), out.data_ptr(),
                           lse.data_ptr() if lse is not None else None, B, Hq, D, n_splits,
                           _stream_handle(o_part.device, stream))
    _check(st, "fd_combine")
    return out, lse


def workspace_status(workspace: Optional[Workspace] = None, device=None, stream=None) -> int:
    """Synchronise and return (then clear) the kernels' error word of a workspace (0 = no error)."""
    torch = _torch()
    device = device or torch.device("cuda", torch.cuda.current_device())
    ws = workspace or _default_workspace(device)
    if ws.buf is None:
        return FD_OK
    return int(_lib().fd_workspace_status(ws.buf.data_ptr(), ws.buf.numel(), _stream_handle(ws.buf.device, stream)))
