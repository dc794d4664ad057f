"""Thin Python binding of the C ABI (include/rpe_attn.h), one function per
entry point and with the same names. It only marshals torch CUDA tensors
into pointers and sizes: every step of the computation runs in the
library's CUDA kernels, on the tensors' device and the current stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import check

_DTYPES = {torch.bfloat16: _lib.RPE_DTYPE_BF16, torch.float32: _lib.RPE_DTYPE_F32}


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype=None, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


def rpe_build_bucket_ids(H, W, alpha, beta, gamma, device="cuda", with_ids=False,
                         mode=_lib.RPE_MAP_PRODUCT):
    """iRPE eq. 18 with a mapping of section 3.2 on the GPU. Returns (bucket_lut, ids or
    None, num_buckets): bucket_lut int32 [(2H-1)*(2W-1)] indexed by offset, ids int32
    [N, N] ([2, N, N] for the Cross mapping: row buckets, then column buckets)."""
    device = torch.device(device)
    lut = torch.empty((2 * H - 1) * (2 * W - 1), dtype=torch.int32, device=device)
    shape = (2, H * W, H * W) if mode == _lib.RPE_MAP_CROSS else (H * W, H * W)
    ids = torch.empty(shape, dtype=torch.int32, device=device) if with_ids else None
    nb = ctypes.c_int(0)
    with torch.cuda.device(device):
        check("rpe_build_bucket_ids", _lib.lib().rpe_build_bucket_ids(
            H, W, mode, float(alpha), float(beta), float(gamma), _ptr(lut), _ptr(ids),
            ctypes.byref(nb), _stream(lut)))
    return lut, ids, nb.value


def rpe_attn_fwd(q, k, v, bucket_lut, num_buckets, H, W, terms, table_q=None, table_k=None,
                 table_v=None, out=None, cls_token=False):
    """iRPE contextual attention (eqs. 13, 15-17) on q, k, v [B, heads, H*W, d]; terms
    may carry RPE_TABLES_CROSS for tables of the Cross mapping (eqs. 22-24). Tables
    are [num_buckets, d] (shared by every head) or [heads, num_buckets, d] (one per
    head; RPE_TABLES_PER_HEAD is then set here). cls_token: token 0 is a class token
    (section 4.1; q, k, v hold H*W + 1 tokens, its pairs use bucket num_buckets - 1)."""
    _need(q, "q")
    B, heads, N, d = q.shape
    if cls_token:
        terms |= _lib.RPE_CLS_TOKEN
    if N != H * W + (1 if terms & _lib.RPE_CLS_TOKEN else 0):
        raise ValueError(f"q has {N} tokens; the {H}x{W} grid needs H*W (+1 with a class token)")
    if q.dtype not in _DTYPES:
        raise TypeError("q must be bfloat16 or float32")
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, q.shape, q.device)
    _need(bucket_lut, "bucket_lut", torch.int32, ((2 * H - 1) * (2 * W - 1),), q.device)
    tabs = {"table_q": (table_q, _lib.RPE_TERM_Q), "table_k": (table_k, _lib.RPE_TERM_K),
            "table_v": (table_v, _lib.RPE_TERM_V)}
    used = [t for t, bit in tabs.values() if terms & bit]
    per_head = bool(used) and used[0].dim() == 3
    for name, (t, bit) in tabs.items():
        if terms & bit:
            _need(t, name, q.dtype, (heads, num_buckets, d) if per_head else (num_buckets, d),
                  q.device)
    if per_head:
        terms |= _lib.RPE_TABLES_PER_HEAD
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", q.dtype, q.shape, q.device)
    use = lambda t, bit: _ptr(t) if terms & bit else None  # noqa: E731
    with torch.cuda.device(q.device):
        check("rpe_attn_fwd", _lib.lib().rpe_attn_fwd(
            _ptr(q), _ptr(k), _ptr(v), use(table_q, _lib.RPE_TERM_Q),
            use(table_k, _lib.RPE_TERM_K), use(table_v, _lib.RPE_TERM_V), _ptr(bucket_lut),
            num_buckets, B, heads, H, W, d, terms, _DTYPES[q.dtype], _ptr(out), _stream(q)))
    return out


def rpe_attn_bias_fwd(q, k, v, bias_table, bucket_lut, num_buckets, H, W, out=None, cross=False,
                      cls_token=False):
    """iRPE bias mode (eqs. 13-14) on q, k, v [B, heads, H*W, d]: bias_table is fp32
    [num_buckets, heads] (per head) or [num_buckets] / [num_buckets, 1] (shared);
    cross: the table is laid out for the Cross mapping (eqs. 22-24); cls_token:
    token 0 is a class token (section 4.1, H*W + 1 tokens)."""
    _need(q, "q")
    B, heads, N, d = q.shape
    if N != H * W + (1 if cls_token else 0):
        raise ValueError(f"q has {N} tokens; the {H}x{W} grid needs H*W (+1 with a class token)")
    if q.dtype not in _DTYPES:
        raise TypeError("q must be bfloat16 or float32")
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, q.shape, q.device)
    if bias_table.dim() == 1:
        bias_table = bias_table.reshape(-1, 1)
    bias_heads = bias_table.shape[1]
    _need(bias_table, "bias_table", torch.float32, (num_buckets, bias_heads), q.device)
    _need(bucket_lut, "bucket_lut", torch.int32, None, q.device)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", q.dtype, q.shape, q.device)
    with torch.cuda.device(q.device):
        check("rpe_attn_bias_fwd", _lib.lib().rpe_attn_bias_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table), bias_heads, _ptr(bucket_lut),
            num_buckets, (_lib.RPE_TABLES_CROSS if cross else 0) | (_lib.RPE_CLS_TOKEN if cls_token else 0),
            B, heads, H, W, d,
            _DTYPES[q.dtype], _ptr(out), _stream(q)))
    return out


def swin_window_attn_fwd(q, k, v, bias_table, M, out=None):
    """Swin window attention SoftMax(QK^T/sqrt(d) + B)V on [windows, heads, M*M, d]."""
    _need(q, "q")
    nw, heads, n, d = q.shape
    if q.dtype not in _DTYPES:
        raise TypeError("q must be bfloat16 or float32")
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, q.shape, q.device)
    _need(bias_table, "bias_table", torch.float32, ((2 * M - 1) ** 2, heads), q.device)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", q.dtype, q.shape, q.device)
    with torch.cuda.device(q.device):
        check("swin_window_attn_fwd", _lib.lib().swin_window_attn_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table), nw, heads, M, d, _DTYPES[q.dtype],
            _ptr(out), _stream(q)))
    return out


def swin_window_attn_fwd_fmap(q, k, v, bias_table, M, out=None):
    """Swin window attention on channels-last bf16 feature maps q, k, v
    [batch, img_h, img_w, heads * d]: every M x M window of every head is
    attended as swin_window_attn_fwd does, with the window partition and its
    reverse done by the kernel's loads and stores."""
    _need(q, "q")
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bfloat16")
    if q.dim() != 4:
        raise ValueError("q must be [batch, img_h, img_w, heads * d]")
    batch, img_h, img_w, channels = q.shape
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, q.shape, q.device)
    if bias_table.dim() != 2 or bias_table.shape[0] != (2 * M - 1) ** 2:
        raise ValueError("bias_table must be [(2M-1)^2, heads]")
    heads = bias_table.shape[1]
    _need(bias_table, "bias_table", torch.float32, ((2 * M - 1) ** 2, heads), q.device)
    if channels % heads:
        raise ValueError("channels must be heads * d")
    d = channels // heads
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", q.dtype, q.shape, q.device)
    with torch.cuda.device(q.device):
        check("swin_window_attn_fwd_fmap", _lib.lib().swin_window_attn_fwd_fmap(
            _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table), batch, img_h, img_w, heads, M, d,
            _ptr(out), _stream(q)))
    return out


def rpe_device_status(clear=True):
    """Synchronises the device; returns the device status word (0 = none; bits
    0-4 a bounded wait ran out, bit 5 an offset table held an id out of range)."""
    st = ctypes.c_uint(0)
    rc = _lib.lib().rpe_device_status(ctypes.byref(st), int(bool(clear)))
    if rc not in (_lib.RPE_OK, _lib.RPE_ERR_TIMEOUT, _lib.RPE_ERR_INVALID_ARG) or (
            rc == _lib.RPE_ERR_INVALID_ARG and st.value == 0):
        check("rpe_device_status", rc)
    return st.value


def rpe_release_stream(stream=None):
    """Frees the split-tail workspace the library keeps for `stream` (default:
    the current stream) on the current device, if there is one."""
    s = stream if stream is not None else torch.cuda.current_stream()
    check("rpe_release_stream", _lib.lib().rpe_release_stream(ctypes.c_void_p(s.cuda_stream)))


def rpe_shutdown():
    """Frees every device allocation of the library and forgets the offset
    tables it recorded as checked; the next call allocates again."""
    check("rpe_shutdown", _lib.lib().rpe_shutdown())


def swin_window_attn_fwd_noalloc(q, k, v, bias_table, M, out=None):
    """swin_window_attn_fwd (bf16) through the entry point that allocates no
    device memory: its status word is a word of a fixed array in the library."""
    _need(q, "q", torch.bfloat16)
    nw, heads, n, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _need(t, name, q.dtype, q.shape, q.device)
    _need(bias_table, "bias_table", torch.float32, ((2 * M - 1) ** 2, heads), q.device)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", q.dtype, q.shape, q.device)
    with torch.cuda.device(q.device):
        check("swin_window_attn_fwd_noalloc", _lib.lib().swin_window_attn_fwd_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table), nw, heads, M, d, _ptr(out), _stream(q)))
    return out


def swin_noalloc_status(clear=True):
    """Synchronises the device; returns the no-allocation entry point's status word."""
    st = ctypes.c_uint(0)
    rc = _lib.lib().swin_noalloc_status(ctypes.byref(st), int(bool(clear)))
    if rc not in (_lib.RPE_OK, _lib.RPE_ERR_TIMEOUT):
        check("swin_noalloc_status", rc)
    return st.value


def swin_noalloc_status_word():
    """Device address (int) of the no-allocation entry point's status word."""
    w = ctypes.c_void_p(0)
    check("swin_noalloc_status_word", _lib.lib().swin_noalloc_status_word(ctypes.byref(w)))
    return w.value


def rpe_wait_probe(limit_ns=1_000_000):
    """Runs the bounded wait on a barrier nothing arrives at (a timeout self-test)."""
    check("rpe_wait_probe", _lib.lib().rpe_wait_probe(
        int(limit_ns), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
