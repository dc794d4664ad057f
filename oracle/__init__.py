"""The oracle: a plain fp64 CPU statement of relative-position attention.

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` are the only callers. The CUDA
library (``vision_transformer_attention_gb300``) never imports this package
and shares no code with it; inputs reach both sides from the seeded
generators in ``vision_transformer_attention_gb300.workloads``, which hold
none of the method's arithmetic.

The arithmetic lives in ``rpe_oracle.c`` (plain C, double precision, every
pair computed explicitly). This module only compiles it with gcc and
marshals numpy arrays through ctypes. Sources are cited in the C file:
"Rethinking and Improving Relative Position Encoding for Vision Transformer"
(eqs. 13-18, 25-28), "Swin 的二维 RPE" (sections 3.1-3.3), "Swin Transformer,
section 3.2 and Table 4", and "Implementation: Relative Position in
Self-Attention".

Every function is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import concurrent.futures
import ctypes
import os
import subprocess

import numpy as np

FLAG_K = 1
FLAG_Q = 2
FLAG_V = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rpe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile rpe_oracle.c into _build/liboracle.so with gcc (no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32, dbl, u32 = ctypes.c_int, ctypes.c_double, ctypes.c_uint
        p = ctypes.c_void_p
        lib.orc_piecewise_index.restype = i32
        lib.orc_piecewise_index.argtypes = [dbl, dbl, dbl, dbl]
        lib.orc_product_bucket_ids.restype = i32
        lib.orc_product_bucket_ids.argtypes = [i32, i32, dbl, dbl, dbl, p]
        lib.orc_swin_bias_index.restype = i32
        lib.orc_swin_bias_index.argtypes = [i32, p]
        lib.orc_clip_ids_1d.restype = None
        lib.orc_clip_ids_1d.argtypes = [i32, i32, p]
        lib.orc_attention.restype = i32
        lib.orc_attention.argtypes = [i32, i32, p, p, p, p, p, i32, p, p, p, p, p, dbl,
                                      i32, p, p, p]
        lib.orc_cross_bucket_ids.restype = i32
        lib.orc_cross_bucket_ids.argtypes = [i32, i32, dbl, dbl, dbl, p, p]
        lib.orc_add_cls_bucket.restype = i32
        lib.orc_add_cls_bucket.argtypes = [i32, p, i32, p]
        lib.orc_clip_product_bucket_ids.restype = i32
        lib.orc_clip_product_bucket_ids.argtypes = [i32, i32, i32, p]
        lib.orc_euclidean_bucket_ids.restype = i32
        lib.orc_euclidean_bucket_ids.argtypes = [i32, i32, dbl, dbl, dbl, p]
        lib.orc_irpe_attention_ids.restype = i32
        lib.orc_irpe_attention_ids.argtypes = [i32, i32, i32, i32, p, p, i32, u32, p, p, p,
                                               p, p, p, i32, p, i32, i32, p, i32, p, p]
        lib.orc_attention_efficient.restype = i32
        lib.orc_attention_efficient.argtypes = [i32, i32, p, p, p, p, i32, p, p, p,
                                                p, dbl, p]
        lib.orc_irpe_attention.restype = i32
        lib.orc_irpe_attention.argtypes = [i32, i32, i32, i32, i32, dbl, dbl, dbl, u32,
                                           p, p, p, p, p, p, i32, p, i32, p, p]
        lib.orc_swin_attention.restype = i32
        lib.orc_swin_attention.argtypes = [i32, i32, i32, i32, p, p, p, p, i32, p, p]
        _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # a torch tensor: exact upcast of its values
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _out_like(q, out):
    if out is None:
        return np.zeros_like(q)
    assert out.dtype == np.float64 and out.shape == q.shape and out.flags.c_contiguous
    return out


def parallel_slices(run, slices, threads=None):
    """Calls run(part) on disjoint parts of the slice list from `threads`
    threads (default: every host core). The C calls release the GIL, so the
    parts run in parallel; each call writes only its own slices of a shared
    output. Returns the number of threads used."""
    _load()  # once, before any thread calls in
    slices = np.asarray(slices, dtype=np.int32)
    threads = max(1, min(threads or os.cpu_count() or 1, len(slices)))
    parts = [p for p in np.array_split(slices, threads) if len(p)]
    if len(parts) == 1:
        run(parts[0])
        return 1
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        for f in [ex.submit(run, p) for p in parts]:
            f.result()
    return len(parts)


def _check(status):
    if status != 0:
        raise ValueError(f"oracle call failed with status {status}")


def piecewise_index(x: float, alpha: float, beta: float, gamma: float) -> int:
    """Eq. 18 of the iRPE page, one axis offset."""
    return int(_load().orc_piecewise_index(float(x), alpha, beta, gamma))


def product_bucket_ids(H: int, W: int, alpha: float, beta: float, gamma: float):
    """Eq. 25 Product ids, shape [N, N] int32 (query-major); returns (ids, K)."""
    N = H * W
    ids = np.zeros((N, N), dtype=np.int32)
    K = _load().orc_product_bucket_ids(H, W, alpha, beta, gamma, _ptr(ids))
    return ids, int(K)


def euclidean_bucket_ids(H: int, W: int, alpha: float, beta: float, gamma: float):
    """Euclidean-mapping ids (section 3.2, distance rounded first), shape [N, N]
    int32 (query-major); returns (ids, K) with K = 2*int(beta)+1."""
    N = H * W
    ids = np.zeros((N, N), dtype=np.int32)
    K = _load().orc_euclidean_bucket_ids(H, W, alpha, beta, gamma, _ptr(ids))
    return ids, int(K)


def cross_bucket_ids(H: int, W: int, alpha: float, beta: float, gamma: float):
    """Cross-mapping ids (section 3.2, eqs. 22-24): (ids_row, ids_col, K), both
    [N, N] int32, row buckets in [0, span), column buckets in [span, 2 span),
    K = 2 span, span = 2*int(beta)+1."""
    N = H * W
    ids_row = np.zeros((N, N), dtype=np.int32)
    ids_col = np.zeros((N, N), dtype=np.int32)
    K = _load().orc_cross_bucket_ids(H, W, alpha, beta, gamma, _ptr(ids_row), _ptr(ids_col))
    return ids_row, ids_col, int(K)


def add_cls_bucket(ids, K: int):
    """Section 4.1's class-token bucket: the [N, N] patch id map becomes the
    [N+1, N+1] map of token 0 (class) and the patches; returns (ids, K + 1)."""
    ids = _i32(ids)
    N = ids.shape[0]
    out = np.zeros((N + 1, N + 1), dtype=np.int32)
    K1 = _load().orc_add_cls_bucket(N, _ptr(ids), K, _ptr(out))
    return out, int(K1)


def clip_product_bucket_ids(H: int, W: int, k: int):
    """Product ids of the per-axis clipped offsets (table 3's clip index): (ids, (2k+1)^2)."""
    N = H * W
    ids = np.zeros((N, N), dtype=np.int32)
    K = _load().orc_clip_product_bucket_ids(H, W, k, _ptr(ids))
    return ids, int(K)


def irpe_attention_ids(q, k, v, ids, num_buckets, flags=0, tab_q=None, tab_k=None,
                       tab_v=None, bias_in=None, slices=None, rows=None, ids2=None, out=None):
    """iRPE attention on [B, heads, N, d] with a given [N, N] id map; bias_in is a
    bias-mode table [num_buckets, bias_heads] (bias_heads 1 = shared by all heads);
    ids2, a second [N, N] map whose entries are added (the Cross mapping).
    Contextual tables are [num_buckets, d] (shared by every head) or
    [heads, num_buckets, d] (one per head). ``out`` (float64, q's shape) receives
    the picked slices and is returned; by default a zeroed array."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, heads, N, d = q.shape
    ids = _i32(ids)
    assert ids.shape == (N, N)
    ids2 = _i32(ids2)
    assert ids2 is None or ids2.shape == (N, N)
    tab_q, tab_k, tab_v = _f64(tab_q), _f64(tab_k), _f64(tab_v)
    tabs = [t for t in (tab_q, tab_k, tab_v) if t is not None]
    tab_heads = tabs[0].shape[0] if tabs and tabs[0].ndim == 3 else 1
    for t in tabs:
        assert t.shape[-2:] == (num_buckets, d) and (t.ndim == 2 or t.shape[0] == heads)
        assert t.ndim == tabs[0].ndim  # all shared or all per head
    bias_in = _f64(bias_in)
    bias_heads = 0 if bias_in is None else (1 if bias_in.ndim == 1 else bias_in.shape[1])
    slices, rows = _i32(slices), _i32(rows)
    out = _out_like(q, out)
    _check(_load().orc_irpe_attention_ids(
        B, heads, N, d, _ptr(ids), _ptr(ids2), num_buckets, flags, _ptr(q), _ptr(k), _ptr(v),
        _ptr(tab_q), _ptr(tab_k), _ptr(tab_v), tab_heads, _ptr(bias_in), bias_heads,
        0 if slices is None else len(slices), _ptr(slices),
        0 if rows is None else len(rows), _ptr(rows), _ptr(out)))
    return out


def swin_bias_index(M: int):
    """Flattened Swin table index of every pair in an M x M window; (idx, (2M-1)^2)."""
    n = M * M
    idx = np.zeros((n, n), dtype=np.int32)
    nb = _load().orc_swin_bias_index(M, _ptr(idx))
    return idx, int(nb)


def clip_ids_1d(n: int, k: int):
    """Shaw clip-and-shift ids clip(j - i, -k, k) + k, shape [n, n]."""
    ids = np.zeros((n, n), dtype=np.int32)
    _load().orc_clip_ids_1d(n, k, _ptr(ids))
    return ids


def attention(q, k, v, ids, num_buckets, tab_k=None, tab_q=None, tab_v=None,
              bias=None, scale=None, rows=None, want_attn=False, bias_in=None, ids2=None):
    """One slice, every pair explicit. q, k, v: [n, d]. Returns out (and attn).
    bias: Swin scalar per bucket after the scaling; bias_in: iRPE bias-mode
    scalar per bucket inside it; ids2: a second id map added to ids (Cross)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = q.shape
    ids = _i32(ids)
    ids2 = _i32(ids2)
    tab_k, tab_q, tab_v, bias = _f64(tab_k), _f64(tab_q), _f64(tab_v), _f64(bias)
    bias_in = _f64(bias_in)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = _i32(rows)
    out = np.zeros((n, d))
    attn = np.zeros((n, n)) if want_attn else None
    _check(_load().orc_attention(n, d, _ptr(q), _ptr(k), _ptr(v), _ptr(ids), _ptr(ids2),
                                 num_buckets,
                                 _ptr(tab_k), _ptr(tab_q), _ptr(tab_v), _ptr(bias),
                                 _ptr(bias_in), scale,
                                 0 if rows is None else len(rows), _ptr(rows),
                                 _ptr(out), _ptr(attn)))
    return (out, attn) if want_attn else out


def attention_efficient(q, k, v, ids, num_buckets, tab_k=None, tab_q=None, tab_v=None,
                        bias=None, scale=None):
    """One slice by the eqs. 26-28 route (QR / KR gathers, per-bucket sums)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = q.shape
    ids = _i32(ids)
    tab_k, tab_q, tab_v, bias = _f64(tab_k), _f64(tab_q), _f64(tab_v), _f64(bias)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.zeros((n, d))
    _check(_load().orc_attention_efficient(n, d, _ptr(q), _ptr(k), _ptr(v), _ptr(ids),
                                           num_buckets, _ptr(tab_k), _ptr(tab_q),
                                           _ptr(tab_v), _ptr(bias), scale, _ptr(out)))
    return out


def irpe_attention(q, k, v, H, W, alpha, beta, gamma, flags,
                   tab_q=None, tab_k=None, tab_v=None, slices=None, rows=None):
    """iRPE contextual Product attention on [B, heads, N, d] tensors.

    ``slices`` picks flattened (b*heads + h) slices and ``rows`` query rows;
    the result has the input's shape with only the picked entries written
    (the rest stay zero)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, heads, N, d = q.shape
    assert N == H * W
    tab_q, tab_k, tab_v = _f64(tab_q), _f64(tab_k), _f64(tab_v)
    slices, rows = _i32(slices), _i32(rows)
    out = np.zeros_like(q)
    _check(_load().orc_irpe_attention(
        B, heads, H, W, d, alpha, beta, gamma, flags, _ptr(q), _ptr(k), _ptr(v),
        _ptr(tab_q), _ptr(tab_k), _ptr(tab_v),
        0 if slices is None else len(slices), _ptr(slices),
        0 if rows is None else len(rows), _ptr(rows), _ptr(out)))
    return out


def swin_attention(q, k, v, table, M, slices=None, out=None):
    """Swin window attention on [num_windows, heads, M*M, d] with a
    [(2M-1)^2, heads] bias table (``out`` as for irpe_attention_ids)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    nw, heads, n, d = q.shape
    assert n == M * M
    table = _f64(table)
    assert table.shape == ((2 * M - 1) ** 2, heads)
    slices = _i32(slices)
    out = _out_like(q, out)
    _check(_load().orc_swin_attention(nw, heads, M, d, _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(table), 0 if slices is None else len(slices),
                                      _ptr(slices), _ptr(out)))
    return out
