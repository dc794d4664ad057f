"""Seeded synthetic workloads: shapes and input generators, nothing else.

This module holds none of the attention arithmetic. It is the one module that
both the CUDA path and the oracle receive inputs from, so that a parity test
compares the two on identical values.

Shapes follow the pages' workloads: DeiT-S uses a 14 x 14 token grid with 6
heads of 64 channels ("Rethinking and Improving Relative Position Encoding for
Vision Transformer", Problem; section 4.1), and Swin attends inside 7 x 7
windows ("Swin Transformer, section 3.2 and Table 4", Conditions). Swin-T
stage 1 has 3 heads of 32 channels on a 56 x 56 map. No dataset is used:
q, k, v ~ N(0, 1) and every relative-position table ~ N(0, 0.02^2), drawn in
fp32 from a CPU ``torch.Generator`` and then cast to the working dtype.
Seeds: q 0, k 1, v 2, table t (Q, K, V, or the Swin bias) 3 + t, each offset
by ``seed``.
"""
from __future__ import annotations

import dataclasses

import torch

FLAG_K = 1
FLAG_Q = 2
FLAG_V = 4

# The iRPE index-function constants scale with a ratio r as alpha = r,
# beta = 2r, gamma = 8r; the DeiT Product configuration uses r = 1.9
# (iRPE page, Paper-vs-code list, "Product and the ratio").
IRPE_RATIO = 1.9


def index_constants(ratio: float = IRPE_RATIO):
    return float(ratio), 2.0 * ratio, 8.0 * ratio


@dataclasses.dataclass(frozen=True)
class SwinConfig:
    name: str
    num_windows: int
    heads: int
    M: int
    d: int
    dtype: str  # "bf16" or "f32"
    # (batch, img_h, img_w) when q/k/v/out are channels-last feature maps that
    # the kernel partitions itself; () for pre-partitioned windows
    fmap: tuple = ()

    @property
    def n(self) -> int:
        return self.M * self.M

    @property
    def tokens(self) -> int:
        return self.num_windows * self.n


@dataclasses.dataclass(frozen=True)
class IrpeConfig:
    name: str
    B: int
    heads: int
    H: int
    W: int
    d: int
    flags: int
    dtype: str
    ratio: float = IRPE_RATIO
    cls: bool = False  # a class token at token 0, with its own extra bucket

    @property
    def N(self) -> int:
        return self.H * self.W + (1 if self.cls else 0)

    @property
    def num_buckets(self) -> int:
        span = 2 * int(2.0 * self.ratio) + 1
        return span * span + (1 if self.cls else 0)

    @property
    def tokens(self) -> int:
        return self.B * self.N


CONFIGS = {
    # 4 windows of 7x7, 3 heads, d = 32, fp32 (the small parity case)
    "swin_w7_small_fp32": SwinConfig("swin_w7_small_fp32", 4, 3, 7, 32, "f32"),
    # Swin-T stage 1: 56x56 map = 64 windows, batch 32 -> 2048 windows
    "swin_t_stage1": SwinConfig("swin_t_stage1", 2048, 3, 7, 32, "bf16"),
    # the same, read from and written to the [32, 56, 56, 96] feature maps
    "swin_t_stage1_fmap": SwinConfig("swin_t_stage1_fmap", 2048, 3, 7, 32, "bf16",
                                     fmap=(32, 56, 56)),
    # iRPE-K at the DeiT-S shape, 14x14 grid, no class token
    "irpe_k_deit_s": IrpeConfig("irpe_k_deit_s", 64, 6, 14, 14, 64, FLAG_K, "bf16"),
    # iRPE on queries, keys and values, same shape
    "irpe_qkv_deit_s": IrpeConfig("irpe_qkv_deit_s", 64, 6, 14, 14, 64,
                                  FLAG_Q | FLAG_K | FLAG_V, "bf16"),
    # high-resolution global attention, 56x56 grid
    "irpe_k_56x56": IrpeConfig("irpe_k_56x56", 8, 6, 56, 56, 64, FLAG_K, "bf16"),
    # the r = 2.0 index function (9 x 9 = 81 Product buckets, as DETR's encoder
    # uses it) on the DeiT-S shape
    "irpe_k_r2_deit_s": IrpeConfig("irpe_k_r2_deit_s", 64, 6, 14, 14, 64, FLAG_K, "bf16",
                                   ratio=2.0),
    # DeiT-S with its class token: 197 tokens, 49 + 1 buckets
    "irpe_k_deit_s_cls": IrpeConfig("irpe_k_deit_s_cls", 64, 6, 14, 14, 64, FLAG_K, "bf16",
                                    cls=True),
}

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def _normal(shape, seed, std=1.0):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std


def swin_inputs(num_windows, heads, M, d, dtype="bf16", table_std=0.02, seed=0):
    """q, k, v [num_windows, heads, M*M, d] and the bias table [(2M-1)^2, heads]."""
    dt = _TORCH_DTYPE[dtype]
    n = M * M
    shape = (num_windows, heads, n, d)
    q = _normal(shape, seed + 0).to(dt)
    k = _normal(shape, seed + 1).to(dt)
    v = _normal(shape, seed + 2).to(dt)
    table = _normal(((2 * M - 1) ** 2, heads), seed + 3, table_std)  # fp32
    return {"q": q, "k": k, "v": v, "table": table}


def swin_fmap_inputs(batch, img_h, img_w, heads, M, d, table_std=0.02, seed=0):
    """Channels-last bf16 feature maps q, k, v [batch, img_h, img_w, heads * d]
    and the bias table [(2M-1)^2, heads] fp32 (same draws as swin_inputs)."""
    shape = (batch, img_h, img_w, heads * d)
    q = _normal(shape, seed + 0).to(torch.bfloat16)
    k = _normal(shape, seed + 1).to(torch.bfloat16)
    v = _normal(shape, seed + 2).to(torch.bfloat16)
    table = _normal(((2 * M - 1) ** 2, heads), seed + 3, table_std)
    return {"q": q, "k": k, "v": v, "table": table}


def window_partition(x, M, heads):
    """[batch, img_h, img_w, heads * d] -> [windows, heads, M*M, d]: windows in
    (image, window row, window column) order, token i of a window at (i / M, i % M)."""
    b, h, w, c = x.shape
    d = c // heads
    x = x.reshape(b, h // M, M, w // M, M, heads, d)
    return x.permute(0, 1, 3, 5, 2, 4, 6).reshape(b * (h // M) * (w // M), heads, M * M, d)


def window_reverse(x, M, batch, img_h, img_w):
    """Inverse of window_partition."""
    nw, heads, n, d = x.shape
    x = x.reshape(batch, img_h // M, img_w // M, heads, M, M, d)
    return x.permute(0, 1, 4, 2, 5, 3, 6).reshape(batch, img_h, img_w, heads * d)


def irpe_inputs(B, heads, N, d, num_buckets, flags, dtype="bf16", table_std=0.02, seed=0,
                per_head=False):
    """q, k, v [B, heads, N, d] and tables for the enabled terms (None for a disabled
    one): [num_buckets, d] shared by every head, or [heads, num_buckets, d] per head."""
    dt = _TORCH_DTYPE[dtype]
    shape = (B, heads, N, d)
    out = {
        "q": _normal(shape, seed + 0).to(dt),
        "k": _normal(shape, seed + 1).to(dt),
        "v": _normal(shape, seed + 2).to(dt),
    }
    for t, (name, flag) in enumerate((("tab_q", FLAG_Q), ("tab_k", FLAG_K), ("tab_v", FLAG_V))):
        shape_t = (heads, num_buckets, d) if per_head else (num_buckets, d)
        out[name] = (_normal(shape_t, seed + 3 + t, table_std).to(dt)
                     if flags & flag else None)
    return out


def bias_table(num_buckets, heads, table_std=0.02, seed=6):
    """iRPE bias-mode table [num_buckets, heads] fp32 (heads = 1: shared)."""
    return _normal((num_buckets, heads), seed, table_std)


def config_inputs(cfg, table_std=0.02, seed=0):
    if isinstance(cfg, SwinConfig) and cfg.fmap:
        b, h, w = cfg.fmap
        return swin_fmap_inputs(b, h, w, cfg.heads, cfg.M, cfg.d, table_std, seed)
    if isinstance(cfg, SwinConfig):
        return swin_inputs(cfg.num_windows, cfg.heads, cfg.M, cfg.d, cfg.dtype,
                           table_std, seed)
    return irpe_inputs(cfg.B, cfg.heads, cfg.N, cfg.d, cfg.num_buckets, cfg.flags,
                       cfg.dtype, table_std, seed)
