"""The Euclidean and Cross mappings, the clip index and iRPE bias mode
("Rethinking and Improving Relative Position Encoding for Vision Transformer",
Method, section 3.2, eqs. 13-14 and 22-24, table 3) on the GPU against the
oracle."""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_attention_gb300 import api, workloads
from vision_transformer_attention_gb300._lib import (RPE_MAP_CLIP_PRODUCT, RPE_MAP_CROSS,
                                                    RPE_MAP_EUCLIDEAN, RPE_MAP_PRODUCT,
                                                    RPE_TABLES_CROSS, RpeError)
from vision_transformer_attention_gb300.workloads import FLAG_K, FLAG_Q, FLAG_V

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F32 = 1e-4
R19 = workloads.index_constants(1.9)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert api.rpe_device_status(clear=True) == 0


def _maxerr(gpu, ref):
    return float(np.max(np.abs(gpu.detach().float().cpu().numpy().astype(np.float64) - ref)))


def _ids(H, W, mode, consts=R19):
    if mode == RPE_MAP_EUCLIDEAN:
        return oracle.euclidean_bucket_ids(H, W, *consts)
    return oracle.product_bucket_ids(H, W, *consts)


@pytest.mark.parametrize("H,W,ratio", [(14, 14, 1.9), (56, 56, 1.9), (5, 9, 1.9), (1, 7, 1.9),
                                       (14, 14, 2.0), (9, 4, 3.5), (1, 1, 1.9)])
def test_euclidean_ids_bit_exact(H, W, ratio):
    consts = workloads.index_constants(ratio)
    lut, ids, nb = api.rpe_build_bucket_ids(H, W, *consts, with_ids=True, mode=RPE_MAP_EUCLIDEAN)
    ref, nb_ref = oracle.euclidean_bucket_ids(H, W, *consts)
    assert nb == nb_ref == 2 * int(consts[1]) + 1
    assert np.array_equal(ids.cpu().numpy(), ref)


# With only 7 Euclidean buckets the value term gathers a row's probability mass
# on few table rows, and at table_std 1 outputs reach 4, where half a bf16 ulp
# alone is 2^-6; the value-term case therefore uses table_std 0.5.
@pytest.mark.parametrize("B,heads,H,W,flags,dtype,table_std", [
    (2, 3, 14, 14, FLAG_K, "bf16", 1.0),                    # two-warpgroup kernel, W = 14
    (2, 3, 14, 14, FLAG_K | FLAG_Q, "bf16", 1.0),           # same, with the query term
    # the value term's bucket sums need each id to form one run along a grid row
    # of keys; Euclidean ids repeat on both sides of the query column, so this
    # runs on the general kernel
    (2, 3, 14, 14, FLAG_K | FLAG_Q | FLAG_V, "bf16", 0.5),
    (1, 2, 9, 12, FLAG_K | FLAG_Q | FLAG_V, "bf16", 0.5),   # general kernel
    (1, 2, 5, 9, FLAG_K | FLAG_V, "f32", 1.0),              # fp32 path
])
def test_euclidean_attention_matches_oracle(B, heads, H, W, flags, dtype, table_std):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=RPE_MAP_EUCLIDEAN)
    inp = workloads.irpe_inputs(B, heads, H * W, 64 if dtype == "bf16" else 32, nb, flags, dtype,
                                table_std=table_std, seed=H + W)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    ids, K = _ids(H, W, RPE_MAP_EUCLIDEAN)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags,
                                    tab_q=inp["tab_q"], tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert _maxerr(out, ref) <= (TOL_BF16 if dtype == "bf16" else TOL_F32)


def _row_runs(lut, H, W):
    """Python statement of the offset-table property the value term's bucket
    sums rely on: seen from any query column, each id forms one run along a
    grid row of W keys."""
    t = lut.cpu().numpy().reshape(2 * H - 1, 2 * W - 1)
    for r in range(2 * H - 1):
        for qx in range(W):
            seq = [int(t[r, qx - kx + W - 1]) for kx in range(W)]
            runs = [a for i, a in enumerate(seq) if i == 0 or a != seq[i - 1]]
            if len(runs) != len(set(runs)):
                return False
    return True


@pytest.mark.parametrize("mode", [RPE_MAP_PRODUCT, RPE_MAP_EUCLIDEAN, RPE_MAP_CROSS,
                                  RPE_MAP_CLIP_PRODUCT])
def test_built_tables_row_run_property(mode):
    # the library records this property for the tables it builds without reading
    # them back: true for Product, Cross and clip ids, false for Euclidean
    for H, W, ratio in [(14, 14, 1.9), (10, 14, 2.0), (14, 14, 3.5)]:
        lut, _, _ = api.rpe_build_bucket_ids(H, W, *workloads.index_constants(ratio), mode=mode)
        assert _row_runs(lut, H, W) == (mode != RPE_MAP_EUCLIDEAN)


@pytest.mark.parametrize("mode", [RPE_MAP_PRODUCT, RPE_MAP_EUCLIDEAN])
def test_value_term_with_a_foreign_table(mode):
    # a table the library did not build is read back once and checked for the
    # property; either way the result matches the oracle
    H, W, flags = 14, 14, FLAG_K | FLAG_V
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=mode)
    foreign = lut.clone()
    inp = workloads.irpe_inputs(2, 3, H * W, 64, nb, flags, "bf16", table_std=0.5, seed=31)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], foreign, nb, H, W, flags,
                           table_k=g["tab_k"], table_v=g["tab_v"])
    ids, K = _ids(H, W, mode)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags,
                                    tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert _maxerr(out, ref) <= TOL_BF16


def test_euclidean_attention_56x56_sampled():
    B, heads, H, W = 2, 3, 56, 56
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=RPE_MAP_EUCLIDEAN)
    inp = workloads.irpe_inputs(B, heads, H * W, 64, nb, FLAG_K, "bf16", table_std=1.0, seed=7)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, FLAG_K, table_k=g["tab_k"])
    ids, K = _ids(H, W, RPE_MAP_EUCLIDEAN)
    rows = np.unique(np.concatenate([np.arange(0, 24), np.arange(1500, 1520), np.arange(3110, 3136)]))
    sl = np.array([0, 5])
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, FLAG_K,
                                    tab_k=inp["tab_k"], slices=sl, rows=rows)
    S = B * heads
    got = out.reshape(S, H * W, 64)[torch.as_tensor(sl, device=out.device)][:, torch.as_tensor(rows, device=out.device)]
    assert _maxerr(got, ref.reshape(S, H * W, 64)[sl][:, rows]) <= TOL_BF16


def _bias_case(B, heads, H, W, mode, shared, dtype, table_std, seed):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=mode)
    d = 64 if dtype == "bf16" else 32
    inp = workloads.irpe_inputs(B, heads, H * W, d, nb, 0, dtype, seed=seed)
    bias = workloads.bias_table(nb, 1 if shared else heads, table_std, seed + 100)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_bias_fwd(g["q"], g["k"], g["v"], bias.cuda(), lut, nb, H, W)
    ids, K = _ids(H, W, mode)
    return inp, bias, ids, K, out


@pytest.mark.parametrize("H,W,mode,shared,dtype", [
    (14, 14, RPE_MAP_PRODUCT, False, "bf16"),
    (14, 14, RPE_MAP_PRODUCT, True, "bf16"),
    (14, 14, RPE_MAP_EUCLIDEAN, False, "bf16"),
    (9, 14, RPE_MAP_PRODUCT, False, "bf16"),     # 126 rows: one query tile per item
    (6, 9, RPE_MAP_PRODUCT, False, "bf16"),      # general kernel (W not 14 or 56)
    (20, 13, RPE_MAP_EUCLIDEAN, True, "bf16"),   # general kernel, two key tiles
    (5, 9, RPE_MAP_PRODUCT, False, "f32"),
    (5, 9, RPE_MAP_EUCLIDEAN, True, "f32"),
])
def test_bias_mode_matches_oracle(H, W, mode, shared, dtype):
    inp, bias, ids, K, out = _bias_case(2, 3, H, W, mode, shared, dtype, 2.0, seed=H * W)
    b = bias.numpy()[:, 0] if shared else bias.numpy()
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, 0, bias_in=b)
    assert _maxerr(out, ref) <= (TOL_BF16 if dtype == "bf16" else TOL_F32)
    # negative control: at this size the bias moves the output well beyond the tolerance
    plain = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, 0)
    assert np.max(np.abs(plain - ref)) > 3 * TOL_BF16


def test_bias_mode_56x56_sampled():
    B, heads, H, W = 2, 3, 56, 56
    inp, bias, ids, K, out = _bias_case(B, heads, H, W, RPE_MAP_PRODUCT, False, "bf16", 2.0, seed=9)
    rows = np.unique(np.concatenate([np.arange(0, 24), np.arange(3110, 3136)]))
    sl = np.array([1, 4])
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, 0, bias_in=bias.numpy(),
                                    slices=sl, rows=rows)
    S = B * heads
    got = out.reshape(S, H * W, 64)[torch.as_tensor(sl, device=out.device)][:, torch.as_tensor(rows, device=out.device)]
    assert _maxerr(got, ref.reshape(S, H * W, 64)[sl][:, rows]) <= TOL_BF16


def test_bias_mode_bf16_unsupported_head_dim_is_an_error():
    lut, _, nb = api.rpe_build_bucket_ids(6, 9, *R19)
    inp = workloads.irpe_inputs(1, 2, 54, 32, nb, 0, "bf16")
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    with pytest.raises(RpeError):
        api.rpe_attn_bias_fwd(g["q"], g["k"], g["v"], workloads.bias_table(nb, 2).cuda(), lut, nb, 6, 9)


# ------------------------------------------------------------ Cross mapping (eqs. 22-24)

@pytest.mark.parametrize("H,W,ratio", [(14, 14, 1.9), (5, 9, 1.9), (56, 56, 1.9), (9, 4, 2.0),
                                       (1, 1, 1.9)])
def test_cross_ids_bit_exact(H, W, ratio):
    consts = workloads.index_constants(ratio)
    lut, ids, nb = api.rpe_build_bucket_ids(H, W, *consts, with_ids=True, mode=RPE_MAP_CROSS)
    ref_row, ref_col, nb_ref = oracle.cross_bucket_ids(H, W, *consts)
    assert nb == nb_ref == 2 * (2 * int(consts[1]) + 1)
    got = ids.cpu().numpy()
    assert np.array_equal(got[0], ref_row) and np.array_equal(got[1], ref_col)


def _cross_case(B, heads, H, W, flags, dtype, table_std, seed, rows=None, slices=None):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=RPE_MAP_CROSS)
    inp = workloads.irpe_inputs(B, heads, H * W, 64 if dtype == "bf16" else 32, nb, flags, dtype,
                                table_std=table_std, seed=seed)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags | RPE_TABLES_CROSS,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    ids_row, ids_col, K = oracle.cross_bucket_ids(H, W, *R19)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids_row, K, flags,
                                    tab_q=inp["tab_q"], tab_k=inp["tab_k"], tab_v=inp["tab_v"],
                                    ids2=ids_col, rows=rows, slices=slices)
    return inp, out, ref


@pytest.mark.parametrize("B,heads,H,W,flags,dtype,table_std", [
    (2, 3, 14, 14, FLAG_K, "bf16", 1.0),                    # two-warpgroup kernel
    (1, 2, 20, 14, FLAG_K, "bf16", 1.0),                    # same, ragged last key tile
    (1, 2, 9, 12, FLAG_K | FLAG_Q | FLAG_V, "bf16", 0.5),   # general kernel, all terms
    (1, 2, 11, 7, FLAG_Q | FLAG_V, "bf16", 0.5),
    (1, 2, 5, 9, FLAG_K | FLAG_Q | FLAG_V, "f32", 1.0),     # fp32 path
])
def test_cross_attention_matches_oracle(B, heads, H, W, flags, dtype, table_std):
    inp, out, ref = _cross_case(B, heads, H, W, flags, dtype, table_std, seed=H * W + flags)
    assert _maxerr(out, ref) <= (TOL_BF16 if dtype == "bf16" else TOL_F32)
    # negative control: the column half of the tables matters beyond the tolerance
    ids_row, _, K = oracle.cross_bucket_ids(H, W, *R19)
    rows_only = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids_row, K, flags,
                                          tab_q=inp["tab_q"], tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert np.max(np.abs(rows_only - ref)) > 3 * TOL_BF16


def test_cross_attention_56x56_sampled():
    rows = np.unique(np.concatenate([np.arange(0, 24), np.arange(3110, 3136)]))
    sl = np.array([0, 5])
    B, heads, H, W = 2, 3, 56, 56
    _, out, ref = _cross_case(B, heads, H, W, FLAG_K, "bf16", 1.0, seed=11, rows=rows, slices=sl)
    S = B * heads
    got = out.reshape(S, H * W, 64)[torch.as_tensor(sl, device=out.device)][:, torch.as_tensor(rows, device=out.device)]
    assert _maxerr(got, ref.reshape(S, H * W, 64)[sl][:, rows]) <= TOL_BF16


@pytest.mark.parametrize("H,W,dtype", [(14, 14, "bf16"), (9, 12, "bf16"), (5, 9, "f32")])
def test_cross_bias_mode_matches_oracle(H, W, dtype):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=RPE_MAP_CROSS)
    d = 64 if dtype == "bf16" else 32
    inp = workloads.irpe_inputs(2, 3, H * W, d, nb, 0, dtype, seed=H + 3)
    bias = workloads.bias_table(nb, 3, 2.0, seed=H + 4)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_bias_fwd(g["q"], g["k"], g["v"], bias.cuda(), lut, nb, H, W, cross=True)
    ids_row, ids_col, K = oracle.cross_bucket_ids(H, W, *R19)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids_row, K, 0,
                                    bias_in=bias.numpy(), ids2=ids_col)
    assert _maxerr(out, ref) <= (TOL_BF16 if dtype == "bf16" else TOL_F32)


def test_cross_tables_beyond_64_joint_ids_are_refused():
    lut, _, nb = api.rpe_build_bucket_ids(14, 14, *workloads.index_constants(2.0), mode=RPE_MAP_CROSS)
    assert nb == 18   # span 9: 81 joint ids
    inp = workloads.irpe_inputs(1, 1, 196, 64, nb, FLAG_K, "bf16")
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    with pytest.raises(RpeError):
        api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, 14, 14, FLAG_K | RPE_TABLES_CROSS,
                         table_k=g["tab_k"])


# ------------------------------------------------------------ clip index (table 3)

@pytest.mark.parametrize("H,W,ratio", [(14, 14, 1.9), (7, 20, 1.9), (9, 9, 1.0), (56, 56, 2.0)])
def test_clip_product_ids_bit_exact(H, W, ratio):
    consts = workloads.index_constants(ratio)
    lut, ids, nb = api.rpe_build_bucket_ids(H, W, *consts, with_ids=True, mode=RPE_MAP_CLIP_PRODUCT)
    ref, nb_ref = oracle.clip_product_bucket_ids(H, W, int(consts[1]))
    assert nb == nb_ref
    assert np.array_equal(ids.cpu().numpy(), ref)


@pytest.mark.parametrize("H,W,flags", [(14, 14, FLAG_K), (6, 10, FLAG_K | FLAG_V)])
def test_clip_product_attention_matches_oracle(H, W, flags):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=RPE_MAP_CLIP_PRODUCT)
    inp = workloads.irpe_inputs(2, 3, H * W, 64, nb, flags, "bf16", table_std=1.0, seed=H + W + 1)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags,
                           table_k=g["tab_k"], table_v=g["tab_v"])
    ids, K = oracle.clip_product_bucket_ids(H, W, int(R19[1]))
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags,
                                    tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert _maxerr(out, ref) <= TOL_BF16


# ------------------------------------------------------------ per-head tables (section 4.2)

@pytest.mark.parametrize("B,heads,H,W,flags,mode,dtype,table_std", [
    (2, 3, 14, 14, FLAG_K, RPE_MAP_PRODUCT, "bf16", 1.0),      # two-warpgroup kernel
    (3, 2, 20, 14, FLAG_K, RPE_MAP_CROSS, "bf16", 1.0),        # same, Cross tables
    (2, 3, 10, 10, FLAG_K, RPE_MAP_PRODUCT, "bf16", 1.0),      # general kernel
    (2, 2, 9, 12, FLAG_K | FLAG_Q | FLAG_V, RPE_MAP_PRODUCT, "bf16", 0.5),
    (1, 3, 12, 11, FLAG_Q | FLAG_V, RPE_MAP_CROSS, "bf16", 0.5),
    (2, 2, 5, 9, FLAG_K | FLAG_Q | FLAG_V, RPE_MAP_PRODUCT, "f32", 1.0),
])
def test_per_head_tables_match_oracle(B, heads, H, W, flags, mode, dtype, table_std):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19, mode=mode)
    inp = workloads.irpe_inputs(B, heads, H * W, 64 if dtype == "bf16" else 32, nb, flags, dtype,
                                table_std=table_std, seed=H * W + 5, per_head=True)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    cross = RPE_TABLES_CROSS if mode == RPE_MAP_CROSS else 0
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags | cross,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    if mode == RPE_MAP_CROSS:
        ids, ids2, K = oracle.cross_bucket_ids(H, W, *R19)
    else:
        (ids, K), ids2 = oracle.product_bucket_ids(H, W, *R19), None
    tabs = {n: inp[n] for n in ("tab_q", "tab_k", "tab_v")}
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags, ids2=ids2, **tabs)
    assert _maxerr(out, ref) <= (TOL_BF16 if dtype == "bf16" else TOL_F32)
    # negative control: head 0's tables for every head would fail the bar
    head0 = {n: (None if t is None else t[0]) for n, t in tabs.items()}
    shared = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags, ids2=ids2,
                                       **head0)
    assert np.max(np.abs(shared - ref)) > 3 * TOL_BF16


def test_per_head_tables_56x56_sampled():
    B, heads, H, W = 2, 3, 56, 56
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    inp = workloads.irpe_inputs(B, heads, H * W, 64, nb, FLAG_K, "bf16", table_std=1.0, seed=13,
                                per_head=True)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, FLAG_K, table_k=g["tab_k"])
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    rows = np.unique(np.concatenate([np.arange(0, 24), np.arange(3110, 3136)]))
    sl = np.array([1, 2, 3])
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, FLAG_K,
                                    tab_k=inp["tab_k"], slices=sl, rows=rows)
    S = B * heads
    got = out.reshape(S, H * W, 64)[torch.as_tensor(sl, device=out.device)][:, torch.as_tensor(rows, device=out.device)]
    assert _maxerr(got, ref.reshape(S, H * W, 64)[sl][:, rows]) <= TOL_BF16


# ------------------------------------------------------------ more than 64 buckets (r = 2.0)

R20 = workloads.index_constants(2.0)


def test_product_ids_r2_bit_exact():
    lut, ids, nb = api.rpe_build_bucket_ids(25, 34, *R20, with_ids=True)
    ref, K = oracle.product_bucket_ids(25, 34, *R20)
    assert nb == K == 81
    assert np.array_equal(ids.cpu().numpy(), ref)


@pytest.mark.parametrize("B,heads,H,W,flags,dtype,table_std", [
    (2, 3, 14, 14, FLAG_K, "bf16", 1.0),            # general kernel, two QR rounds
    (1, 2, 13, 17, FLAG_K | FLAG_V, "bf16", 0.5),   # ragged grid, 128-bucket PB R^V
    (1, 2, 9, 9, FLAG_V, "bf16", 0.5),
    (1, 2, 9, 11, FLAG_K | FLAG_Q | FLAG_V, "f32", 1.0),
])
def test_r2_81_buckets_match_oracle(B, heads, H, W, flags, dtype, table_std):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R20)
    assert nb == 81
    inp = workloads.irpe_inputs(B, heads, H * W, 64 if dtype == "bf16" else 32, nb, flags, dtype,
                                table_std=table_std, seed=H * W + 17)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    ids, K = oracle.product_bucket_ids(H, W, *R20)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags,
                                    tab_q=inp["tab_q"], tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert _maxerr(out, ref) <= (TOL_BF16 if dtype == "bf16" else TOL_F32)
    # negative control: buckets 64..80 (offsets with row index +3 or +4) matter
    tabs = {n: inp[n] for n in ("tab_q", "tab_k", "tab_v")}
    cut = {n: (None if t is None else torch.cat([t[:64], 0 * t[64:]])) for n, t in tabs.items()}
    low = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags, **cut)
    assert np.max(np.abs(low - ref)) > 3 * TOL_BF16


def test_r2_deit_s_config_sampled():
    cfg = workloads.CONFIGS["irpe_k_r2_deit_s"]
    lut, _, nb = api.rpe_build_bucket_ids(cfg.H, cfg.W, *workloads.index_constants(cfg.ratio))
    assert nb == cfg.num_buckets == 81
    inp = workloads.config_inputs(cfg)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, cfg.H, cfg.W, cfg.flags,
                           table_k=g["tab_k"])
    S = cfg.B * cfg.heads
    rng = np.random.default_rng(4)
    sl = np.unique(np.concatenate([rng.choice(S, 12, replace=False), [0, S - 1]]))
    ids, K = oracle.product_bucket_ids(cfg.H, cfg.W, *R20)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, cfg.flags,
                                    tab_k=inp["tab_k"], slices=sl).reshape(S, cfg.N, 64)[sl]
    got = out.reshape(S, cfg.N, 64)[torch.as_tensor(sl, device=out.device)]
    assert _maxerr(got, ref) <= TOL_BF16


def test_r2_bias_mode_on_the_two_warpgroup_kernel():
    H, W = 14, 14
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R20)
    inp = workloads.irpe_inputs(2, 3, H * W, 64, nb, 0, "bf16", seed=21)
    bias = workloads.bias_table(nb, 3, 2.0, seed=22)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_bias_fwd(g["q"], g["k"], g["v"], bias.cuda(), lut, nb, H, W)
    ids, K = oracle.product_bucket_ids(H, W, *R20)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, 0, bias_in=bias.numpy())
    assert _maxerr(out, ref) <= TOL_BF16


def test_fp32_takes_225_buckets():
    ratio = 3.5   # beta 7: 15 x 15 buckets
    H, W = 8, 12
    consts = workloads.index_constants(ratio)
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *consts)
    assert nb == 225
    inp = workloads.irpe_inputs(1, 2, H * W, 16, nb, FLAG_K | FLAG_V, "f32", table_std=1.0, seed=3)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, FLAG_K | FLAG_V,
                           table_k=g["tab_k"], table_v=g["tab_v"])
    ids, K = oracle.product_bucket_ids(H, W, *consts)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, FLAG_K | FLAG_V,
                                    tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert _maxerr(out, ref) <= TOL_F32


def test_query_term_beyond_64_buckets_is_refused_in_bf16():
    lut, _, nb = api.rpe_build_bucket_ids(14, 14, *R20)
    inp = workloads.irpe_inputs(1, 1, 196, 64, nb, FLAG_Q, "bf16")
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    with pytest.raises(RpeError):
        api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, 14, 14, FLAG_Q, table_q=g["tab_q"])


# ------------------------------------------------------------ class token (section 4.1)

def _cls_case(B, heads, H, W, flags, dtype, table_std, seed, ratio=1.9, per_head=False,
              rows=None, slices=None):
    consts = workloads.index_constants(ratio)
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *consts)
    K1 = nb + 1
    inp = workloads.irpe_inputs(B, heads, H * W + 1, 64 if dtype == "bf16" else 32, K1, flags,
                                dtype, table_std=table_std, seed=seed, per_head=per_head)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, K1, H, W, flags, cls_token=True,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    ids, K = oracle.add_cls_bucket(*oracle.product_bucket_ids(H, W, *consts))
    tabs = {n: inp[n] for n in ("tab_q", "tab_k", "tab_v")}
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags, rows=rows,
                                    slices=slices, **tabs)
    return inp, out, ref, ids, K


@pytest.mark.parametrize("B,heads,H,W,flags,dtype,table_std,ratio,per_head", [
    (2, 3, 14, 14, FLAG_K, "bf16", 1.0, 1.9, False),           # DeiT-S grid + class token
    (1, 2, 9, 12, FLAG_K | FLAG_Q | FLAG_V, "bf16", 0.5, 1.9, False),
    (2, 2, 11, 11, FLAG_K, "bf16", 1.0, 1.9, True),            # per-head tables
    (1, 2, 10, 13, FLAG_K | FLAG_V, "bf16", 0.5, 2.0, False),  # 82 buckets
    (1, 1, 1, 1, FLAG_K, "bf16", 1.0, 1.9, False),             # one patch and the class token
    (2, 2, 5, 9, FLAG_K | FLAG_Q | FLAG_V, "f32", 1.0, 1.9, False),
])
def test_cls_token_matches_oracle(B, heads, H, W, flags, dtype, table_std, ratio, per_head):
    inp, out, ref, ids, K = _cls_case(B, heads, H, W, flags, dtype, table_std, seed=H * W + 31,
                                      ratio=ratio, per_head=per_head)
    assert _maxerr(out, ref) <= (TOL_BF16 if dtype == "bf16" else TOL_F32)
    if H * W > 1:
        # negative control: the class bucket's table row matters beyond the tolerance
        tabs = {n: inp[n] for n in ("tab_q", "tab_k", "tab_v")}
        cut = {}
        for n, t in tabs.items():
            if t is not None:
                t = t.clone()
                t[..., K - 1, :] = 0
            cut[n] = t
        without = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags, **cut)
        assert np.max(np.abs(without - ref)) > 3 * TOL_BF16


def test_cls_token_56x56_whole_slices():
    # two whole slices (3137 rows each) of a 56 x 56 grid with the class token,
    # on the two-warpgroup kernel (its widened QR' product in 96-column slots)
    B, heads, H, W = 1, 6, 56, 56
    consts = workloads.index_constants(1.9)
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *consts)
    inp = workloads.irpe_inputs(B, heads, H * W + 1, 64, nb + 1, FLAG_K, "bf16", table_std=1.0,
                                seed=41)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb + 1, H, W, FLAG_K, cls_token=True,
                           table_k=g["tab_k"])
    ids, K = oracle.add_cls_bucket(*oracle.product_bucket_ids(H, W, *consts))
    sl = np.array([0, 5])
    f64 = {k: oracle._f64(t) for k, t in inp.items() if t is not None}
    ref = np.zeros_like(f64["q"])
    oracle.parallel_slices(lambda s_: oracle.irpe_attention_ids(
        f64["q"], f64["k"], f64["v"], ids, K, FLAG_K, tab_k=f64["tab_k"], slices=s_, out=ref), sl)
    N, S = H * W + 1, B * heads
    got = out.reshape(S, N, 64)[torch.as_tensor(sl, device=out.device)]
    assert _maxerr(got, ref.reshape(S, N, 64)[sl]) <= TOL_BF16


@pytest.mark.parametrize("H,W,dtype,shared", [(6, 7, "f32", False), (6, 7, "bf16", False),
                                              (14, 14, "bf16", True), (9, 20, "bf16", False)])
def test_cls_bias_mode(H, W, dtype, shared):
    # the class bucket's bias on every pair with token 0 (bf16: the general kernel)
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    d = 32 if dtype == "f32" else 64
    inp = workloads.irpe_inputs(2, 3, H * W + 1, d, nb + 1, 0, dtype, seed=43)
    bias = workloads.bias_table(nb + 1, 1 if shared else 3, 2.0, seed=44)
    bias[-1] = 16.0   # the class bucket: about two logits above the rest, so that it shows
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_bias_fwd(g["q"], g["k"], g["v"], bias.cuda(), lut, nb + 1, H, W,
                                cls_token=True)
    ids, K = oracle.add_cls_bucket(*oracle.product_bucket_ids(H, W, *R19))
    b = bias.numpy()[:, 0] if shared else bias.numpy()
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, 0, bias_in=b)
    assert _maxerr(out, ref) <= (TOL_F32 if dtype == "f32" else TOL_BF16)
    # negative control: dropping the class bucket's bias moves the output past the tolerance
    b0 = b.copy()
    b0[-1] = 0.0
    off = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, 0, bias_in=b0)
    assert np.max(np.abs(off - ref)) > 3 * TOL_BF16


def test_deit_s_cls_config_sampled():
    cfg = workloads.CONFIGS["irpe_k_deit_s_cls"]
    assert (cfg.N, cfg.num_buckets) == (197, 50)
    lut, _, nb = api.rpe_build_bucket_ids(cfg.H, cfg.W, *workloads.index_constants(cfg.ratio))
    inp = workloads.config_inputs(cfg)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, cfg.num_buckets, cfg.H, cfg.W, cfg.flags,
                           cls_token=True, table_k=g["tab_k"])
    S = cfg.B * cfg.heads
    sl = np.array([0, 77, S - 1])
    ids, K = oracle.add_cls_bucket(*oracle.product_bucket_ids(cfg.H, cfg.W, *R19))
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, cfg.flags,
                                    tab_k=inp["tab_k"], slices=sl).reshape(S, cfg.N, 64)[sl]
    got = out.reshape(S, cfg.N, 64)[torch.as_tensor(sl, device=out.device)]
    assert _maxerr(got, ref) <= TOL_BF16


@pytest.mark.parametrize("B,heads,H,W,per_head", [
    (2, 3, 14, 14, False),   # two-warpgroup kernel, 5-row key tiles, 197 tokens
    (1, 2, 28, 14, False),   # 6-row key tiles, 393 tokens
    (2, 2, 1, 14, False),    # one grid row: 15 tokens, one query tile
    (1, 3, 9, 14, True),     # 127 tokens (one query tile), per-head tables
    (1, 2, 10, 14, True),    # 141 tokens (a pair of query tiles), per-head tables
    (1, 2, 3, 56, False),    # W = 56: 169 tokens (a pair of query tiles)
    (2, 2, 2, 56, True),     # 113 tokens (one query tile), per-head tables
    (1, 2, 5, 56, False),    # 281 tokens (a pair and an odd last tile)
])
def test_cls_token_two_warpgroup_kernel(B, heads, H, W, per_head):
    # the class key is folded into each row after the grid keys and the class
    # query reads the class bucket for every key; the hard-to-fake part is the
    # class key's own term, so the tables are large (std 1)
    inp, out, ref, ids, K = _cls_case(B, heads, H, W, FLAG_K, "bf16", 1.0, seed=H * 7 + heads,
                                      per_head=per_head)
    assert _maxerr(out, ref) <= TOL_BF16
    tab = inp["tab_k"].clone()
    tab[..., K - 1, :] = 0
    without = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, FLAG_K, tab_k=tab)
    assert np.max(np.abs(without - ref)) > 3 * TOL_BF16


@pytest.mark.parametrize("B,heads,H,W,sampled", [
    (1, 3, 28, 14, False),   # two-warpgroup kernel, 6-row key tiles, two QR' rounds
    (2, 2, 1, 14, False),    # one grid row
    (1, 3, 56, 56, True),    # W = 56
])
def test_r2_81_buckets_two_warpgroup_kernel(B, heads, H, W, sampled):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R20)
    inp = workloads.irpe_inputs(B, heads, H * W, 64, nb, FLAG_K, "bf16", table_std=1.0, seed=H + W + 61)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, FLAG_K, table_k=g["tab_k"])
    ids, K = oracle.product_bucket_ids(H, W, *R20)
    N, S = H * W, B * heads
    rows = np.unique(np.concatenate([np.arange(0, 40), np.arange(N - 40, N)])) if sampled else None
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, FLAG_K,
                                    tab_k=inp["tab_k"], rows=rows)
    if sampled:
        idx = torch.as_tensor(rows, device=out.device)
        assert _maxerr(out.reshape(S, N, 64)[:, idx], ref.reshape(S, N, 64)[:, rows]) <= TOL_BF16
    else:
        assert _maxerr(out, ref) <= TOL_BF16
