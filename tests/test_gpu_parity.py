"""GPU parity: the CUDA library, called through its C ABI, against the oracle.

Tolerances: bucket ids bit-exact (integer work);
bf16 attention <= 2e-2 max abs error (bf16 inputs, fp32 accumulation,
probabilities rounded to bf16 before the value products); fp32 attention
<= 1e-4 max abs error.
"""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_attention_gb300 import api, workloads
from vision_transformer_attention_gb300.workloads import CONFIGS, FLAG_K, FLAG_Q, FLAG_V

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


def _dev(d):
    return {k: (None if t is None else t.cuda()) for k, t in d.items()}


def _maxerr(gpu, ref):
    return float(np.max(np.abs(gpu.detach().float().cpu().numpy().astype(np.float64) - ref)))


# ------------------------------------------------------------------ bucket ids

@pytest.mark.parametrize("H,W,ratio", [(14, 14, 1.9), (56, 56, 1.9), (5, 9, 1.9), (1, 7, 1.9),
                                       (14, 14, 2.0), (9, 4, 3.5), (1, 1, 1.9)])
def test_bucket_ids_bit_exact(H, W, ratio):
    a, b, g = workloads.index_constants(ratio)
    lut, ids, nb = api.rpe_build_bucket_ids(H, W, a, b, g, with_ids=True)
    ref, nb_ref = oracle.product_bucket_ids(H, W, a, b, g)
    assert nb == nb_ref
    assert np.array_equal(ids.cpu().numpy(), ref)


# ------------------------------------------------------------------ Swin

def _swin_case(nw, heads, d, dtype, table_std=0.02, seed=0):
    inp = workloads.swin_inputs(nw, heads, 7, d, dtype, table_std, seed)
    g = _dev(inp)
    out = api.swin_window_attn_fwd(g["q"], g["k"], g["v"], g["table"], 7)
    return inp, out


@pytest.mark.parametrize("table_std", [0.02, 2.0])
def test_swin_fp32_small_config(table_std):
    cfg = CONFIGS["swin_w7_small_fp32"]
    inp, out = _swin_case(cfg.num_windows, cfg.heads, cfg.d, "f32", table_std)
    ref = oracle.swin_attention(inp["q"], inp["k"], inp["v"], inp["table"], 7)
    assert _maxerr(out, ref) <= TOL_F32
    if table_std > 1:  # negative control: the bias matters far beyond the tolerance
        plain = oracle.swin_attention(inp["q"], inp["k"], inp["v"], 0 * inp["table"], 7)
        assert np.max(np.abs(plain - ref)) > 50 * TOL_F32


@pytest.mark.parametrize("nw,heads,d", [(4, 3, 32), (5, 3, 32), (1, 1, 32), (3, 5, 64), (37, 3, 32)])
@pytest.mark.parametrize("table_std", [0.02, 2.0])
def test_swin_bf16_small(nw, heads, d, table_std):
    inp, out = _swin_case(nw, heads, d, "bf16", table_std, seed=nw)
    ref = oracle.swin_attention(inp["q"], inp["k"], inp["v"], inp["table"], 7)
    assert _maxerr(out, ref) <= TOL_BF16


def _swin_ref_threads(inp, M):
    """The oracle on every (window, head) unit, the units split over host cores."""
    f64 = {k: oracle._f64(t) for k, t in inp.items()}
    out = np.zeros_like(f64["q"])
    units = f64["q"].shape[0] * f64["q"].shape[1]
    oracle.parallel_slices(lambda sl: oracle.swin_attention(
        f64["q"], f64["k"], f64["v"], f64["table"], M, slices=sl, out=out), np.arange(units))
    return out


@pytest.mark.parametrize("table_std", [0.02, 2.0])
def test_swin_bf16_swin_t_stage1_whole(table_std):
    # every one of the 6144 (window, head) units, element by element
    cfg = CONFIGS["swin_t_stage1"]
    inp, out = _swin_case(cfg.num_windows, cfg.heads, cfg.d, "bf16", table_std)
    units = cfg.num_windows * cfg.heads
    assert _maxerr(out, _swin_ref_threads(inp, 7)) <= TOL_BF16
    # property at any size: every output row is a convex combination of its window's v rows
    v = inp["v"].float().reshape(units, 49, cfg.d).cuda()
    o = out.float().reshape(units, 49, cfg.d)
    assert torch.all(o <= v.amax(dim=1, keepdim=True) + TOL_BF16)
    assert torch.all(o >= v.amin(dim=1, keepdim=True) - TOL_BF16)


def test_swin_bf16_repeat_is_deterministic():
    inp, out1 = _swin_case(9, 3, 32, "bf16")
    g = _dev(inp)
    out2 = api.swin_window_attn_fwd(g["q"], g["k"], g["v"], g["table"], 7)
    assert torch.equal(out1, out2)


# ------------------------------------------------------------------ iRPE, fp32 path

@pytest.mark.parametrize("H,W,flags", [(4, 5, FLAG_K), (7, 7, FLAG_Q | FLAG_K | FLAG_V),
                                       (14, 14, FLAG_K | FLAG_V), (3, 30, FLAG_Q)])
def test_irpe_fp32_small(H, W, flags):
    B, heads, d = 2, 3, 64
    nb = 49
    inp = workloads.irpe_inputs(B, heads, H * W, d, nb, flags, "f32", table_std=1.0)
    g = _dev(inp)
    lut, _, nb_dev = api.rpe_build_bucket_ids(H, W, *R19)
    assert nb_dev == nb
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    ref = oracle.irpe_attention(inp["q"], inp["k"], inp["v"], H, W, *R19, flags,
                                tab_q=inp["tab_q"], tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert _maxerr(out, ref) <= TOL_F32


# ------------------------------------------------------------------ bounded waits

def test_wait_probe_times_out_and_reports():
    assert api.rpe_device_status(clear=True) == 0
    api.rpe_wait_probe(200_000)  # 0.2 ms bound on a barrier nothing arrives at
    status = api.rpe_device_status(clear=True)
    assert status != 0
    assert api.rpe_device_status(clear=True) == 0
    # the context is still usable afterwards
    inp, out = _swin_case(2, 3, 32, "bf16")
    ref = oracle.swin_attention(inp["q"], inp["k"], inp["v"], inp["table"], 7)
    assert _maxerr(out, ref) <= TOL_BF16


# ------------------------------------------------------------------ iRPE, bf16 tensor-core path

def _irpe_run(B, heads, H, W, flags, table_std=0.02, seed=0, inp=None):
    nb = 49
    if inp is None:
        inp = workloads.irpe_inputs(B, heads, H * W, 64, nb, flags, "bf16", table_std, seed)
    g = _dev(inp)
    lut, _, nb_dev = api.rpe_build_bucket_ids(H, W, *R19)
    assert nb_dev == nb
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    return inp, out


def _irpe_ref(inp, H, W, flags, slices=None, rows=None):
    return oracle.irpe_attention(inp["q"], inp["k"], inp["v"], H, W, *R19, flags,
                                 tab_q=inp["tab_q"], tab_k=inp["tab_k"], tab_v=inp["tab_v"],
                                 slices=slices, rows=rows)


ALL_TERMS = [0, FLAG_K, FLAG_Q, FLAG_V, FLAG_K | FLAG_Q, FLAG_K | FLAG_V, FLAG_Q | FLAG_V,
             FLAG_Q | FLAG_K | FLAG_V]


@pytest.mark.parametrize("flags", ALL_TERMS)
@pytest.mark.parametrize("table_std", [0.02, 1.0])
def test_irpe_bf16_terms_deit_grid(flags, table_std):
    # 14x14: two query tiles (128 + 68 rows) and two key tiles (128 + 68 keys)
    inp, out = _irpe_run(2, 3, 14, 14, flags, table_std, seed=flags)
    assert _maxerr(out, _irpe_ref(inp, 14, 14, flags)) <= TOL_BF16


@pytest.mark.parametrize("flags", ALL_TERMS)
def test_irpe_bf16_terms_general_kernel(flags):
    # a width the two-warpgroup kernel does not take: every term mix on the
    # general kernel (two query tiles, two key tiles with a ragged second)
    inp, out = _irpe_run(2, 3, 13, 11, flags, 1.0, seed=flags + 20)
    assert _maxerr(out, _irpe_ref(inp, 13, 11, flags)) <= TOL_BF16


@pytest.mark.parametrize("H,W,flags", [(4, 5, FLAG_K), (1, 1, FLAG_K), (3, 43, FLAG_Q | FLAG_K | FLAG_V),
                                       (16, 16, FLAG_K), (20, 13, FLAG_K | FLAG_V),
                                       (7, 64, FLAG_Q | FLAG_K)])
def test_irpe_bf16_ragged_grids(H, W, flags):
    inp, out = _irpe_run(1, 5, H, W, flags, table_std=1.0, seed=H * W)
    assert _maxerr(out, _irpe_ref(inp, H, W, flags)) <= TOL_BF16


def test_irpe_bf16_online_rescale_path():
    # keys of the later tiles get far larger logits than the first tile's, so the
    # running max jumps by more than 2^8 and the accumulator must be rescaled.
    # Rows become nearly one-hot, where rounding P and PB to bf16 (unit roundoff
    # 2^-8) costs up to 2^-8 * (max|v| + max|R^V|); v and R^V are halved so that
    # bound stays under the tolerance and only a real rescaling error can fail.
    H, W, flags = 20, 20, FLAG_K | FLAG_V
    inp = workloads.irpe_inputs(1, 2, H * W, 64, 49, flags, "bf16", 1.0, seed=5)
    k = inp["k"].float()
    k[:, :, 128:256] *= 6.0
    k[:, :, 256:] *= 12.0
    inp["k"] = k.to(torch.bfloat16)
    inp["v"] = (0.5 * inp["v"].float()).to(torch.bfloat16)
    inp["tab_v"] = (0.5 * inp["tab_v"].float()).to(torch.bfloat16)
    _, out = _irpe_run(1, 2, H, W, flags, inp=inp)
    assert _maxerr(out, _irpe_ref(inp, H, W, flags)) <= TOL_BF16


def _irpe_ref_threads(inp, H, W, flags, slices):
    """The oracle on the given (batch, head) slices, split over host cores,
    with the id map built once."""
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    f64 = {k: oracle._f64(t) for k, t in inp.items() if t is not None}
    out = np.zeros_like(f64["q"])
    oracle.parallel_slices(lambda sl: oracle.irpe_attention_ids(
        f64["q"], f64["k"], f64["v"], ids, K, flags, tab_q=f64.get("tab_q"),
        tab_k=f64.get("tab_k"), tab_v=f64.get("tab_v"), slices=sl, out=out), slices)
    return out


@pytest.mark.parametrize("name", ["irpe_k_deit_s", "irpe_qkv_deit_s"])
@pytest.mark.parametrize("table_std", [0.02, 1.0])
def test_irpe_bf16_deit_s_configs_whole(name, table_std):
    # every one of the 384 (batch, head) slices, element by element, in the
    # launch configuration bench.py times
    cfg = CONFIGS[name]
    inp, out = _irpe_run(cfg.B, cfg.heads, cfg.H, cfg.W, cfg.flags, table_std)
    S = cfg.B * cfg.heads
    assert _maxerr(out, _irpe_ref_threads(inp, cfg.H, cfg.W, cfg.flags, np.arange(S))) <= TOL_BF16


@pytest.mark.parametrize("flags", [FLAG_K, FLAG_Q | FLAG_K | FLAG_V])
def test_irpe_bf16_56x56_whole_slices(flags):
    # eight whole slices of the 56x56 workload (3136 rows each). With 624 items
    # on 152 SMs the last 16 items -- the odd last query tiles of slices 32..47
    # -- run as two parts merged through the workspace: slices 32, 40, 46 and
    # 47 cover those split items, 0, 1, 17 and 31 whole ones.
    cfg = CONFIGS["irpe_k_56x56"]
    inp, out = _irpe_run(cfg.B, cfg.heads, cfg.H, cfg.W, flags)
    S = cfg.B * cfg.heads
    sl = np.array([0, 1, 17, 31, 32, 40, 46, S - 1])
    ref = _irpe_ref_threads(inp, cfg.H, cfg.W, flags, sl).reshape(S, cfg.N, 64)[sl]
    got = out.reshape(S, cfg.N, 64)[torch.as_tensor(sl, device=out.device)]
    assert _maxerr(got, ref) <= TOL_BF16
    # any size: rows are convex combinations of v (plus the value term when on)
    if not flags & FLAG_V:
        v = inp["v"].float().cuda()
        o = out.float()
        assert torch.all(o <= v.amax(dim=2, keepdim=True) + TOL_BF16)
        assert torch.all(o >= v.amin(dim=2, keepdim=True) - TOL_BF16)


def test_irpe_bf16_repeat_is_deterministic():
    inp, out1 = _irpe_run(2, 2, 14, 14, FLAG_Q | FLAG_K | FLAG_V, 1.0)
    _, out2 = _irpe_run(2, 2, 14, 14, FLAG_Q | FLAG_K | FLAG_V, 1.0, inp=inp)
    assert torch.equal(out1, out2)


# ------------------------------------------------------------------ two-warpgroup path (W in {14, 56})

@pytest.mark.parametrize("H,W,flags", [(20, 14, FLAG_K), (10, 56, FLAG_K), (1, 14, FLAG_K),
                                       (9, 14, 0), (3, 56, 0), (28, 14, FLAG_K),
                                       # query / value terms: pairs of query tiles, ragged
                                       # second tile (10 x 14: 128 + 12 rows), two items
                                       # per slice (28 x 14), and grids they leave to the
                                       # general kernel (odd query-tile counts)
                                       (10, 14, FLAG_Q | FLAG_K | FLAG_V), (28, 14, FLAG_Q | FLAG_K | FLAG_V),
                                       (18, 14, FLAG_K | FLAG_V), (28, 14, FLAG_Q),
                                       (20, 14, FLAG_Q | FLAG_K | FLAG_V), (9, 14, FLAG_V)])
def test_irpe_bf16_pingpong_grids(H, W, flags):
    # odd and even numbers of query tiles, single-tile grids, ragged last key tile
    inp, out = _irpe_run(2, 3, H, W, flags, table_std=1.0, seed=H + W)
    assert _maxerr(out, _irpe_ref(inp, H, W, flags)) <= TOL_BF16


@pytest.mark.parametrize("B,heads,H,W,flags", [
    (1, 2, 28, 14, FLAG_K),                    # one item per CTA: the rescale at a group's last tile
    (1, 2, 10, 56, FLAG_K),                    # same at W = 56
    (40, 4, 28, 14, FLAG_K),                   # 320 items: some CTAs run three, so an item's last
    (40, 4, 28, 14, FLAG_Q | FLAG_K | FLAG_V),  # tile is followed by the next item's first unit
])
def test_irpe_bf16_pingpong_rescale_at_last_tiles(B, heads, H, W, flags):
    # the last grid row of keys gets far larger logits, so the reference max
    # jumps at the last key tile of every item (see the rescale test above for
    # the bound that halving v and R^V keeps under the tolerance)
    N = H * W
    inp = workloads.irpe_inputs(B, heads, N, 64, 49, flags, "bf16", 1.0, seed=13)
    k = inp["k"].float()
    k[:, :, N - W:] *= 12.0
    inp["k"] = k.to(torch.bfloat16)
    inp["v"] = (0.5 * inp["v"].float()).to(torch.bfloat16)
    if inp["tab_v"] is not None:
        inp["tab_v"] = (0.5 * inp["tab_v"].float()).to(torch.bfloat16)
    _, out = _irpe_run(B, heads, H, W, flags, inp=inp)
    S = B * heads
    sl = np.array(sorted({0, 1, S // 2, S - 1}))
    ref = _irpe_ref_threads(inp, H, W, flags, sl).reshape(S, N, 64)[sl]
    got = out.reshape(S, N, 64)[torch.as_tensor(sl, device=out.device)]
    assert _maxerr(got, ref) <= TOL_BF16


@pytest.mark.parametrize("flags", [FLAG_Q | FLAG_K | FLAG_V, FLAG_K | FLAG_V])
def test_irpe_bf16_qv_bucket_count_past_the_fast_layout(flags):
    # 60 declared buckets (ids 0..48 used): the two-warpgroup kernel's query /
    # value layout holds at most 51 next to each other, so the request runs on
    # the general kernel, with the same result as the oracle
    H, W, nb = 14, 14, 60
    lut, _, nb49 = api.rpe_build_bucket_ids(H, W, *R19)
    assert nb49 == 49
    inp = workloads.irpe_inputs(2, 3, H * W, 64, nb, flags, "bf16", 1.0, seed=61)
    g = _dev(inp)
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags,
                           table_q=g["tab_q"], table_k=g["tab_k"], table_v=g["tab_v"])
    ids, _ = oracle.product_bucket_ids(H, W, *R19)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, nb, flags,
                                    tab_q=inp["tab_q"], tab_k=inp["tab_k"], tab_v=inp["tab_v"])
    assert _maxerr(out, ref) <= TOL_BF16


@pytest.mark.parametrize("flags", [FLAG_K, FLAG_K | FLAG_V, FLAG_Q | FLAG_K | FLAG_V])
def test_irpe_bf16_pingpong_rescale_path(flags):
    # as test_irpe_bf16_online_rescale_path, on a width served by the two-warpgroup
    # kernel (with the value term, the bucket sums are rescaled with O)
    H, W = 28, 14
    inp = workloads.irpe_inputs(1, 2, H * W, 64, 49, flags, "bf16", 1.0, seed=7)
    k = inp["k"].float()
    k[:, :, 126:252] *= 6.0
    k[:, :, 252:] *= 12.0
    inp["k"] = k.to(torch.bfloat16)
    inp["v"] = (0.5 * inp["v"].float()).to(torch.bfloat16)
    if inp["tab_v"] is not None:
        inp["tab_v"] = (0.5 * inp["tab_v"].float()).to(torch.bfloat16)
    _, out = _irpe_run(1, 2, H, W, flags, inp=inp)
    assert _maxerr(out, _irpe_ref(inp, H, W, flags)) <= TOL_BF16


# ------------------------------------------------------------ split tail items (two-warpgroup kernel)

@pytest.mark.parametrize("flags,bias", [(FLAG_K, False), (0, True)])
def test_irpe_bf16_split_tail_items(flags, bias):
    # 200 slices of one item each on 152 SMs: the last 48 items run as two parts
    # on two CTAs each and are merged; check whole slices on both sides of the
    # boundary, and that repeating the call gives the same bits
    B, heads, H, W = 40, 5, 14, 14
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *workloads.index_constants())
    inp = workloads.irpe_inputs(B, heads, H * W, 64, nb, flags, "bf16", 1.0, seed=51)
    g = {k: (None if t is None else t.cuda()) for k, t in inp.items()}
    ids, K = oracle.product_bucket_ids(H, W, *workloads.index_constants())
    if bias:
        tab = workloads.bias_table(nb, heads, 2.0, seed=52)
        run = lambda: api.rpe_attn_bias_fwd(g["q"], g["k"], g["v"], tab.cuda(), lut, nb, H, W)  # noqa: E731
    else:
        tab = None
        run = lambda: api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags,  # noqa: E731
                                       table_k=g["tab_k"])
    out = run()
    S = B * heads
    sl = np.array([0, 151, 152, 170, S - 1])
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, flags, tab_k=inp["tab_k"],
                                    bias_in=None if tab is None else tab.numpy(), slices=sl)
    got = out.reshape(S, H * W, 64)[torch.as_tensor(sl, device=out.device)]
    assert _maxerr(got, ref.reshape(S, H * W, 64)[sl]) <= TOL_BF16
    assert torch.equal(run(), out)
