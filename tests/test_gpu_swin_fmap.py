"""Swin window attention on channels-last feature maps (swin_window_attn_fwd_fmap)
against the oracle: the windows are cut out of the map on the CPU by the plain
partition of "Swin Transformer", section 3.2 (non-overlapping M x M windows),
attended by the oracle, and put back."""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_attention_gb300 import api, workloads
from vision_transformer_attention_gb300._lib import RpeError

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
M = 7


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert api.rpe_device_status(clear=True) == 0


def _run(batch, img_h, img_w, heads, d, table_std=0.02, seed=0):
    inp = workloads.swin_fmap_inputs(batch, img_h, img_w, heads, M, d, table_std, seed)
    g = {k: t.cuda() for k, t in inp.items()}
    out = api.swin_window_attn_fwd_fmap(g["q"], g["k"], g["v"], g["table"], M)
    return inp, g, out


def _oracle(inp, heads, windows=None):
    parts = [workloads.window_partition(inp[n], M, heads) for n in ("q", "k", "v")]
    return oracle.swin_attention(parts[0], parts[1], parts[2], inp["table"], M, slices=windows)


@pytest.mark.parametrize("batch,img_h,img_w,heads,d", [
    (1, 14, 14, 3, 32),   # 4 windows x 3 heads
    (1, 7, 21, 3, 32),    # 9 units: an odd last tile
    (2, 14, 7, 2, 64),
    (1, 7, 7, 1, 32),     # a single unit
])
@pytest.mark.parametrize("table_std", [0.02, 2.0])
def test_fmap_matches_oracle(batch, img_h, img_w, heads, d, table_std):
    inp, _, out = _run(batch, img_h, img_w, heads, d, table_std, seed=img_w + d)
    ref = _oracle(inp, heads)  # [windows, heads, 49, d], fp64
    ref_map = workloads.window_reverse(torch.from_numpy(ref), M, batch, img_h, img_w).numpy()
    err = np.max(np.abs(out.float().cpu().numpy().astype(np.float64) - ref_map))
    assert err <= TOL_BF16


def test_fmap_equals_partitioned_kernel():
    # same kernel arithmetic on the same windows: the results must be identical
    batch, img_h, img_w, heads, d = 2, 28, 21, 3, 32
    inp, g, out = _run(batch, img_h, img_w, heads, d, seed=5)
    parts = [workloads.window_partition(g[n], M, heads).contiguous() for n in ("q", "k", "v")]
    win = api.swin_window_attn_fwd(parts[0], parts[1], parts[2], g["table"], M)
    assert torch.equal(workloads.window_reverse(win, M, batch, img_h, img_w), out)


def test_fmap_swin_t_stage1_sampled():
    # Swin-T stage 1: batch 32, 56 x 56 map, 3 heads, d = 32
    batch, img_h, img_w, heads, d = 32, 56, 56, 3, 32
    inp, g, out = _run(batch, img_h, img_w, heads, d)
    parts = [workloads.window_partition(g[n], M, heads).contiguous() for n in ("q", "k", "v")]
    win = api.swin_window_attn_fwd(parts[0], parts[1], parts[2], g["table"], M)
    assert torch.equal(workloads.window_reverse(win, M, batch, img_h, img_w), out)
    nw = batch * (img_h // M) * (img_w // M)
    rng = np.random.default_rng(3)
    sl = np.unique(np.concatenate([rng.choice(nw * heads, 48, replace=False), [0, nw * heads - 1]]))
    ref = _oracle(inp, heads, windows=sl).reshape(nw * heads, 49, d)[sl]
    got = workloads.window_partition(out, M, heads).reshape(nw * heads, 49, d)[
        torch.as_tensor(sl, device=out.device)]
    assert float(np.max(np.abs(got.float().cpu().numpy() - ref))) <= TOL_BF16


def test_fmap_rejects_maps_not_tiled_by_windows():
    inp = workloads.swin_fmap_inputs(1, 14, 10, 3, M, 32)
    g = {k: t.cuda() for k, t in inp.items()}
    with pytest.raises(RpeError):
        api.swin_window_attn_fwd_fmap(g["q"], g["k"], g["v"], g["table"], M)
