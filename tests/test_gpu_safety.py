"""GPU checks of the library's safety contracts, through the C ABI.

- Offset tables: a table that rpe_build_bucket_ids did not write is read back
  and checked on its first use; an id outside the table's range is refused
  before any launch. A checked table rewritten in place with a bad id is
  caught by the kernels, which set the status bit that rpe_device_status
  reports (no read leaves the tables meanwhile); so is a table rewritten so
  that its ids no longer form one run per grid row of keys, which the value
  term's bucket sums rely on.
- Split tail items: the two-warpgroup kernel merges split items through a
  workspace owned by the launching stream, so launches on two streams may
  overlap; a capture on a stream that has no workspace yet runs every item
  whole (no allocation inside a capture) and still matches the oracle.
- Shared-memory limits: a bf16 request whose offset table and bucket tables
  do not fit in shared memory returns RPE_ERR_UNSUPPORTED before any launch;
  the largest requests that fit match the oracle. The largest grid the calls
  take (256 x 256) runs in fp32 and is refused in bf16.
"""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_attention_gb300 import _lib, api, workloads
from vision_transformer_attention_gb300.workloads import FLAG_K, FLAG_Q, FLAG_V

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F32 = 1e-4
R19 = workloads.index_constants(1.9)
BAD_BUCKET_BIT = 1 << 5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.rpe_device_status(clear=True)
    yield
    assert api.rpe_device_status(clear=True) == 0


def _dev(d):
    return {k: (None if t is None else t.cuda()) for k, t in d.items()}


def _maxerr(gpu, ref):
    return float(np.max(np.abs(gpu.detach().float().cpu().numpy().astype(np.float64) - ref)))


@pytest.mark.parametrize("dtype,flags", [("bf16", FLAG_K), ("bf16", FLAG_Q | FLAG_K | FLAG_V),
                                         ("f32", FLAG_K)])
def test_table_with_a_bad_id_is_refused(dtype, flags):
    H = W = 14
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    inp = _dev(workloads.irpe_inputs(1, 2, H * W, 64, nb, flags, dtype, 1.0, seed=3))
    for bad in (nb, -1, 1000):
        custom = lut.clone()  # a table the library has not seen
        custom[(2 * W - 1) * 3 + 5] = bad
        with pytest.raises(_lib.RpeError) as e:
            api.rpe_attn_fwd(inp["q"], inp["k"], inp["v"], custom, nb, H, W, flags,
                             table_q=inp["tab_q"], table_k=inp["tab_k"], table_v=inp["tab_v"])
        assert e.value.status == _lib.RPE_ERR_INVALID_ARG
    # bias mode (any dtype) checks the same way
    custom = lut.clone()
    custom[0] = nb
    with pytest.raises(_lib.RpeError) as e:
        api.rpe_attn_bias_fwd(inp["q"], inp["k"], inp["v"],
                              workloads.bias_table(nb, 2, 1.0).cuda(), custom, nb, H, W)
    assert e.value.status == _lib.RPE_ERR_INVALID_ARG
    # a class token reserves the last bucket: a grid id equal to it is refused
    inp_c = _dev(workloads.irpe_inputs(1, 2, H * W + 1, 64, nb + 1, FLAG_K, dtype, 1.0, seed=4))
    with pytest.raises(_lib.RpeError) as e:
        api.rpe_attn_fwd(inp_c["q"], inp_c["k"], inp_c["v"], lut.clone(), nb, H, W, FLAG_K,
                         table_k=inp_c["tab_k"][:nb], cls_token=True)
    assert e.value.status == _lib.RPE_ERR_INVALID_ARG
    assert api.rpe_device_status(clear=True) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_valid_custom_table_is_accepted(dtype):
    H = W = 14
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    inp = _dev(workloads.irpe_inputs(2, 3, H * W, 64, nb, FLAG_K, dtype, 1.0, seed=5))
    ref = api.rpe_attn_fwd(inp["q"], inp["k"], inp["v"], lut, nb, H, W, FLAG_K,
                           table_k=inp["tab_k"])
    custom = lut.clone()
    for _ in range(2):  # checked on the first use, known afterwards
        out = api.rpe_attn_fwd(inp["q"], inp["k"], inp["v"], custom, nb, H, W, FLAG_K,
                               table_k=inp["tab_k"])
        assert torch.equal(out, ref)
    assert api.rpe_device_status(clear=True) == 0


@pytest.mark.parametrize("dtype,H,W", [("bf16", 14, 14), ("bf16", 9, 20), ("f32", 14, 14)])
def test_table_rewritten_in_place_sets_the_status_bit(dtype, H, W):
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    inp = _dev(workloads.irpe_inputs(1, 2, H * W, 64, nb, FLAG_K, dtype, 1.0, seed=6))
    assert api.rpe_device_status(clear=True) == 0
    lut[7] = nb + 3  # after the library recorded the table as valid
    out = api.rpe_attn_fwd(inp["q"], inp["k"], inp["v"], lut, nb, H, W, FLAG_K,
                           table_k=inp["tab_k"])
    status = api.rpe_device_status(clear=True)
    assert status & BAD_BUCKET_BIT
    assert bool(torch.isfinite(out.float()).all())
    assert api.rpe_device_status(clear=True) == 0


@pytest.mark.parametrize("flags", [FLAG_K | FLAG_V, FLAG_V])
def test_table_rewritten_without_row_runs_sets_the_status_bit(flags):
    # the value term's bucket sums need each id to form one run along a grid
    # row of keys; a Product table (recorded with that property) rewritten in
    # place with Euclidean ids -- in range, but repeating on both sides of a
    # query column -- is caught by the kernel
    H, W = 14, 14
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    eu, _, nbe = api.rpe_build_bucket_ids(H, W, *R19, mode=_lib.RPE_MAP_EUCLIDEAN)
    assert nbe <= nb
    inp = _dev(workloads.irpe_inputs(1, 2, H * W, 64, nb, flags, "bf16", 1.0, seed=8))
    run = lambda t: api.rpe_attn_fwd(inp["q"], inp["k"], inp["v"], t, nb, H, W, flags,  # noqa: E731
                                     table_k=inp["tab_k"], table_v=inp["tab_v"])
    assert api.rpe_device_status(clear=True) == 0
    lut.copy_(eu)
    out = run(lut)
    status = api.rpe_device_status(clear=True)
    assert status & BAD_BUCKET_BIT
    assert bool(torch.isfinite(out.float()).all())
    # the Euclidean table as the library built it is recorded without the
    # property: the request runs on the general kernel and raises nothing
    run(eu)
    assert api.rpe_device_status(clear=True) == 0


def _split_case(seed):
    # 40 x 5 = 200 slices of one item each on 152 SMs: the last 48 items run
    # as two parts on two CTAs each, merged through the stream's workspace
    B, heads, H, W = 40, 5, 14, 14
    inp = workloads.irpe_inputs(B, heads, H * W, 64, 49, FLAG_K, "bf16", 1.0, seed=seed)
    return (B, heads, H, W), inp


def _split_ref(inp, shape, sl):
    B, heads, H, W = shape
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    ref = oracle.irpe_attention_ids(inp["q"], inp["k"], inp["v"], ids, K, FLAG_K,
                                    tab_k=inp["tab_k"], slices=sl)
    return ref.reshape(B * heads, H * W, 64)[sl]


def test_split_tail_launches_on_two_streams_overlap_safely():
    shape, inp_a = _split_case(61)
    _, inp_b = _split_case(62)
    B, heads, H, W = shape
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    ga, gb = _dev(inp_a), _dev(inp_b)
    run = lambda g: api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, FLAG_K,  # noqa: E731
                                     table_k=g["tab_k"])
    ref_a, ref_b = run(ga), run(gb)  # one stream, in order
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs_a, outs_b = [], []
    for _ in range(3):  # first calls set up each stream's workspace
        with torch.cuda.stream(s1):
            outs_a.append(run(ga))
        with torch.cuda.stream(s2):
            outs_b.append(run(gb))
    torch.cuda.synchronize()
    for oa, ob in zip(outs_a, outs_b):
        assert torch.equal(oa, ref_a)
        assert torch.equal(ob, ref_b)
    S = B * heads
    sl = np.array([0, 151, 152, 170, S - 1])
    for inp, out in ((inp_a, ref_a), (inp_b, ref_b)):
        got = out.reshape(S, H * W, 64)[torch.as_tensor(sl, device=out.device)]
        assert _maxerr(got, _split_ref(inp, shape, sl)) <= TOL_BF16


def test_release_stream_and_shutdown_free_and_reallocate():
    # a stream's split-tail workspace can be freed and comes back on its next
    # split call; rpe_shutdown frees everything (status words included) and
    # forgets the recorded tables; results stay bit-identical throughout
    shape, inp = _split_case(seed=23)
    B, heads, H, W = shape
    g = _dev(inp)
    s = torch.cuda.Stream()

    def run():
        lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
        with torch.cuda.stream(s):
            out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, FLAG_K, table_k=g["tab_k"])
        s.synchronize()
        return out

    first = run()
    api.rpe_release_stream(s)
    api.rpe_release_stream(s)  # nothing left to free: still fine
    assert torch.equal(run(), first)
    api.rpe_shutdown()
    assert torch.equal(run(), first)
    assert api.rpe_device_status(clear=True) == 0
    sl = np.array([0, B * heads - 1])
    got = first.reshape(B * heads, H * W, 64)[torch.as_tensor(sl, device=first.device)]
    assert float((got.float().cpu() - torch.as_tensor(_split_ref(inp, shape, sl))).abs().max()) <= TOL_BF16


def test_capture_on_a_stream_without_workspace_runs_items_whole():
    shape, inp = _split_case(63)
    B, heads, H, W = shape
    lut, _, nb = api.rpe_build_bucket_ids(H, W, *R19)
    g = _dev(inp)
    out = torch.empty_like(g["q"])
    s = torch.cuda.Stream()  # never used eagerly: no workspace of its own
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, FLAG_K, table_k=g["tab_k"],
                         out=out)
    graph.replay()
    torch.cuda.synchronize()
    S = B * heads
    sl = np.array([0, 151, 152, 170, S - 1])
    got = out.reshape(S, H * W, 64)[torch.as_tensor(sl, device=out.device)]
    assert _maxerr(got, _split_ref(inp, shape, sl)) <= TOL_BF16


# bf16 requests keep the offset table and one query tile's bucket tables in
# shared memory: the largest request that fits runs and matches the oracle,
# one step beyond is refused before any launch (tables of `nb` rows; the
# Product ids of these grids use the first 49)
@pytest.mark.parametrize("flags,nb,H", [(FLAG_K, 64, 164), (FLAG_Q | FLAG_K | FLAG_V, 64, 78),
                                        (FLAG_K | FLAG_V, 110, 14)])
def test_largest_request_that_fits_in_shared_memory_matches_the_oracle(flags, nb, H):
    W = H
    N = H * W
    lut, _, K = api.rpe_build_bucket_ids(H, W, *R19)
    inp = workloads.irpe_inputs(1, 2, N, 64, nb, flags, "bf16", 0.5, seed=9)
    g = _dev(inp)
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags, table_q=g["tab_q"],
                           table_k=g["tab_k"], table_v=g["tab_v"])
    torch.cuda.synchronize()
    rows = np.array([0, 1, W - 1, W, N // 2, N - W, N - 1])
    tabs = {n: (None if inp[n] is None else inp[n][:K]) for n in ("tab_q", "tab_k", "tab_v")}
    ref = oracle.irpe_attention(inp["q"], inp["k"], inp["v"], H, W, *R19, flags, rows=rows, **tabs)
    got = out[:, :, torch.as_tensor(rows, device=out.device)]
    assert _maxerr(got, ref[:, :, rows]) <= TOL_BF16


@pytest.mark.parametrize("flags,nb,H", [(FLAG_K, 64, 165), (FLAG_Q | FLAG_K | FLAG_V, 64, 79),
                                        (FLAG_K | FLAG_V, 111, 14), (FLAG_K | FLAG_V, 128, 14)])
def test_request_beyond_shared_memory_is_unsupported(flags, nb, H):
    W = H
    lut, _, _ = api.rpe_build_bucket_ids(H, W, *R19)
    g = _dev(workloads.irpe_inputs(1, 1, H * W, 64, nb, flags, "bf16", 0.5, seed=5))
    out = torch.full_like(g["q"], 7.0)
    with pytest.raises(_lib.RpeError) as e:
        api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, nb, H, W, flags, table_q=g["tab_q"],
                         table_k=g["tab_k"], table_v=g["tab_v"], out=out)
    assert e.value.status == _lib.RPE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool(torch.all(out == 7.0))  # nothing was launched


def test_largest_grid_runs_in_fp32_and_is_refused_in_bf16():
    # N = 65536, the most the attention calls take: the library builds the
    # grid's offset table (no N x N map), fp32 matches the oracle on sampled
    # rows, and bf16, whose shared memory cannot hold the 511 x 511 table,
    # is refused before any launch
    H = W = 256
    N = H * W
    lut, _, K = api.rpe_build_bucket_ids(H, W, *R19)
    inp = workloads.irpe_inputs(1, 1, N, 32, K, FLAG_K, "f32", 2.0, seed=13)
    g = _dev(inp)
    out = api.rpe_attn_fwd(g["q"], g["k"], g["v"], lut, K, H, W, FLAG_K, table_k=g["tab_k"])
    torch.cuda.synchronize()
    rows = np.array([0, 1, W - 1, W, N // 2 + W // 2, N - W, N - 1])
    ref = oracle.irpe_attention(inp["q"], inp["k"], inp["v"], H, W, *R19, FLAG_K,
                                tab_k=inp["tab_k"], rows=rows)[:, :, rows]
    got = out[:, :, torch.as_tensor(rows, device=out.device)]
    assert _maxerr(got, ref) <= TOL_F32
    plain = oracle.irpe_attention(inp["q"], inp["k"], inp["v"], H, W, *R19, 0, rows=rows)[:, :, rows]
    assert np.max(np.abs(plain - ref)) > 100 * TOL_F32  # the key term matters here
    b = _dev(workloads.irpe_inputs(1, 1, N, 64, K, FLAG_K, "bf16", 0.5, seed=13))
    with pytest.raises(_lib.RpeError) as e:
        api.rpe_attn_fwd(b["q"], b["k"], b["v"], lut, K, H, W, FLAG_K, table_k=b["tab_k"])
    assert e.value.status == _lib.RPE_ERR_UNSUPPORTED
