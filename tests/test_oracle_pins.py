"""Pins for the oracle: values the pages print, closed forms, invariants and
library special cases. None of these re-types the oracle's own formulas; each
is a fact fixed by the pages or by the mathematics, chosen so that a dropped
term, a wrong sign or index, or a transposed operand in the oracle fails one.

Sources: "Rethinking and Improving Relative Position Encoding for Vision
Transformer" (eqs. 13-18, 25-28; Pitfalls), "Swin 的二维 RPE" (sections 2.2,
3.1-3.3), "Swin Transformer, section 3.2 and Table 4", and "Implementation:
Relative Position in Self-Attention" (Testing the Implementation).
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

R19 = (1.9, 3.8, 15.2)


# ---------------------------------------------------------------- eq. 18 g(x)

def test_piecewise_r19_matches_pitfalls_table():
    rows = read_golden("piecewise_r1p9.txt")
    alpha, beta, gamma = rows[0]
    for off, idx in rows[1:]:
        assert oracle.piecewise_index(off, alpha, beta, gamma) == int(idx), off
        assert oracle.piecewise_index(-off, alpha, beta, gamma) == -int(idx), off


def test_piecewise_r20_nine_buckets_and_shared_pair():
    rows = read_golden("piecewise_r2p0.txt")
    alpha, beta, gamma, span = rows[0]
    a, b = rows[1]
    assert 2 * int(beta) + 1 == int(span)
    assert oracle.piecewise_index(a, alpha, beta, gamma) == oracle.piecewise_index(
        b, alpha, beta, gamma)
    # the index range is exactly [-int(beta), int(beta)] over a long axis
    vals = {oracle.piecewise_index(x, alpha, beta, gamma) for x in range(-300, 301)}
    assert vals == set(range(-int(beta), int(beta) + 1))


@pytest.mark.parametrize("ratio", [1.0, 1.9, 2.0, 3.5, 7.0])
def test_piecewise_identity_below_alpha_and_odd(ratio):
    alpha, beta, gamma = ratio, 2 * ratio, 8 * ratio
    for x in range(0, int(np.floor(alpha)) + 1):  # exact for |x| <= alpha (eq. 18)
        assert oracle.piecewise_index(x, alpha, beta, gamma) == x
    prev = 0
    for x in range(0, 200):
        g = oracle.piecewise_index(x, alpha, beta, gamma)
        assert oracle.piecewise_index(-x, alpha, beta, gamma) == -g   # odd symmetry
        assert 0 <= g <= int(beta)                                      # capped at beta
        assert g >= prev                                                # monotone
        prev = g
    # at x = gamma the log share is exactly 1, so the spread is beta itself
    if float(gamma).is_integer() and float(beta).is_integer():
        assert oracle.piecewise_index(gamma, alpha, beta, gamma) == int(beta)
        assert oracle.piecewise_index(-gamma, alpha, beta, gamma) == -int(beta)


def test_product_table_has_fifty_entries_with_cls():
    # Pitfalls: "the Product table has 7 x 7 + 1 = 50 entries" at r = 1.9
    _, K = oracle.product_bucket_ids(14, 14, *R19)
    assert K + 1 == 50


# ---------------------------------------------------------------- eq. 25 ids

def test_product_ids_range_mirror_centre():
    H = W = 14
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    assert K == 49 and ids.shape == (196, 196)
    assert ids.min() == 0 and ids.max() == K - 1
    assert set(np.unique(ids)) == set(range(K))
    # g is odd, so swapping query and key mirrors the id: id(j,i) = K-1-id(i,j)
    assert np.array_equal(ids.T, K - 1 - ids)
    assert np.all(np.diag(ids) == (K - 1) // 2)


def test_product_ids_sign_and_axis_order():
    # Offsets are query minus key (Swin notes 3.2 worked example), row offset is the
    # major index (iRPE eq. 25 pseudocode: offsets[...,0] is the row).
    H = W = 14
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    span = 7
    at = lambda r, c: r * W + c  # noqa: E731
    # query (0,0), key (2,2): offset (-2,-2) -> indices (-2,-2) -> (1,1) after +3
    assert ids[at(0, 0), at(2, 2)] == 1 * span + 1
    # query (0,0), key (0,1): row 0 -> 3, col -1 -> 2
    assert ids[at(0, 0), at(0, 1)] == 3 * span + 2
    # query (0,0), key (1,0): row -1 -> 2, col 0 -> 3 (differs from the above: axes not swapped)
    assert ids[at(0, 0), at(1, 0)] == 2 * span + 3
    # far corner: offset (-13,-13) -> (-3,-3) -> id 0; reversed pair -> K-1
    assert ids[at(0, 0), at(13, 13)] == 0
    assert ids[at(13, 13), at(0, 0)] == K - 1


def test_product_ids_translation_invariant():
    # the id depends only on the offset between the two positions (Swin notes 2.2)
    H, W = 9, 11
    ids, _ = oracle.product_bucket_ids(H, W, *R19)
    seen = {}
    for i in range(H * W):
        for j in range(H * W):
            key = (i // W - j // W, i % W - j % W)
            assert seen.setdefault(key, ids[i, j]) == ids[i, j]


# ---------------------------------------------------------------- Swin index

def test_swin_worked_example_m3():
    for M, qr, qc, kr, kc, tr, tc in read_golden("swin_m3_example.txt"):
        M = int(M)
        idx, nb = oracle.swin_bias_index(M)
        side = 2 * M - 1
        assert nb == side * side == 25
        i, j = int(qr) * M + int(qc), int(kr) * M + int(kc)
        assert idx[i, j] == int(tr) * side + int(tc)


def test_swin_table_sizes():
    for M, brute, compact in read_golden("swin_table_sizes.txt"):
        M = int(M)
        idx, nb = oracle.swin_bias_index(M)
        assert nb == int(compact)
        assert idx.size == int(brute)                 # one entry per pair: M^2 x M^2
        assert len(np.unique(idx)) == int(compact)    # every table entry is used


def test_swin_index_translation_invariant_and_centre():
    M = 7
    idx, nb = oracle.swin_bias_index(M)
    for i in range(M * M):
        for j in range(M * M):
            dr, dc = i // M - j // M, i % M - j % M
            # shifted offsets land in [0, 2M-2] on both axes
            assert 0 <= idx[i, j] // (2 * M - 1) <= 2 * M - 2
            assert idx[i, j] == idx[(i // M) * M + i % M, j]
            if dr == 0 and dc == 0:
                assert idx[i, j] == (M - 1) * (2 * M - 1) + (M - 1) == 84


# ---------------------------------------------------------------- Shaw clip + printed weights

def test_clip_ids_shift():
    k = 3
    ids = oracle.clip_ids_1d(6, k)
    assert ids[0, 0] == k          # offset 0 -> index k
    assert ids[5, 0] == 0          # offset -5 clipped to -k -> 0
    assert ids[0, 5] == 2 * k      # offset +5 clipped to +k -> 2k
    assert ids[2, 1] == k - 1 and ids[1, 2] == k + 1


def _shaw_inputs():
    rs = np.random  # the page's example uses numpy's legacy seeded generator
    rs.seed(42)
    X = rs.randn(6, 8)
    rs.seed(123)
    s_qk = np.sqrt(2.0 / (8 + 4))
    Wq, Wk, Wv = rs.randn(8, 4) * s_qk, rs.randn(8, 4) * s_qk, rs.randn(8, 4) * s_qk
    rs.seed(123)
    s_tab = np.sqrt(2.0 / (7 + 4))
    aK = rs.randn(7, 4) * s_tab
    aV = rs.randn(7, 4) * s_tab
    return X @ Wq, X @ Wk, X @ Wv, aK, aV


def test_shaw_printed_attention_weights():
    Q, K, V, aK, aV = _shaw_inputs()
    ids = oracle.clip_ids_1d(6, 3)
    out, attn = oracle.attention(Q, K, V, ids, 7, tab_k=aK, tab_v=aV, want_attn=True)
    printed = np.array(read_golden("shaw_weights_6x6.txt"))
    assert np.max(np.abs(attn - printed)) <= 5e-4 + 1e-12
    assert np.allclose(attn.sum(axis=1), 1.0, atol=1e-12)
    # the position term matters here: without it the weights are far off
    _, plain = oracle.attention(Q, K, V, ids, 7, want_attn=True)
    assert np.max(np.abs(plain - printed)) > 1e-2


# ---------------------------------------------------------------- attention special cases

def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]  # noqa: E731
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v))[0, 0].numpy()


def test_zero_tables_equal_library_sdpa():
    H, W, d = 5, 6, 16
    n = H * W
    q, k, v = _rand((n, d), 1), _rand((n, d), 2), _rand((n, d), 3)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    z = np.zeros((K, d))
    out = oracle.attention(q, k, v, ids, K, tab_k=z, tab_q=z, tab_v=z, bias=np.zeros(K))
    assert np.max(np.abs(out - _sdpa(q, k, v))) < 1e-12


def test_constant_key_table_is_softmax_shift():
    # q.(k_j + c) = q.k_j + q.c: a per-row constant, which softmax removes
    H, W, d = 4, 5, 8
    n = H * W
    q, k, v = _rand((n, d), 4), _rand((n, d), 5), _rand((n, d), 6)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    c = _rand((d,), 7)
    out = oracle.attention(q, k, v, ids, K, tab_k=np.tile(c, (K, 1)))
    assert np.max(np.abs(out - _sdpa(q, k, v))) < 1e-12


def test_constant_query_table_is_query_shift():
    # k_j.c is added to logit (i,j): (q_i + c).k_j -- attention with q shifted by c.
    # A transposed operand (q_i.c) would instead leave the output unchanged.
    H, W, d = 4, 5, 8
    n = H * W
    q, k, v = _rand((n, d), 8), _rand((n, d), 9), _rand((n, d), 10)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    c = _rand((d,), 11)
    out = oracle.attention(q, k, v, ids, K, tab_q=np.tile(c, (K, 1)))
    assert np.max(np.abs(out - _sdpa(q + c, k, v))) < 1e-12
    assert np.max(np.abs(out - _sdpa(q, k, v))) > 1e-3


def test_constant_value_table_adds_constant():
    # sum_j a_ij = 1, so a value table with every row c adds exactly c (eq. 17)
    H, W, d = 4, 5, 8
    n = H * W
    q, k, v = _rand((n, d), 12), _rand((n, d), 13), _rand((n, d), 14)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    c = _rand((d,), 15)
    out = oracle.attention(q, k, v, ids, K, tab_v=np.tile(c, (K, 1)))
    assert np.max(np.abs(out - (_sdpa(q, k, v) + c))) < 1e-12


def test_hard_bias_selects_one_neighbour_and_its_value_entry():
    # A bias of -1e4 on every bucket but one forces each query onto the key at that
    # offset. With offset (0,+1) in query-minus-key terms the chosen key is the left
    # neighbour (same row, column - 1); the value term then adds R^V at that bucket.
    H = W = 6
    n, d = H * W, 8
    q, k, v = 0.1 * _rand((n, d), 16), 0.1 * _rand((n, d), 17), _rand((n, d), 18)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    target = (0 + 3) * 7 + (1 + 3)  # row offset 0, column offset +1
    bias = np.full(K, -1e4)
    bias[target] = 0.0
    tv = _rand((K, d), 19)
    out = oracle.attention(q, k, v, ids, K, tab_v=tv, bias=bias)
    for i in range(n):
        r, c = divmod(i, W)
        if c >= 1:
            assert np.allclose(out[i], v[i - 1] + tv[target], atol=1e-9)


def test_efficient_form_equals_per_pair():
    # eqs. 26-28 re-associate the same sums: QR / KR gathers and per-bucket sums
    H, W, d = 6, 7, 16
    n = H * W
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    q, k, v = _rand((n, d), 20), _rand((n, d), 21), _rand((n, d), 22)
    tk, tq, tv = _rand((K, d), 23), _rand((K, d), 24), _rand((K, d), 25)
    bias = _rand((K,), 26)
    a = oracle.attention(q, k, v, ids, K, tab_k=tk, tab_q=tq, tab_v=tv, bias=bias)
    b = oracle.attention_efficient(q, k, v, ids, K, tab_k=tk, tab_q=tq, tab_v=tv, bias=bias)
    assert np.max(np.abs(a - b)) < 1e-12


def test_swin_constant_table_and_self_mask():
    M, d, heads = 7, 32, 3
    n = M * M
    q, k, v = (_rand((2, heads, n, d), s) for s in (27, 28, 29))
    zero = oracle.swin_attention(q, k, v, np.zeros(((2 * M - 1) ** 2, heads)), M)
    for w in range(2):
        for h in range(heads):
            assert np.max(np.abs(zero[w, h] - _sdpa(q[w, h], k[w, h], v[w, h]))) < 1e-12
    const = oracle.swin_attention(q, k, v, np.full(((2 * M - 1) ** 2, heads), 0.7), M)
    assert np.max(np.abs(const - zero)) < 1e-12
    mask = np.full(((2 * M - 1) ** 2, heads), -1e4)
    mask[(M - 1) * (2 * M - 1) + (M - 1), :] = 0.0     # only offset (0,0) survives
    self_only = oracle.swin_attention(0.1 * q, 0.1 * k, v, mask, M)
    assert np.max(np.abs(self_only - v)) < 1e-9


def test_swin_bias_is_added_after_scaling():
    # with q = k = 0 the logits are the bias alone, so weights are softmax(B[i, :])
    M, d = 3, 4
    n = M * M
    z = np.zeros((1, 1, n, d))
    v = _rand((1, 1, n, d), 30)
    table = _rand(((2 * M - 1) ** 2, 1), 31) * 2.0
    out = oracle.swin_attention(z, z, v, table, M)
    idx, _ = oracle.swin_bias_index(M)
    B = table[idx, 0]
    a = np.exp(B - B.max(axis=1, keepdims=True))
    a /= a.sum(axis=1, keepdims=True)
    assert np.max(np.abs(out[0, 0] - a @ v[0, 0])) < 1e-12


def test_irpe_batched_matches_slices_and_rows():
    H, W, d = 4, 4, 8
    n = H * W
    B, heads = 2, 3
    q, k, v = (_rand((B, heads, n, d), s) for s in (32, 33, 34))
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    tk, tq, tv = (_rand((K, d), s) for s in (35, 36, 37))
    full = oracle.irpe_attention(q, k, v, H, W, *R19, 7, tab_q=tq, tab_k=tk, tab_v=tv)
    for b in range(B):
        for h in range(heads):
            one = oracle.attention(q[b, h], k[b, h], v[b, h], ids, K, tab_k=tk, tab_q=tq,
                                   tab_v=tv)
            assert np.array_equal(one, full[b, h])
    part = oracle.irpe_attention(q, k, v, H, W, *R19, 7, tab_q=tq, tab_k=tk, tab_v=tv,
                                 slices=[4], rows=[0, 5, 15])
    assert np.array_equal(part[1, 1, [0, 5, 15]], full[1, 1, [0, 5, 15]])
    assert np.all(part[0] == 0)


def test_stress_tables_move_output_beyond_tolerance():
    # negative control: at std 1.0 the position term changes outputs by far more
    # than the 2e-2 bf16 tolerance, so a kernel that drops a term cannot pass
    H = W = 14
    d = 64
    n = H * W
    q, k, v = (_rand((1, 1, n, d), s) for s in (38, 39, 40))
    _, K = oracle.product_bucket_ids(H, W, *R19)
    for flag, name in ((1, "tab_k"), (2, "tab_q"), (4, "tab_v")):
        tab = _rand((K, d), 41)
        with_term = oracle.irpe_attention(q, k, v, H, W, *R19, flag, **{name: tab})
        without = oracle.irpe_attention(q, k, v, H, W, *R19, 0)
        assert np.max(np.abs(with_term - without)) > 0.2, name
    M = 7
    qs, ks, vs = (_rand((1, 3, 49, 32), s) for s in (42, 43, 44))
    t = 2.0 * _rand((169, 3), 45)
    assert np.max(np.abs(oracle.swin_attention(qs, ks, vs, t, M)
                         - oracle.swin_attention(qs, ks, vs, 0 * t, M))) > 0.2


# ------------------------------------------------------------ Euclidean mapping

def test_euclidean_axis_offsets_follow_the_1d_index():
    # on one axis the distance is the offset's length, so the Euclidean index is
    # the printed piecewise index of |offset| (shifted by int(beta))
    rows = read_golden("piecewise_r1p9.txt")
    alpha, beta, gamma = rows[0]
    half = int(beta)
    for H, W in ((1, 56), (56, 1)):
        ids, K = oracle.euclidean_bucket_ids(H, W, alpha, beta, gamma)
        assert K == 2 * half + 1
        for off, idx in rows[1:]:
            off = int(off)
            if off < max(H, W):
                assert ids[0, off] - half == int(idx), (H, W, off)
                assert ids[off, 0] - half == int(idx), (H, W, off)


def test_euclidean_ids_are_undirected_and_axis_symmetric():
    H, W = 6, 9
    ids, K = oracle.euclidean_bucket_ids(H, W, *R19)
    assert np.array_equal(ids, ids.T)          # offset and its negation share a bucket
    tr, _ = oracle.euclidean_bucket_ids(W, H, *R19)
    for i in range(H * W):
        for j in range(H * W):
            ri, ci, rj, cj = i // W, i % W, j // W, j % W
            # the same pair with rows and columns swapped
            assert tr[ci * H + ri, cj * H + rj] == ids[i, j]
    assert ids.min() >= int(R19[1]) and ids.max() < K   # indices of distances are >= 0


def test_euclidean_pythagorean_offsets_hit_exact_distances():
    rows = dict((int(o), int(i)) for o, i in read_golden("piecewise_r1p9.txt")[1:])
    H, W = 9, 9
    ids, _ = oracle.euclidean_bucket_ids(H, W, *R19)
    half = int(R19[1])
    for dr, dc, dist in ((3, 4, 5), (4, 3, 5), (6, 8, 10), (8, 6, 10), (0, 7, 7)):
        i, j = dr * W + dc, 0  # query at (dr, dc), key at (0, 0)
        assert ids[i, j] - half == rows[dist]


# ------------------------------------------------------------ bias mode (eq. 14)

def test_constant_bias_mode_table_is_a_softmax_shift():
    H, W, d = 4, 5, 8
    n = H * W
    q, k, v = _rand((n, d), 40), _rand((n, d), 41), _rand((n, d), 42)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    out = oracle.attention(q, k, v, ids, K, bias_in=np.full(K, 3.7))
    assert np.max(np.abs(out - _sdpa(q, k, v))) < 1e-12


def test_bias_mode_is_added_inside_the_scaling():
    # b inside the 1/sqrt(d) scaling equals b / sqrt(d) added after it (the
    # pinned Swin placement); b added after would differ by the factor sqrt(d)
    H, W, d = 4, 5, 16
    n = H * W
    q, k, v = _rand((n, d), 43), _rand((n, d), 44), _rand((n, d), 45)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    b = 3.0 * _rand((K,), 46)
    inside = oracle.attention(q, k, v, ids, K, bias_in=b)
    after = oracle.attention(q, k, v, ids, K, bias=b / np.sqrt(d))
    assert np.max(np.abs(inside - after)) < 1e-12
    wrong = oracle.attention(q, k, v, ids, K, bias=b)
    assert np.max(np.abs(inside - wrong)) > 1e-3


def test_hard_bias_mode_picks_the_keys_of_one_bucket():
    # q = k = 0: the logits are the bias alone, so with a large bias on bucket b0
    # (zero elsewhere) each query averages v over the keys in that bucket
    H, W, d = 5, 5, 4
    n = H * W
    z = np.zeros((n, d))
    v = _rand((n, d), 47)
    ids, K = oracle.euclidean_bucket_ids(H, W, *R19)
    b0 = int(R19[1]) + 1  # distance 1: the four axis neighbours
    bias = np.zeros(K)
    bias[b0] = 60.0 * np.sqrt(d)  # 60 after the scaling: other keys weigh ~e^-60
    out = oracle.attention(z, z, v, ids, K, bias_in=bias)
    for i in range(n):
        sel = ids[i] == b0
        assert sel.sum() >= 2
        assert np.allclose(out[i], v[sel].mean(axis=0), atol=1e-12)


def test_irpe_attention_ids_matches_per_slice_calls():
    B, heads, H, W, d = 2, 3, 4, 5, 8
    n = H * W
    q, k, v = (_rand((B, heads, n, d), s) for s in (50, 51, 52))
    ids, K = oracle.euclidean_bucket_ids(H, W, *R19)
    tk = _rand((K, d), 53)
    bias = _rand((K, heads), 54)
    out = oracle.irpe_attention_ids(q, k, v, ids, K, 1, tab_k=tk, bias_in=bias)
    for b in range(B):
        for h in range(heads):
            ref = oracle.attention(q[b, h], k[b, h], v[b, h], ids, K, tab_k=tk, bias_in=bias[:, h])
            assert np.max(np.abs(out[b, h] - ref)) < 1e-12
    shared = oracle.irpe_attention_ids(q, k, v, ids, K, 0, bias_in=bias[:, 1])
    ref = oracle.attention(q[1, 2], k[1, 2], v[1, 2], ids, K, bias_in=bias[:, 1])
    assert np.max(np.abs(shared[1, 2] - ref)) < 1e-12


# ------------------------------------------------------------ Cross mapping (eqs. 22-24)

def test_cross_ids_are_the_printed_axis_indices():
    # a row bucket is g(row offset) alone and a column bucket g(column offset)
    # alone; 2 x (2 beta + 1) buckets (section 3.2), row buckets first
    rows = read_golden("piecewise_r1p9.txt")
    alpha, beta, gamma = rows[0]
    half = int(beta)
    span = 2 * half + 1
    g = dict((int(o), int(i)) for o, i in rows[1:])
    H, W = 9, 12
    ids_row, ids_col, K = oracle.cross_bucket_ids(H, W, alpha, beta, gamma)
    assert K == 2 * span == 14
    for i in range(H * W):
        for j in range(H * W):
            dr, dc = i // W - j // W, i % W - j % W
            assert ids_row[i, j] == half + (g[dr] if dr >= 0 else -g[-dr])
            assert ids_col[i, j] == span + half + (g[dc] if dc >= 0 else -g[-dc])


def test_cross_and_product_share_their_axis_indices():
    # eq. 25 pairs the same two axis buckets that eqs. 22-24 add
    H, W = 7, 11
    ids_row, ids_col, K = oracle.cross_bucket_ids(H, W, *R19)
    prod, Kp = oracle.product_bucket_ids(H, W, *R19)
    span = K // 2
    assert Kp == span * span
    assert np.array_equal(prod, ids_row * span + (ids_col - span))


def test_cross_terms_are_added():
    # contextual K, Q, V and bias mode at once: the Cross result equals the
    # Product result with the joint table T[a span + b] = R[a] + R[span + b]
    # (encodings added); zeroing one half leaves the other half's single-id
    # result, so a dropped row or column term fails
    H, W, d = 4, 6, 8
    n = H * W
    q, k, v = _rand((n, d), 60), _rand((n, d), 61), _rand((n, d), 62)
    ids_row, ids_col, K = oracle.cross_bucket_ids(H, W, *R19)
    prod, Kp = oracle.product_bucket_ids(H, W, *R19)
    span = K // 2
    tk, tq, tv, bi = _rand((K, d), 63), _rand((K, d), 64), _rand((K, d), 65), _rand((K,), 66)
    cross = oracle.attention(q, k, v, ids_row, K, tab_k=tk, tab_q=tq, tab_v=tv, bias_in=bi,
                             ids2=ids_col)
    a, b = np.divmod(np.arange(Kp), span)

    def joint(t):
        return t[a] + t[span + b]

    ref = oracle.attention(q, k, v, prod, Kp, tab_k=joint(tk), tab_q=joint(tq), tab_v=joint(tv),
                           bias_in=joint(bi))
    assert np.max(np.abs(cross - ref)) < 1e-12
    for keep in (slice(0, span), slice(span, K)):
        m = np.zeros((K, 1))
        m[keep] = 1
        only = oracle.attention(q, k, v, ids_row, K, tab_k=tk * m, tab_q=tq * m, tab_v=tv * m,
                                bias_in=bi * m[:, 0], ids2=ids_col)
        single = ids_row if keep.start == 0 else ids_col
        ref1 = oracle.attention(q, k, v, single, K, tab_k=tk * m, tab_q=tq * m, tab_v=tv * m,
                                bias_in=bi * m[:, 0])
        assert np.max(np.abs(only - ref1)) < 1e-12
    assert np.max(np.abs(cross - oracle.attention(q, k, v, ids_row, K, tab_k=tk, tab_q=tq,
                                                  tab_v=tv, bias_in=bi))) > 1e-2


def test_cross_hard_bias_picks_the_left_neighbour():
    # q = k = 0; a large bias on row bucket "row offset 0" and on column bucket
    # "column offset +1" (query minus key): only the key one column to the left
    # gets both, so each query with a left neighbour returns that key's v
    H, W, d = 4, 5, 4
    n = H * W
    z = np.zeros((n, d))
    v = _rand((n, d), 67)
    ids_row, ids_col, K = oracle.cross_bucket_ids(H, W, *R19)
    half, span = int(R19[1]), K // 2
    bias = np.zeros(K)
    bias[half + 0] = 40.0 * np.sqrt(d)
    bias[span + half + 1] = 40.0 * np.sqrt(d)
    out = oracle.attention(z, z, v, ids_row, K, bias_in=bias, ids2=ids_col)
    for i in range(n):
        if i % W > 0:
            assert np.allclose(out[i], v[i - 1], atol=1e-12), i


# ------------------------------------------------------------ clip index (table 3)

def test_clip_product_on_one_row_is_shaws_1d_clip():
    # on a 1 x n grid only the column index varies; it is the pinned Shaw clip
    # of the offset with the opposite sign (Shaw clips key minus query)
    n, k = 11, 3
    span = 2 * k + 1
    ids, K = oracle.clip_product_bucket_ids(1, n, k)
    assert K == span * span == 49   # table 3: 50 buckets with the class token
    shaw = oracle.clip_ids_1d(n, k)
    assert np.array_equal(ids, k * span + (2 * k - shaw))


def test_clip_and_piecewise_agree_up_to_their_first_difference():
    # g is exact up to alpha and g(2) = 2 at r = 1.9, so the two index functions
    # agree while both axis offsets are within 2; at 3 the piecewise index
    # still says 2 (the Pitfalls list) where the clip says 3
    H, W = 9, 9
    clip, _ = oracle.clip_product_bucket_ids(H, W, 3)
    pw, _ = oracle.product_bucket_ids(H, W, *R19)
    for i in range(H * W):
        for j in range(H * W):
            dr, dc = abs(i // W - j // W), abs(i % W - j % W)
            if max(dr, dc) <= 2:
                assert clip[i, j] == pw[i, j]
            elif max(dr, dc) == 3:
                assert clip[i, j] != pw[i, j]


def test_clip_product_is_translation_invariant_and_saturates():
    H, W, k = 8, 10, 2
    ids, K = oracle.clip_product_bucket_ids(H, W, k)
    span = 2 * k + 1
    assert set(np.unique(ids)) == set(range(K))
    # (0, 0) attending every key at row offset <= -k, column offset <= -k: the corner bucket
    far = [j for j in range(H * W) if j // W >= k and j % W >= k]
    assert all(ids[0, j] == 0 for j in far)
    # pairs with equal offsets share a bucket wherever they sit on the grid
    seen = {}
    for i in range(H * W):
        for j in range(H * W):
            off = (i // W - j // W, i % W - j % W)
            assert seen.setdefault(off, ids[i, j]) == ids[i, j]
    # query (3, 4) vs key (1, 5): offsets (2, -1) -> ((2+k) span + (-1+k))
    assert ids[3 * W + 4, 1 * W + 5] == (2 + k) * span + (-1 + k)


# ------------------------------------------------------------ per-head tables (section 4.2)

def test_per_head_tables_serve_their_own_head():
    # head h of every batch reads table h: each slice equals the pinned one-table
    # attention with that head's tables, and heads given different tables differ
    B, heads, H, W, d = 2, 3, 4, 5, 8
    n = H * W
    q, k, v = (_rand((B, heads, n, d), s) for s in (70, 71, 72))
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    tk, tq, tv = (_rand((heads, K, d), s) for s in (73, 74, 75))
    out = oracle.irpe_attention_ids(q, k, v, ids, K, 7, tab_q=tq, tab_k=tk, tab_v=tv)
    for b in range(B):
        for h in range(heads):
            ref = oracle.attention(q[b, h], k[b, h], v[b, h], ids, K, tab_k=tk[h], tab_q=tq[h],
                                   tab_v=tv[h])
            assert np.max(np.abs(out[b, h] - ref)) < 1e-12
            if h > 0:
                other = oracle.attention(q[b, h], k[b, h], v[b, h], ids, K, tab_k=tk[0],
                                         tab_q=tq[0], tab_v=tv[0])
                assert np.max(np.abs(out[b, h] - other)) > 1e-2
    # one table repeated per head is the shared table
    shared = oracle.irpe_attention_ids(q, k, v, ids, K, 7, tab_q=tq[1], tab_k=tk[1], tab_v=tv[1])
    rep = oracle.irpe_attention_ids(q, k, v, ids, K, 7, tab_q=np.stack([tq[1]] * heads),
                                    tab_k=np.stack([tk[1]] * heads), tab_v=np.stack([tv[1]] * heads))
    assert np.max(np.abs(shared - rep)) < 1e-12


# ------------------------------------------------------------ class-token bucket (section 4.1)

def test_cls_bucket_count_is_the_pages_fifty():
    # Pitfalls and table 3: 7 x 7 Product buckets plus one for the class token
    H, W = 14, 14
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    cls, K1 = oracle.add_cls_bucket(ids, K)
    assert (K, K1) == (49, 50)
    assert cls.shape == (H * W + 1, H * W + 1)
    assert np.all(cls[0] == 49) and np.all(cls[:, 0] == 49)
    assert np.array_equal(cls[1:, 1:], ids)


def test_cls_hard_bias_routes_every_patch_to_the_class_token():
    # q = k = 0 and a large bias on the class bucket: each patch query sees one
    # key in that bucket (token 0) and returns v_0; the class query has every
    # pair in that bucket, so its logits are equal and it averages all of v
    H, W, d = 3, 4, 4
    n = H * W + 1
    z = np.zeros((n, d))
    v = _rand((n, d), 80)
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    cls, K1 = oracle.add_cls_bucket(ids, K)
    bias = np.zeros(K1)
    bias[K] = 50.0 * np.sqrt(d)
    out = oracle.attention(z, z, v, cls, K1, bias_in=bias)
    assert np.allclose(out[1:], v[0], atol=1e-12)
    assert np.allclose(out[0], v.mean(axis=0), atol=1e-12)


def test_cls_suppressed_leaves_the_patch_attention():
    # a -1e4 logit on the class bucket removes key 0 for every patch query, whose
    # result is then the patch-only attention with the same tables
    H, W, d = 4, 5, 8
    n = H * W
    q, k, v = (_rand((n + 1, d), s) for s in (81, 82, 83))
    ids, K = oracle.product_bucket_ids(H, W, *R19)
    cls, K1 = oracle.add_cls_bucket(ids, K)
    tk, tv = _rand((K1, d), 84), _rand((K1, d), 85)
    bias = np.zeros(K1)
    bias[K] = -1e4 * np.sqrt(d)
    full = oracle.attention(q, k, v, cls, K1, tab_k=tk, tab_v=tv, bias_in=bias)
    patch = oracle.attention(q[1:], k[1:], v[1:], ids, K, tab_k=tk[:K], tab_v=tv[:K])
    assert np.max(np.abs(full[1:] - patch)) < 1e-12
