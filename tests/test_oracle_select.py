"""Pins for the oracle's pooling, block scores, top-k and sparse attention.

Pooling: equal keys pool to that key, small integers give their exact mean,
and the bf16 rounding of a mean lands where round-to-nearest-even puts it
(hand-worked values).  Scores: one-hot indexer queries read a pooled
element exactly, and random scores stay inside the float32 recursive-sum
error bound of the exact dot product.  Top-k: brute force by full sort on
small rows, planted ties, k above the block count.  Sparse attention: taking
every block reduces to dense attention over those positions.
"""
import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import synth

DI = 128


def bf(x):
    f = np.asarray(x, np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), f)
    return b


def widen(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ik_cache(orc, ik, ptok=8, paged=True):
    T = ik.shape[0]
    shape = orc.Shape(1, 1, 256, DI)
    if paged:
        n = synth.pages_for(T, ptok)
        ps = orc.page_elems(shape, ptok)
        c = orc.paged(shape, np.zeros((n + 1) * ps, np.uint16), ptok,
                      synth.reversed_table(n, first=1))
    else:
        c = orc.contiguous(shape, -(-T // 4) * 4)
    orc.put_rows(shape, c, 0, orc.IK, 0, ik)
    return shape, c


def _pooled(orc, ik, block_values):
    shape, c = _ik_cache(orc, bf(ik))
    nb = ik.shape[0] // 4
    orc.pool(shape, c, 0, 0, nb)
    return widen(orc.get_rows(shape, c, 0, orc.P, 0, nb))


def test_pool_of_equal_keys_is_that_key(orc):
    row = widen(synth.normal_bf16(1, (DI,))).astype(np.float32)
    got = _pooled(orc, np.tile(row, (8, 1)), None)
    assert np.array_equal(got[0], row) and np.array_equal(got[1], row)


def test_pool_of_small_integers_is_exact_mean(orc):
    ik = np.zeros((4, DI), np.float32)
    ik[:, 0] = [1, 2, 3, 6]          # mean 3
    ik[:, 1] = [-7, 1, 1, 1]         # mean -1
    ik[:, 2] = [0.5, 0.25, 0.25, 1]  # mean 0.5
    got = _pooled(orc, ik, None)[0]
    assert got[:3].tolist() == [3.0, -1.0, 0.5] and (got[3:] == 0).all()


def test_pool_rounds_mean_to_nearest_even_bf16(orc):
    # bf16 keeps 7 fraction bits: the spacing above 1.0 is 2**-7.
    ulp = 2.0 ** -7
    ik = np.zeros((4, DI), np.float32)
    ik[:, 0] = [1, 1, 1, 1 + 4 * ulp / 4]        # mean 1 + ulp/4        -> 1
    ik[:, 1] = [1, 1, 1 + ulp, 1 + ulp]          # mean 1 + ulp/2 (tie)  -> 1 (even)
    ik[:, 2] = [1 + ulp, 1 + ulp, 1 + 2 * ulp, 1 + 2 * ulp]  # 1 + 1.5 ulp (tie) -> 1 + 2 ulp
    ik[:, 3] = [1, 1 + ulp, 1 + ulp, 1 + ulp]    # 1 + 0.75 ulp         -> 1 + ulp
    got = _pooled(orc, ik, None)[0]
    assert got[:4].tolist() == [1.0, 1.0, 1 + 2 * ulp, 1 + ulp]


def test_pool_within_half_ulp_of_exact_mean(orc):
    ik = synth.normal_bf16(2, (64, DI))
    shape, c = _ik_cache(orc, ik, ptok=16)
    orc.pool(shape, c, 0, 0, 16)
    got = widen(orc.get_rows(shape, c, 0, orc.P, 0, 16))
    exact = widen(ik).reshape(16, 4, DI).mean(axis=1)
    # half a bf16 ulp of the binade of the mean (7 fraction bits) plus the
    # float32 summation error of four terms
    half_ulp = 2.0 ** (np.floor(np.log2(np.abs(exact) + 1e-300)) - 8)
    sum_err = 4 * 2.0 ** -24 * np.abs(widen(ik)).reshape(16, 4, DI).sum(1) / 4
    assert (np.abs(got - exact) <= half_ulp + sum_err).all()
    # and never a whole ulp away
    assert (np.abs(got - exact) < 2 * half_ulp + sum_err).all()


def test_pool_paged_equals_contiguous(orc):
    ik = synth.normal_bf16(3, (96, DI))
    res = []
    for paged in (True, False):
        shape, c = _ik_cache(orc, ik, ptok=12, paged=paged)
        orc.pool(shape, c, 0, 0, 24)
        res.append(orc.get_rows(shape, c, 0, orc.P, 0, 24))
    assert np.array_equal(res[0], res[1])


def _scores(orc, ik, qi, T):
    shape, c = _ik_cache(orc, ik, ptok=16)
    orc.pool(shape, c, 0, 0, T // 4)
    pooled = orc.get_rows(shape, c, 0, orc.P, 0, T // 4)
    return orc.scores(shape, c, 0, qi.shape[0], T, qi), pooled


def test_one_hot_indexer_query_reads_a_pooled_element(orc):
    T = 64
    ik = synth.normal_bf16(4, (T, DI))
    qi = np.zeros((3, DI), np.float32)
    qi[0, 0] = 1; qi[1, 77] = 1; qi[2, 127] = -2
    s, pooled = _scores(orc, ik, bf(qi), T)
    p = widen(pooled)
    assert np.array_equal(s[0], p[:, 0].astype(np.float32))
    assert np.array_equal(s[1], p[:, 77].astype(np.float32))
    assert np.array_equal(s[2], (-2 * p[:, 127]).astype(np.float32))


def test_scores_within_float32_sum_bound(orc):
    T = 400
    ik = synth.normal_bf16(5, (T, DI))
    qi = synth.normal_bf16(6, (16, DI))
    s, pooled = _scores(orc, ik, qi, T)
    q, p = widen(qi), widen(pooled)
    exact = q @ p.T
    gamma = DI * 2.0 ** -24 / (1 - DI * 2.0 ** -24)
    bound = gamma * (np.abs(q) @ np.abs(p).T)
    assert (np.abs(s - exact) <= bound).all()
    assert s.shape == (16, T // 4)


def test_partial_trailing_block_is_not_scored(orc):
    ik = synth.normal_bf16(7, (23, DI))
    shape, c = _ik_cache(orc, ik, ptok=8)
    assert orc.scores(shape, c, 0, 2, 23, synth.normal_bf16(8, (2, DI))).shape == (2, 5)


def _brute_topk(row, k):
    order = sorted(range(row.size), key=lambda b: (-float(row[b]), b))[:k]
    return sorted(order) + [-1] * (k - min(k, row.size))


@pytest.mark.parametrize("nb,k", [(1, 1), (7, 3), (64, 64), (50, 64), (63, 8), (64, 1)])
def test_topk_matches_full_sort(orc, nb, k):
    rng = np.random.default_rng(nb * 100 + k)
    s = rng.standard_normal((5, nb)).astype(np.float32)
    s[1] = np.round(s[1])            # many exact ties
    got = orc.topk(s, k)
    for r in range(5):
        assert got[r].tolist() == _brute_topk(s[r], k)


def test_topk_ties_go_to_lower_ids_and_signed_zeros_tie(orc):
    s = np.array([[0.0, 5.0, -0.0, 5.0, 1.0, 0.0, 5.0]], np.float32)
    assert orc.topk(s, 2).tolist() == [[1, 3]]
    assert orc.topk(s, 4).tolist() == [[1, 3, 4, 6]]
    s2 = np.array([[-0.0, 0.0, -1.0]], np.float32)
    assert orc.topk(s2, 1).tolist() == [[0]]


def test_topk_planted_distinct_scores(orc):
    s = np.full((2, 2250), -1.0, np.float32)
    planted = [3, 100, 2249, 1500, 7]
    s[0, planted] = [9, 8, 7, 6, 5]
    s[1, planted] = [1, 2, 3, 4, 5]
    assert orc.topk(s, 5).tolist() == [sorted(planted)] * 2
    assert orc.topk(s, 2).tolist() == [[3, 100], [7, 1500]]


def _kv_cache(orc, T, hkv, seed):
    shape = orc.Shape(1, hkv, 256, DI)
    ptok = 16
    n = synth.pages_for(T, ptok)
    ps = orc.page_elems(shape, ptok)
    c = orc.paged(shape, np.zeros(n * ps, np.uint16), ptok, synth.reversed_table(n))
    k = synth.normal_bf16(seed, (T, hkv, 256))
    v = synth.normal_bf16(seed + 1, (T, hkv, 256))
    orc.put_rows(shape, c, 0, orc.K, 0, k)
    orc.put_rows(shape, c, 0, orc.V, 0, v)
    return shape, c, k, v


def test_sparse_with_every_block_is_dense(orc):
    T, hq = 64, 4
    shape, c, _, _ = _kv_cache(orc, T, 2, 30)
    q = synth.normal_bf16(32, (hq, 256))
    ids = np.tile(np.arange(T // 4, dtype=np.int32), (hq, 1))
    sp = orc.sparse_attend(shape, c, 0, hq, T, q, ids)
    for h in range(hq):
        dense = orc.attend_row(shape, c, 0, hq, h, T - 1, q[h])
        assert np.allclose(sp[h], dense, rtol=1e-14, atol=1e-15)


def test_sparse_reads_only_selected_blocks(orc):
    T, hq = 80, 2
    shape, c, k, v = _kv_cache(orc, T, 1, 40)
    q = synth.normal_bf16(42, (hq, 256))
    ids = np.array([[2, 9, -1], [0, 19, 5]], np.int32)
    out = orc.sparse_attend(shape, c, 0, hq, T, q, ids)
    for h in range(hq):
        pos = [4 * b + r for b in ids[h] if b >= 0 for r in range(4)]
        # the same rows placed as a short contiguous stream, read densely
        sub = orc.contiguous(shape, len(pos))
        orc.put_rows(shape, sub, 0, orc.K, 0, k[pos])
        orc.put_rows(shape, sub, 0, orc.V, 0, v[pos])
        dense = orc.attend_row(shape, sub, 0, hq, h, len(pos) - 1, q[h])
        assert np.allclose(out[h], dense, rtol=1e-14, atol=1e-15)


def test_sparse_with_no_blocks_is_zero(orc):
    shape, c, _, _ = _kv_cache(orc, 16, 1, 50)
    out = orc.sparse_attend(shape, c, 0, 1, 16, synth.normal_bf16(52, (1, 256)),
                            np.full((1, 4), -1, np.int32))
    assert (out == 0).all()
