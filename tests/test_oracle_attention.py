"""Pins for the oracle's float64 attention.

The pages read attention rows "within a float64 bound" but do not write the
arithmetic out; the oracle takes scale 1/sqrt(D), KV head h // G and a
max-subtracted softmax.  These tests pin it with closed forms (zero query,
constant values, a single key, two keys with logits 1 and 0, a dominant
key), invariants (value shift and scale, key order, paging) and the special
cases that expose a wrong head mapping or an off-by-one in the causal bound.
"""
import math

import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import synth

D = 256


def bf(x):
    """bf16 bits of values that are exactly representable (checked)."""
    f = np.asarray(x, np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), f)
    return b


def widen(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _cache(orc, k, v, hkv=1, ptok=None, table=None):
    """Place K/V ([T][Hkv][D]) into a contiguous or paged cache."""
    T = k.shape[0]
    shape = orc.Shape(1, hkv, D, 0)
    if table is None:
        c = orc.contiguous(shape, max(4, -(-T // 4) * 4))
    else:
        ps = orc.page_elems(shape, ptok)
        c = orc.paged(shape, np.zeros(int(table.max() + 1) * ps, np.uint16), ptok, table)
    orc.put_rows(shape, c, 0, orc.K, 0, k)
    orc.put_rows(shape, c, 0, orc.V, 0, v)
    return shape, c


def test_zero_query_gives_mean_of_values(orc):
    T = 37
    k = synth.normal_bf16(1, (T, 1, D))
    v = synth.normal_bf16(2, (T, 1, D))
    shape, c = _cache(orc, k, v)
    out = orc.attend_row(shape, c, 0, 1, 0, T - 1, np.zeros(D, np.uint16))
    assert np.allclose(out, widen(v[:, 0]).mean(axis=0), rtol=0, atol=1e-14)


def test_constant_values_give_that_constant(orc):
    T = 50
    k = synth.normal_bf16(3, (T, 1, D))
    row = synth.normal_bf16(4, (D,))
    v = np.broadcast_to(row, (T, 1, D)).copy()
    shape, c = _cache(orc, k, v)
    q = synth.normal_bf16(5, (D,))
    out = orc.attend_row(shape, c, 0, 1, 0, T - 1, q)
    assert np.allclose(out, widen(row), rtol=1e-14, atol=0)


def test_first_position_reads_only_itself(orc):
    k = synth.normal_bf16(6, (5, 1, D))
    v = synth.normal_bf16(7, (5, 1, D))
    shape, c = _cache(orc, k, v)
    out = orc.attend_row(shape, c, 0, 1, 0, 0, synth.normal_bf16(8, (D,)))
    assert np.array_equal(out, widen(v[0, 0]))


def test_two_keys_logits_one_and_zero(orc):
    # q.k0 = 4*4 = 16, scaled by 1/sqrt(256) -> logit 1; k1 = 0 -> logit 0.
    q = np.zeros(D, np.float32); q[0] = 4
    k = np.zeros((2, 1, D), np.float32); k[0, 0, 0] = 4
    v = np.zeros((2, 1, D), np.float32); v[0, 0, :3] = [1, 2, -3]; v[1, 0, :3] = [5, 0, 1]
    shape, c = _cache(orc, bf(k), bf(v))
    out = orc.attend_row(shape, c, 0, 1, 0, 1, bf(q))
    e = math.e
    v64 = v.astype(np.float64)
    want = (e * v64[0, 0, :3] + v64[1, 0, :3]) / (e + 1)
    assert np.allclose(out[:3], want, rtol=0, atol=1e-14)
    assert (out[3:] == 0).all()


def test_dominant_key_closed_form(orc):
    T, j = 100, 37
    q = np.zeros(D, np.float32); q[1] = 8
    k = np.zeros((T, 1, D), np.float32); k[j, 0, 1] = 8      # logit 64/16 = 4
    v = widen(synth.normal_bf16(9, (T, 1, D)))
    shape, c = _cache(orc, bf(k), bf(v.astype(np.float32)))
    out = orc.attend_row(shape, c, 0, 1, 0, T - 1, bf(q))
    w = math.exp(4)
    want = (w * v[j, 0] + (v[:, 0].sum(axis=0) - v[j, 0])) / (w + T - 1)
    assert np.allclose(out, want, rtol=0, atol=1e-13)


def test_huge_logits_do_not_overflow(orc):
    # logits of 2**14 would overflow exp() without the max subtraction.
    T = 6
    q = np.zeros(D, np.float32); q[:64] = 64
    k = np.zeros((T, 1, D), np.float32); k[3, 0, :64] = 64; k[1, 0, :64] = 32
    v = widen(synth.normal_bf16(10, (T, 1, D)))
    shape, c = _cache(orc, bf(k), bf(v.astype(np.float32)))
    out = orc.attend_row(shape, c, 0, 1, 0, T - 1, bf(q))
    assert np.isfinite(out).all()
    assert np.array_equal(out, v[3, 0])


def test_query_heads_share_kv_head_by_group(orc):
    # 4 query heads over 2 KV heads: heads 0,1 read KV head 0, heads 2,3 KV head 1.
    T = 12
    k = synth.normal_bf16(11, (T, 2, D))
    v = np.zeros((T, 2, D), np.float32); v[:, 0] = 1.0; v[:, 1] = 2.0
    shape, c = _cache(orc, k, bf(v), hkv=2)
    q = synth.normal_bf16(12, (1, 4, D))
    out = orc.attend(shape, c, 0, 4, T, q)
    assert np.allclose(out[0, :, 0], [1, 1, 2, 2], rtol=0, atol=1e-14)


def test_causal_window_hides_later_keys(orc):
    # A 4-query window at positions L..L+3: query j must not see L+j+1..
    L, T = 20, 24
    k = synth.normal_bf16(13, (T, 1, D))
    v = synth.normal_bf16(14, (T, 1, D))
    q = synth.normal_bf16(15, (4, 1, D))
    shape, c = _cache(orc, k, v)
    base = orc.attend(shape, c, 0, 1, T, q)
    v2 = v.copy(); v2[L + 2] = synth.normal_bf16(16, (1, D))
    shape, c2 = _cache(orc, k, v2)
    moved = orc.attend(shape, c2, 0, 1, T, q)
    assert np.array_equal(base[:2], moved[:2])          # queries at L, L+1
    assert not np.allclose(base[2:], moved[2:])         # queries at L+2, L+3


def test_value_shift_and_scale(orc):
    T = 40
    rng = np.random.default_rng(17)
    k = synth.normal_bf16(18, (T, 1, D))
    v = rng.integers(-8, 9, (T, 1, D)).astype(np.float32)
    q = synth.normal_bf16(19, (D,))
    shape, c = _cache(orc, k, bf(v))
    o = orc.attend_row(shape, c, 0, 1, 0, T - 1, q)
    shape, c3 = _cache(orc, k, bf(v + 3))
    shape, c2 = _cache(orc, k, bf(2 * v))
    assert np.allclose(orc.attend_row(shape, c3, 0, 1, 0, T - 1, q), o + 3, rtol=0, atol=1e-12)
    assert np.allclose(orc.attend_row(shape, c2, 0, 1, 0, T - 1, q), 2 * o, rtol=0, atol=1e-12)


def test_key_order_does_not_matter(orc):
    T = 33
    k = synth.normal_bf16(20, (T, 1, D))
    v = synth.normal_bf16(21, (T, 1, D))
    q = synth.normal_bf16(22, (D,))
    perm = np.random.default_rng(23).permutation(T)
    shape, c = _cache(orc, k, v)
    shape, cp = _cache(orc, k[perm], v[perm])
    a = orc.attend_row(shape, c, 0, 1, 0, T - 1, q)
    b = orc.attend_row(shape, cp, 0, 1, 0, T - 1, q)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("ptok", [4, 16, 48])
def test_paged_attention_equals_contiguous_bitwise(orc, ptok):
    # Only addresses change: the same rows in the same order.
    T = 150
    k = synth.normal_bf16(24, (T, 2, D))
    v = synth.normal_bf16(25, (T, 2, D))
    q = synth.normal_bf16(26, (3, 8, D))
    shape, c = _cache(orc, k, v, hkv=2)
    n = synth.pages_for(T, ptok)
    shape, p = _cache(orc, k, v, hkv=2, ptok=ptok, table=synth.reversed_table(n, first=2))
    assert np.array_equal(orc.attend(shape, c, 0, 8, T, q), orc.attend(shape, p, 0, 8, T, q))
