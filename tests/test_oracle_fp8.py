"""Pins for the oracle's e4m3 K/V format (TensorFold #1170, commit 5c09685:
a row's e4m3 codes and float32 scale through row8(); the reference
dequantizes e4m3 x scale in float64).

What pins it, other than the oracle itself: the pool size the page prints
for the format; the e4m3 format's own values (the code of 1, of the largest
and smallest magnitudes, NaN); brute-force nearest-value search over every
finite code for the encoder; exact round trips of rows that are e4m3 values
times a power of two; a bound on the quantization error of any row; and the
bf16 attention path, which the e4m3 path must equal exactly when the rows
need no rounding.
"""
import os

import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pool_sizes_e4m3.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("|")[0].strip()
        if line and not line.startswith("#"):
            rows.append([float(x) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _golden_rows())
def test_e4m3_page_bytes_reproduce_printed_pool_size(orc, row):
    layers, hkv, d, di, ptok, pages, gib = row
    shape = orc.Shape(int(layers), int(hkv), int(d), int(di), orc.E4M3)
    assert round(orc.page_elems(shape, int(ptok)) * 2 * int(pages) / 2**30, 2) == gib
    # near misses: scales in bf16, or one scale per position for all heads
    for per_head_row in (2 * (256 + 2), 2 * 256 + 2 * 4 / 4):
        assert round(16 * 4 * per_head_row * 256 * 387 / 2**30, 2) != gib


def test_e4m3_code_values(orc):
    codes = [0x00, 0x01, 0x07, 0x08, 0x38, 0x3F, 0x40, 0x7E, 0x80, 0xB8, 0xFE]
    want = [0.0, 2.0**-9, 7 * 2.0**-9, 2.0**-6, 1.0, 1.875, 2.0, 448.0, -0.0, -1.0, -448.0]
    got = orc.e4m3_to_double(codes)
    assert np.array_equal(got, want)
    assert np.signbit(got[8])
    assert np.isnan(orc.e4m3_to_double([0x7F, 0xFF])).all()


def _finite_table(orc):
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    return codes, orc.e4m3_to_double(codes)


def test_every_finite_code_round_trips(orc):
    codes, vals = _finite_table(orc)
    assert np.array_equal(orc.e4m3_from_float(vals.astype(np.float32)), codes)
    # the positive magnitudes are strictly increasing with the code
    pos = vals[codes < 0x80]
    assert (np.diff(pos) > 0).all()


def test_encoder_picks_the_nearest_code_ties_to_even(orc):
    codes, vals = _finite_table(orc)
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-460, 460, 4000), rng.uniform(-2**-5, 2**-5, 4000),
                        # every midpoint between neighbouring codes
                        (np.sort(vals[codes < 0x80])[:-1] + np.sort(vals[codes < 0x80])[1:]) / 2]
                       ).astype(np.float32)
    got = orc.e4m3_from_float(x)
    for xi, ci in zip(x.astype(np.float64), got):
        a = abs(xi)
        if a >= 448:
            assert ci & 0x7F == 0x7E
            continue
        dist = np.abs(np.abs(vals) - a)
        best = dist.min()
        cand = [c for c, dd in zip(codes, dist) if dd == best and (c & 0x80) == (0x80 if np.signbit(xi) else 0)]
        assert ci in cand
        if len(cand) > 1:                       # a tie: the even mantissa wins
            assert ci & 1 == 0


def test_exactly_representable_rows_quantize_exactly(orc):
    # e4m3 values times 2^-6, the largest being 448 * 2^-6 = 7: scale 2^-6
    rng = np.random.default_rng(2)
    codes, vals = _finite_table(orc)
    pick = rng.choice(vals, 255).astype(np.float64)
    row = np.concatenate([[448.0], pick]) * 2.0**-6
    bits = (row.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(orc.bf16_to_float(bits), row)          # bf16 holds them exactly
    c, sc = orc.quantize_row(bits)
    assert sc == np.float32(2.0**-6)
    assert np.array_equal(orc.e4m3_to_double(c) * float(sc), row)


def test_quantization_error_bound_and_zero_row(orc):
    rng = np.random.default_rng(3)
    for scale in (1.0, 1e-3, 37.0):
        bits = synth.normal_bf16(int(scale * 1000) % 97, (256,))
        x = orc.bf16_to_float(bits) * 1.0
        x = x * scale
        bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        x = orc.bf16_to_float(bits)
        c, sc = orc.quantize_row(bits)
        deq = orc.e4m3_to_double(c) * float(sc)
        amax = np.abs(x).max()
        # the largest magnitude lands on +-448 codes; every element is within
        # half an e4m3 step (2^-4 relative above 2^-6, 2^-10 absolute below), scaled
        assert (c[np.abs(x) == amax] & 0x7F == 0x7E).all()
        q = np.abs(x) / float(sc)
        step = np.where(q >= 2**-6, 2.0 ** (np.floor(np.log2(np.maximum(q, 2**-6))) - 3), 2.0**-9)
        assert (np.abs(deq - x) <= (step / 2 * (1 + 1e-6) + 1e-7 * q) * float(sc)).all()
    c, sc = orc.quantize_row(np.zeros(256, np.uint16))
    assert sc == 0.0 and not c.any()


@pytest.mark.parametrize("ptok", [4, 8, 12])
def test_tiny_e4m3_arena_rows_tile_pages_exactly(orc, ptok):
    shape = orc.Shape(2, 2, 8, 4, orc.E4M3)
    ps = orc.page_elems(shape, ptok)
    n_pages = 7
    tables = synth.shuffled_tables(4, n_pages, [3, 2])
    arena = np.zeros(n_pages * ps, np.uint16)
    hits = np.zeros(n_pages * ps * 2, np.int32)           # bytes
    widths = {orc.K: 8, orc.V: 8, orc.KS: 4, orc.VS: 4, orc.IK: 8, orc.P: 8}
    for t in tables:
        c = orc.paged(shape, arena, ptok, t)
        T = t.size * ptok
        for layer in range(2):
            for kind, width in widths.items():
                heads = 2 if kind in (orc.K, orc.V, orc.KS, orc.VS) else 1
                n = T // 4 if kind == orc.P else T
                for h in range(heads):
                    for pos in range(n):
                        off = orc.row8(shape, c, layer, kind, h, pos)
                        assert 0 <= off and off + width <= hits.size
                        hits[off:off + width] += 1
    used = np.zeros(n_pages, bool)
    for t in tables:
        used[t] = True
    per_page = hits.reshape(n_pages, ps * 2)
    assert (per_page[used] == 1).all() and (per_page[~used] == 0).all()
    # K/V rows of an e4m3 cache are bytes: the 16-bit row lookup refuses them
    c = orc.paged(shape, arena, ptok, tables[0])
    assert orc.row(shape, c, 0, orc.K, 0, 0) == -1
    assert orc.row(shape, c, 0, orc.IK, 0, 1) * 2 == orc.row8(shape, c, 0, orc.IK, 0, 1)
    assert orc.row8(orc.Shape(2, 2, 8, 4), c, 0, orc.K, 0, 0) == -1


def _place8(orc, shape, cache, stream):
    for layer in range(shape.n_layers):
        orc.put_rows8(shape, cache, layer, orc.K, 0, stream.k[layer])
        orc.put_rows8(shape, cache, layer, orc.V, 0, stream.v[layer])
        if shape.idx_dim:
            orc.put_rows(shape, cache, layer, orc.IK, 0, stream.ik[layer])


@pytest.mark.parametrize("ptok", [16, 48, 256])
def test_reversed_table_reads_contiguous_e4m3_bytes(orc, ptok):
    shape = orc.Shape(2, 2, 256, 128, orc.E4M3)
    T = 300
    s = synth.make_stream(11, 2, T, 2, 256, 128)
    cont = orc.contiguous(shape, T)
    _place8(orc, shape, cont, s)
    n = synth.pages_for(T, ptok)
    arena = np.zeros(n * orc.page_elems(shape, ptok), np.uint16)
    paged = orc.paged(shape, arena, ptok, synth.reversed_table(n))
    _place8(orc, shape, paged, s)
    for layer in range(2):
        for kind in (orc.K, orc.V, orc.KS, orc.VS):
            assert np.array_equal(orc.get_rows8(shape, cont, layer, kind, 0, T),
                                  orc.get_rows8(shape, paged, layer, kind, 0, T))
        assert np.array_equal(orc.get_rows(shape, cont, layer, orc.IK, 0, T),
                              orc.get_rows(shape, paged, layer, orc.IK, 0, T))


def test_e4m3_attention_equals_bf16_attention_on_exact_rows(orc):
    # Rows that quantize exactly (e4m3 values x 2^-6 with a 448 x 2^-6 element):
    # dequantized e4m3 attention must equal bf16 attention to the last bit.
    rng = np.random.default_rng(8)
    codes, vals = _finite_table(orc)
    T, H, D = 40, 2, 256

    def exact_rows():
        v = rng.choice(vals[np.abs(vals) <= 64], (1, T, H, D)).astype(np.float64)
        v[..., 0] = 448.0
        v *= 2.0**-6
        return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    s = synth.Stream(T, exact_rows(), exact_rows(), np.zeros((1, T, 0), np.uint16))
    q = synth.queries(9, 3, 8, D)
    out = []
    for fmt in (orc.BF16, orc.E4M3):
        shape = orc.Shape(1, H, D, 0, fmt)
        c = orc.contiguous(shape, T)
        if fmt == orc.BF16:
            orc.put_rows(shape, c, 0, orc.K, 0, s.k[0])
            orc.put_rows(shape, c, 0, orc.V, 0, s.v[0])
        else:
            orc.put_rows8(shape, c, 0, orc.K, 0, s.k[0])
            orc.put_rows8(shape, c, 0, orc.V, 0, s.v[0])
        out.append(orc.attend(shape, c, 0, 8, T, q))
    assert np.array_equal(out[0], out[1])


def test_e4m3_attention_stays_near_bf16_attention(orc):
    # random rows: the e4m3 result moves by about the quantization error only
    T, H, D = 200, 2, 256
    s = synth.make_stream(12, 1, T, H, D, 0)
    q = synth.queries(13, 1, 8, D)
    out = []
    for fmt in (orc.BF16, orc.E4M3):
        shape = orc.Shape(1, H, D, 0, fmt)
        c = orc.contiguous(shape, T)
        put = orc.put_rows if fmt == orc.BF16 else orc.put_rows8
        put(shape, c, 0, orc.K, 0, s.k[0])
        put(shape, c, 0, orc.V, 0, s.v[0])
        out.append(orc.attend(shape, c, 0, 8, T, q))
    err = np.abs(out[0] - out[1])
    assert err.max() < 0.05 and err.max() > 0
