"""Pins for the oracle's page layout and row translation (pg_at).

Each test checks the oracle against something the pages fix, not against a
retyping of its own code: the pool sizes they print, the two address rules
they state in words, the "only addresses change" invariant at every page
size with streams shuffled through one arena, and brute-force coverage of a
tiny arena.  The red controls plant mistakes in the oracle's inputs and
expect the comparison to fail.
"""
import os

import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pool_sizes.txt")
CANARY = 0x7FC1  # a bf16 NaN: any read of an unplaced row poisons a result


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("|")[0].strip()
        if not line or line.startswith("#"):
            continue
        rows.append([float(x) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _golden_rows())
def test_page_bytes_reproduce_printed_pool_sizes(orc, row):
    layers, hkv, d, di, ptok, pages, gib = row
    shape = orc.Shape(int(layers), int(hkv), int(d), int(di))
    bytes_ = orc.page_elems(shape, int(ptok)) * 2 * int(pages)
    assert round(bytes_ / 2**30, 2) == gib


def test_pool_size_rejects_plausible_layout_mistakes(orc):
    # The printed 4.36 GiB separates the layout from its near misses.
    per_pos = {"taken": 2 * 2 * 256 * 2 + 128 * 2 + 128 * 2 / 4,
               "no pooled rows": 2 * 2 * 256 * 2 + 128 * 2,
               "a pooled row per position": 2 * 2 * 256 * 2 + 128 * 2 * 2}
    gib = {k: round(13 * v * 256 * 594 / 2**30, 2) for k, v in per_pos.items()}
    assert gib["taken"] == 4.36
    assert gib["no pooled rows"] != 4.36 and gib["a pooled row per position"] != 4.36
    shape = orc.Shape(13, 2, 256, 128)
    assert orc.page_elems(shape, 256) * 2 == 13 * 256 * per_pos["taken"]


def test_no_table_is_cap_rows_a_head(orc):
    # #1170 commit 3f5b87d: with no table, the old expression, cap rows a head.
    shape = orc.Shape(3, 2, 256, 128)
    cap = 20
    c = orc.contiguous(shape, cap)
    le = orc.layer_elems(shape, cap)
    for layer in range(3):
        for head in range(2):
            for pos in (0, 1, 7, cap - 1):
                assert orc.row(shape, c, layer, orc.K, head, pos) == \
                    layer * le + head * cap * 256 + pos * 256
                assert orc.row(shape, c, layer, orc.V, head, pos) == \
                    layer * le + 2 * cap * 256 + head * cap * 256 + pos * 256
    assert orc.row(shape, c, 0, orc.K, 0, cap) == -1


def test_table_is_page_start_plus_row_inside(orc):
    # #1169 "fn-paged-kv": with a table, the start of the page that holds the
    # position plus the row inside that page; a contiguous buffer of cap =
    # ptok rows is exactly one such page.
    shape = orc.Shape(2, 2, 256, 128)
    ptok, n_pages = 16, 9
    ps = orc.page_elems(shape, ptok)
    table = np.array([4, 0, 7, 2], dtype=np.int32)
    c = orc.paged(shape, np.zeros(n_pages * ps, np.uint16), ptok, table)
    one_page = orc.contiguous(shape, ptok)
    for layer in range(2):
        for kind in (orc.K, orc.V, orc.IK):
            for head in range(2 if kind != orc.IK else 1):
                for pos in range(0, 64, 5):
                    got = orc.row(shape, c, layer, kind, head, pos)
                    inner = orc.row(shape, one_page, layer, kind, head, pos % ptok)
                    assert got == table[pos // ptok] * ps + inner
        for b in range(16):
            got = orc.row(shape, c, layer, orc.P, 0, b)
            inner = orc.row(shape, one_page, layer, orc.P, 0, b % (ptok // 4))
            assert got == table[(4 * b) // ptok] * ps + inner


def test_out_of_range_rows_are_refused(orc):
    shape = orc.Shape(1, 1, 256, 128)
    ptok = 8
    ps = orc.page_elems(shape, ptok)
    c = orc.paged(shape, np.zeros(3 * ps, np.uint16), ptok, np.array([2, 5], np.int32))
    assert orc.row(shape, c, 0, orc.K, 0, 7) >= 0
    assert orc.row(shape, c, 0, orc.K, 0, 8) == -1        # page id 5 >= 3 pages
    assert orc.row(shape, c, 0, orc.K, 0, 16) == -1       # past the table
    assert orc.row(shape, c, 1, orc.K, 0, 0) == -1        # no layer 1
    assert orc.row(shape, c, 0, orc.K, 1, 0) == -1        # no KV head 1


@pytest.mark.parametrize("ptok", [4, 8, 12])
def test_tiny_arena_rows_tile_pages_exactly(orc, ptok):
    # Brute force: every (stream, layer, kind, head, row) of two streams that
    # fill their pages maps to a distinct element range, and together they
    # cover each used page exactly once (no overlap, no gap, nothing outside).
    shape = orc.Shape(2, 2, 8, 4)
    ps = orc.page_elems(shape, ptok)
    n_pages = 7
    tables = synth.shuffled_tables(3, n_pages, [3, 2])
    arena = np.zeros(n_pages * ps, np.uint16)
    hits = np.zeros(n_pages * ps, np.int32)
    for t in tables:
        c = orc.paged(shape, arena, ptok, t)
        T = t.size * ptok
        for layer in range(2):
            for kind in (orc.K, orc.V, orc.IK, orc.P):
                heads = 2 if kind in (orc.K, orc.V) else 1
                n = T // 4 if kind == orc.P else T
                width = 8 if kind in (orc.K, orc.V) else 4
                for h in range(heads):
                    for pos in range(n):
                        off = orc.row(shape, c, layer, kind, h, pos)
                        assert 0 <= off and off + width <= arena.size
                        hits[off:off + width] += 1
    used = np.zeros(n_pages, bool)
    for t in tables:
        used[t] = True
    per_page = hits.reshape(n_pages, ps)
    assert (per_page[used] == 1).all()
    assert (per_page[~used] == 0).all()


def _place(orc, shape, cache, stream):
    for layer in range(shape.n_layers):
        orc.put_rows(shape, cache, layer, orc.K, 0, stream.k[layer])
        orc.put_rows(shape, cache, layer, orc.V, 0, stream.v[layer])
        orc.put_rows(shape, cache, layer, orc.IK, 0, stream.ik[layer])


def _gather(orc, shape, cache, T):
    return [(orc.get_rows(shape, cache, l, orc.K, 0, T), orc.get_rows(shape, cache, l, orc.V, 0, T),
             orc.get_rows(shape, cache, l, orc.IK, 0, T)) for l in range(shape.n_layers)]


def _same(a, b):
    return all(np.array_equal(x, y) for la, lb in zip(a, b) for x, y in zip(la, lb))


@pytest.mark.parametrize("ptok", [16, 48, 128, 256, 512])
def test_reversed_table_reads_contiguous_bytes(orc, ptok):
    # #1169 "fn-paged-kv": a reversed table of n-position pages reads the
    # same bytes as the contiguous caches, at any page size holding whole
    # blocks; cached lengths up to 9,000 as in the kernel contract's cases.
    shape = orc.Shape(2, 2, 256, 128)
    T = 9000
    s = synth.make_stream(1, 2, T, 2, 256, 128)
    cont = orc.contiguous(shape, T, CANARY)
    _place(orc, shape, cont, s)
    n = synth.pages_for(T, ptok)
    ps = orc.page_elems(shape, ptok)
    arena = np.full(n * ps, CANARY, np.uint16)
    pag = orc.paged(shape, arena, ptok, synth.reversed_table(n))
    _place(orc, shape, pag, s)
    got_c, got_p = _gather(orc, shape, cont, T), _gather(orc, shape, pag, T)
    assert _same(got_c, got_p)
    assert np.array_equal(got_p[1][0], s.k[1]) and np.array_equal(got_p[0][2], s.ik[0])
    # the last logical page is physical page 0: its first K row is position (n-1)*ptok
    first = orc.row(shape, pag, 0, orc.K, 0, (n - 1) * ptok)
    assert first == 0


@pytest.mark.parametrize("n_streams", [2, 4])
def test_streams_shuffled_through_one_arena(orc, n_streams):
    shape = orc.Shape(1, 2, 256, 128)
    ptok = 48
    lens = [500, 1201, 77, 2000][:n_streams]
    streams = [synth.make_stream(10 + i, 1, T, 2, 256, 128) for i, T in enumerate(lens)]
    counts = [synth.pages_for(T, ptok) for T in lens]
    n_pages = sum(counts) + 3
    ps = orc.page_elems(shape, ptok)
    arena = np.full(n_pages * ps, CANARY, np.uint16)
    tables = synth.shuffled_tables(5, n_pages, counts)
    caches = [orc.paged(shape, arena, ptok, t) for t in tables]
    for c, s in zip(caches, streams):
        _place(orc, shape, c, s)
    for c, s, T in zip(caches, streams, lens):
        ref = orc.contiguous(shape, T)
        _place(orc, shape, ref, s)
        assert _same(_gather(orc, shape, c, T), _gather(orc, shape, ref, T))
    # pages nobody holds keep their canary
    free = np.setdiff1d(np.arange(n_pages), np.concatenate(tables))
    for p in free:
        assert (arena[p * ps:(p + 1) * ps] == CANARY).all()


# ---- red controls: a planted mistake must make the comparison fail -------

def _two_stream_setup(orc):
    shape = orc.Shape(1, 2, 256, 128)
    ptok, lens = 16, [64, 64]
    streams = [synth.make_stream(20 + i, 1, T, 2, 256, 128) for i, T in enumerate(lens)]
    ps = orc.page_elems(shape, ptok)
    arena = np.full(10 * ps, CANARY, np.uint16)
    tables = synth.shuffled_tables(9, 10, [4, 4])
    for t, s in zip(tables, streams):
        _place(orc, shape, orc.paged(shape, arena, ptok, t), s)
    return shape, ptok, arena, tables, streams


def test_red_swapped_table_over_placed_pages(orc):
    shape, ptok, arena, tables, streams = _two_stream_setup(orc)
    swapped = tables[0].copy()
    swapped[[0, 2]] = swapped[[2, 0]]
    got = orc.get_rows(shape, orc.paged(shape, arena, ptok, swapped), 0, orc.K, 0, 64)
    assert not np.array_equal(got, streams[0].k[0])
    ok = orc.get_rows(shape, orc.paged(shape, arena, ptok, tables[0]), 0, orc.K, 0, 64)
    assert np.array_equal(ok, streams[0].k[0])


def test_red_planted_row(orc):
    shape, ptok, arena, tables, streams = _two_stream_setup(orc)
    c = orc.paged(shape, arena, ptok, tables[1])
    off = orc.row(shape, c, 0, orc.V, 1, 37)
    arena[off + 5] ^= 0x0001
    got = orc.get_rows(shape, c, 0, orc.V, 0, 64)
    assert not np.array_equal(got, streams[1].v[0])
    assert np.argwhere(got != streams[1].v[0]).tolist() == [[37, 1, 5]]


def test_red_every_stream_given_stream_zeros_table(orc):
    # #2244: a grouped lane built without its own table read and wrote other
    # streams' pages.  Reading stream 1 through stream 0's table must go red.
    shape, ptok, arena, tables, streams = _two_stream_setup(orc)
    got = orc.get_rows(shape, orc.paged(shape, arena, ptok, tables[0]), 0, orc.K, 0, 64)
    assert not np.array_equal(got, streams[1].k[0])
