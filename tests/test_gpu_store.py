"""GPU parity: cache store, gather and pooling against the oracle, bit for bit.

The kernel contract of #1169/#1170: streams shuffled through one arena at
pages of 16, 48, 128, 256 and 512 positions, cached lengths up to 9,000;
the stored bytes equal the oracle's placement, reading back through the
tables gives the contiguous bytes, guards and inputs stay intact, and the
red controls (a swapped table over placed pages, a planted row, every
stream given stream 0's table) go red.
"""
import numpy as np
import pytest

import oracle as orc
from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import CANARY, dev_u16, host_u16, place, torch

pytestmark = pytest.mark.gpu

PAGES = [16, 48, 128, 256, 512]


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def _streams(lens, n_layers=2, hkv=2, seed=0):
    return [synth.make_stream(seed + i, n_layers, T, hkv, 256, 128) for i, T in enumerate(lens)]


@pytest.mark.parametrize("ptok", PAGES + [None])
def test_store_bytes_equal_oracle_placement(ptok):
    lay = pkv.layout(2, 2, 256, 128)
    streams = _streams([1000, 3000, 6000, 9000])
    pl = place(lay, streams, ptok, seed=ptok or 0)
    for i in range(len(pl.buffers)):
        assert np.array_equal(host_u16(pl.body(i)), pl.oarenas[i])
    assert pl.guards_intact()


@pytest.mark.parametrize("ptok", PAGES)
def test_gather_through_tables_gives_contiguous_bytes(ptok):
    t = torch()
    lay = pkv.layout(2, 2, 256, 128)
    streams = _streams([777, 4000], seed=7)
    pl = place(lay, streams, ptok, seed=3)
    seqs = pl.seqs()
    for layer in range(2):
        for kind, attr, shape in [(pkv.K, "k", (2, 256)), (pkv.V, "v", (2, 256)),
                                  (pkv.IK, "ik", (128,))]:
            out = t.empty((sum(s.length for s in streams),) + shape, dtype=t.int16, device="cuda")
            pkv.gather(lay, seqs, layer, kind, out)
            want = np.concatenate([getattr(s, attr)[layer] for s in streams])
            assert np.array_equal(host_u16(out), want)


@pytest.mark.parametrize("hkv,ptok", [(3, 16), (8, 48), (8, None)])
def test_store_and_gather_with_many_kv_heads(hkv, ptok):
    # 3 and 8 KV heads: a store lane takes more than one batch of chunks
    # (2*H*32 + 16 chunks a token) and a gather lane more than one batch of
    # heads; bytes must still equal the oracle's placement and read back
    t = torch()
    lay = pkv.layout(1, hkv, 256, 128)
    streams = _streams([333, 1029], n_layers=1, hkv=hkv, seed=40 + hkv)
    pl = place(lay, streams, ptok, seed=hkv)
    for i in range(len(pl.buffers)):
        assert np.array_equal(host_u16(pl.body(i)), pl.oarenas[i])
    assert pl.guards_intact()
    seqs = pl.seqs()
    total = sum(s.length for s in streams)
    for kind, attr, shape in [(pkv.K, "k", (hkv, 256)), (pkv.V, "v", (hkv, 256)),
                              (pkv.IK, "ik", (128,))]:
        out = t.empty((total,) + shape, dtype=t.int16, device="cuda")
        pkv.gather(lay, seqs, 0, kind, out)
        want = np.concatenate([getattr(s, attr)[0] for s in streams])
        assert np.array_equal(host_u16(out), want)


def test_reversed_table_single_stream_matches_contiguous():
    lay = pkv.layout(1, 1, 256, 128)
    s = _streams([64], n_layers=1, hkv=1)
    paged = place(lay, s, 16, tables=[synth.reversed_table(4)], spare_pages=0)
    cont = place(lay, s, None)
    t = torch()
    for kind in (pkv.K, pkv.V, pkv.IK):
        a = t.empty((64, 256 if kind < 2 else 128), dtype=t.int16, device="cuda")
        b = t.empty_like(a)
        pkv.gather(lay, paged.seqs(), 0, kind, a)
        pkv.gather(lay, cont.seqs(), 0, kind, b)
        assert t.equal(a, b)


def test_decode_store_appends_one_row_per_stream():
    t = torch()
    lay = pkv.layout(1, 2, 256, 128)
    streams = _streams([1000, 3000, 6000, 9000], n_layers=1)
    pl = place(lay, streams, 128, seed=11)
    new = [synth.make_stream(50 + i, 1, 1, 2, 256, 128) for i in range(4)]
    seqs = pl.seqs([s.length + 1 for s in streams], [1] * 4)
    k = dev_u16(np.concatenate([n.k[0] for n in new]))
    v = dev_u16(np.concatenate([n.v[0] for n in new]))
    ik = dev_u16(np.concatenate([n.ik[0] for n in new]))
    k_before = host_u16(k).copy()
    pkv.store(lay, seqs, 0, k, v, ik)
    for oc, s, n in zip(pl.ocaches, streams, new):
        orc.put_rows(pl.shape, oc, 0, orc.K, s.length, n.k[0])
        orc.put_rows(pl.shape, oc, 0, orc.V, s.length, n.v[0])
        orc.put_rows(pl.shape, oc, 0, orc.IK, s.length, n.ik[0])
    t.cuda.synchronize()
    assert np.array_equal(host_u16(pl.body()), pl.oarenas[0])
    assert np.array_equal(host_u16(k), k_before)          # inputs intact
    assert pl.guards_intact()


@pytest.mark.parametrize("ptok", [16, 48, 128])
def test_pool_bits_equal_oracle(ptok):
    t = torch()
    lay = pkv.layout(2, 2, 256, 128)
    streams = _streams([1000, 9000, 37], seed=21)
    pl = place(lay, streams, ptok, seed=5)
    # pool every complete block: n_new = len
    seqs = pl.seqs([s.length for s in streams], [s.length for s in streams])
    for layer in range(2):
        pkv.pool(lay, seqs, layer)
        for oc, s in zip(pl.ocaches, streams):
            orc.pool(pl.shape, oc, layer, 0, s.length // 4)
    t.cuda.synchronize()
    assert np.array_equal(host_u16(pl.body()), pl.oarenas[0])


def test_pool_only_blocks_completed_by_new_tokens():
    t = torch()
    lay = pkv.layout(1, 1, 256, 128)
    streams = _streams([31512], n_layers=1, hkv=1, seed=31)
    pl = place(lay, streams, 256, seed=2)
    # a 512-token chunk appended at 31,000 completes blocks 7750 .. 7877
    pkv.pool(lay, pl.seqs([31512], [512]), 0)
    orc.pool(pl.shape, pl.ocaches[0], 0, 7750, 128)
    t.cuda.synchronize()
    assert np.array_equal(host_u16(pl.body()), pl.oarenas[0])
    # one more token that completes no block changes nothing
    pkv.pool(lay, pl.seqs([31511], [1]), 0)
    t.cuda.synchronize()
    assert np.array_equal(host_u16(pl.body()), pl.oarenas[0])


def test_red_swapped_table_and_planted_row():
    t = torch()
    lay = pkv.layout(1, 2, 256, 128)
    streams = _streams([200, 300], n_layers=1, seed=40)
    pl = place(lay, streams, 16, seed=9)
    good = host_u16(pl.body()).copy()
    # swapped table over placed pages
    tab = pl.tables[0].copy()
    tab[[0, 3]] = tab[[3, 0]]
    dt = t.from_numpy(tab).cuda()
    g = pkv.pg(pl.body(), dt, pl.pgs[0].page_elems, 16, pl.pgs[0].n_pages, tab.size)
    out = t.empty((200, 2, 256), dtype=t.int16, device="cuda")
    pkv.gather(lay, [pkv.seq(g, 200, 0)], 0, pkv.K, out)
    assert not np.array_equal(host_u16(out), streams[0].k[0])
    # every stream given stream 0's table (#2244's grouped-lane bug)
    pkv.gather(lay, [pkv.seq(pl.pgs[0], 200, 0)], 0, pkv.K, out)
    assert not np.array_equal(host_u16(out), streams[1].k[0][:200])
    # planted row: one bit of one stored row
    body = pl.body()
    off = pkv.pg_row(lay, pl.pgs[1], pl.tables[1], 0, pkv.V, 1, 123)
    body[off + 7] ^= 1
    got = t.empty((300, 2, 256), dtype=t.int16, device="cuda")
    pkv.gather(lay, [pl.seqs()[1]], 0, pkv.V, got)
    diff = np.argwhere(host_u16(got) != streams[1].v[0])
    assert diff.tolist() == [[123, 1, 7]]
    body[off + 7] ^= 1
    assert np.array_equal(host_u16(body), good)


def test_bad_table_entry_is_reported_not_followed():
    t = torch()
    lay = pkv.layout(1, 1, 256, 128)
    streams = _streams([64], n_layers=1, hkv=1, seed=60)
    pl = place(lay, streams, 16, seed=1)
    before = host_u16(pl.body()).copy()
    bad = pl.tables[0].copy()
    bad[2] = pl.pgs[0].n_pages + 5               # outside the arena
    dt = t.from_numpy(bad).cuda()
    g = pkv.pg(pl.body(), dt, pl.pgs[0].page_elems, 16, pl.pgs[0].n_pages, bad.size)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    new = synth.make_stream(61, 1, 64, 1, 256, 128)
    pkv.store(lay, [pkv.seq(g, 64, 64)], 0, dev_u16(new.k[0]), dev_u16(new.v[0]),
              dev_u16(new.ik[0]), status=status)
    t.cuda.synchronize()
    assert int(status.item()) & pkv.DEV_BAD_PAGE
    after = host_u16(pl.body())
    # rows of the three good pages were rewritten; nothing outside them changed
    changed = np.flatnonzero(after != before)
    ps = pl.pgs[0].page_elems
    pages_touched = set((changed // ps).tolist())
    assert pages_touched <= {int(x) for x in bad[[0, 1, 3]]}
    assert pl.guards_intact()
