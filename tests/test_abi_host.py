"""Host-side checks of the C ABI that need no GPU.

The library must load and export every function ``include/pkv.h`` declares;
host pg_at must agree with the oracle's translation bit for bit; argument
checks must refuse malformed descriptors before anything is launched; the
page arena must hand out the lowest free pages, refuse over-asks with
PKV_EAGAIN, and return pages only after the stream's work is done (checked
with fake event operations, so no GPU is involved).
"""
import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import build, pkv, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pkv.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*int\s+(pkv_\w+)\s*\(", txt, re.M))
    return names


def test_library_exports_every_declared_function(lib):
    declared = _declared()
    assert len(declared) >= 18
    for name in declared:
        assert hasattr(lib, name), name
    assert set(pkv.EXPORTS) <= declared


def test_binding_constants_match_the_header():
    """Every numeric #define of include/pkv.h that the binding mirrors has
    the header's value there (status codes, device status bits, row kinds,
    formats)."""
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "pkv.h")).read()
    defs = {m.group(1): int(m.group(2))
            for m in re.finditer(r"^#define PKV_(\w+) (\d+)u?\b", hdr, re.M)}
    mirrored = {"OK": pkv.OK, "EINVAL": pkv.EINVAL, "EAGAIN": pkv.EAGAIN, "ECUDA": pkv.ECUDA,
                "EDEVICE": pkv.EDEVICE, "DEV_BAD_PAGE": pkv.DEV_BAD_PAGE,
                "DEV_TIMEOUT": pkv.DEV_TIMEOUT, "DEV_SMEM": pkv.DEV_SMEM, "DEV_RANGE": pkv.DEV_RANGE,
                "K": pkv.K, "V": pkv.V, "IK": pkv.IK, "P": pkv.P, "KS": pkv.KS, "VS": pkv.VS,
                "KV_BF16": pkv.KV_BF16, "KV_E4M3": pkv.KV_E4M3}
    for name, value in mirrored.items():
        assert defs.get(name) == value, (name, defs.get(name), value)
    # the device status bits are distinct single bits
    bits = [defs[n] for n in defs if n.startswith("DEV_")]
    assert len(bits) == 4 and all(b and b & (b - 1) == 0 for b in bits) and len(set(bits)) == 4


def test_page_elems_match_oracle(lib, orc):
    for hkv, di, ptok in [(2, 128, 256), (1, 128, 16), (4, 0, 48), (2, 128, 4)]:
        lay = pkv.layout(13, hkv, 256, di)
        assert pkv.page_elems(lay, ptok) == orc.page_elems(orc.Shape(13, hkv, 256, di), ptok)


@pytest.mark.parametrize("ptok", [4, 16, 48, 128, 256, 512])
def test_host_pg_at_equals_oracle(lib, orc, ptok):
    lay = pkv.layout(3, 2, 256, 128)
    shape = orc.Shape(3, 2, 256, 128)
    ps = pkv.page_elems(lay, ptok)
    n_pages = 40
    table = synth.shuffled_tables(ptok, n_pages, [7])[0]
    arena = np.zeros(1, np.uint16)
    oc = orc.Cache(arena, ptok, ps, table, n_pages)
    g = pkv.pg(0x10000, 0x20000, ps, ptok, n_pages, table.size)
    rng = np.random.default_rng(ptok)
    for _ in range(400):
        layer = int(rng.integers(3)); kind = int(rng.integers(4)); head = int(rng.integers(2))
        limit = 7 * ptok // 4 if kind == 3 else 7 * ptok
        pos = int(rng.integers(limit))
        if kind >= 2:
            head = 0
        assert pkv.pg_row(lay, g, table, layer, kind, head, pos) == \
            orc.row(shape, oc, layer, kind, head, pos)
    # contiguous: one page of cap rows
    cap = 7 * ptok
    cont = pkv.pg(0x10000, None, pkv.page_elems(lay, cap), cap)
    occ = orc.Cache(arena, cap, pkv.page_elems(lay, cap), None, 1)
    for pos in (0, 1, cap - 1):
        for kind in range(4):
            p = pos // 4 if kind == 3 else pos
            assert pkv.pg_row(lay, cont, None, 2, kind, 0, p) == orc.row(shape, occ, 2, kind, 0, p)


def test_pg_at_refuses_rows_outside(lib):
    lay = pkv.layout(1, 1, 256, 128)
    ps = pkv.page_elems(lay, 16)
    table = np.array([3, 9], np.int32)
    g = pkv.pg(0x10000, 0x20000, ps, 16, 5, 2)
    with pytest.raises(pkv.PkvError):
        pkv.pg_row(lay, g, table, 0, pkv.K, 0, 16)   # page id 9 >= 5 pages
    with pytest.raises(pkv.PkvError):
        pkv.pg_row(lay, g, table, 0, pkv.K, 0, 32)   # past the table
    with pytest.raises(pkv.PkvError):
        pkv.pg_row(lay, g, table, 1, pkv.K, 0, 0)    # no layer 1


@pytest.mark.parametrize("page_pos", [0, -4, 6, 17])
def test_page_size_must_be_a_multiple_of_four(lib, page_pos):
    with pytest.raises(pkv.PkvError) as e:
        pkv.page_elems(pkv.layout(1, 1), page_pos)
    assert e.value.code == pkv.EINVAL


def _seq(lay, ptok=16, length=10, n_new=1, base=0x10000, table=None, n_table=4, n_pages=8):
    ps = pkv.page_elems(lay, ptok)
    if table is None:
        return pkv.seq(pkv.pg(base, None, ps, ptok), length, n_new)
    return pkv.seq(pkv.Pg(base, table, ps, ptok, n_pages, n_table, 0), length, n_new)


def _store(lay, seqs, layer=0):
    lib = pkv.load()
    arr, n = pkv._seqs(seqs)
    return lib.pkv_store(ctypes.byref(lay), arr, n, layer, 0x1000, 0x1000, 0x1000, None, None)


def test_kernels_refuse_malformed_descriptors_before_launch(lib):
    lay = pkv.layout(2, 2)
    good = _seq(lay, table=0x30000)
    assert _store(pkv.layout(2, 2, 128, 128), [good]) == pkv.EINVAL       # head dim
    assert _store(pkv.layout(2, 2, 256, 64), [good]) == pkv.EINVAL        # indexer dim
    assert _store(lay, [good], layer=2) == pkv.EINVAL                      # no such layer
    bad_ps = _seq(lay, table=0x30000); bad_ps.pg.page_elems += 1
    assert _store(lay, [bad_ps]) == pkv.EINVAL
    assert _store(lay, [_seq(lay, base=0x10008, table=0x30000)]) == pkv.EINVAL  # misaligned
    assert _store(lay, [_seq(lay, length=65, table=0x30000)]) == pkv.EINVAL    # past 4 pages
    assert _store(lay, [_seq(lay, length=17)]) == pkv.EINVAL                   # past cap 16
    assert _store(lay, [_seq(lay, n_new=11)]) == pkv.EINVAL                    # n_new > len
    odd = _seq(lay, table=0x30000); odd.pg.page_pos = 18
    assert _store(lay, [odd]) == pkv.EINVAL                                    # 18 % 4
    assert _store(lay, [_seq(lay, table=0x30000, n_pages=0)]) == pkv.EINVAL
    arr = (pkv.Seq * 65)(*([good] * 65))
    assert pkv.load().pkv_store(ctypes.byref(lay), arr, 65, 0, 1, 1, 1, None, None) == pkv.EINVAL


def test_garbage_descriptor_is_refused(lib):
    # A descriptor left uninitialized must not be read as a valid table
    # (#1170: a test's undefined Cache.paged read as a page table on x86).
    lay = pkv.layout(1, 1)
    raw = (ctypes.c_uint8 * ctypes.sizeof(pkv.Seq))(*([0xAA] * ctypes.sizeof(pkv.Seq)))
    s = pkv.Seq.from_buffer_copy(raw)
    assert _store(lay, [s]) == pkv.EINVAL


def test_decode_refuses_too_many_query_columns(lib):
    lay = pkv.layout(1, 2)
    s = _seq(lay, length=100, n_new=5, ptok=128)
    arr, n = pkv._seqs([s])
    out = ctypes.c_size_t()
    # 5 queries x 8 heads a KV head = 40 columns > 32; checked before any device query
    rc = pkv.load().pkv_decode(ctypes.byref(lay), arr, n, 0, 16, 16, None, None, None, 16, None,
                               0, None, None)
    assert rc == pkv.EINVAL


def test_diag_wait_needs_a_status_word(lib):
    assert lib.pkv_diag_wait_runs_out(None, None) == pkv.EINVAL   # refused before any launch


# ---- arena -------------------------------------------------------------------

@pytest.fixture
def arena(lib):
    lay = pkv.layout(2, 2)
    ps = pkv.page_elems(lay, 16)
    a = pkv.Arena(lay, 16, 0x100000, nbytes=ps * 2 * 10 + 100)
    yield a
    a.close()


def test_arena_counts_pages_and_hands_out_lowest_first(arena):
    n, free, ps = arena.info()
    assert n == 10 and free == 10
    assert arena.take(3).tolist() == [0, 1, 2]
    assert arena.take(2).tolist() == [3, 4]
    arena.give([1, 3], defer=False)
    assert arena.take(3).tolist() == [1, 3, 5]
    assert arena.info()[1] == 4


def test_arena_short_of_pages_says_wait(arena):
    arena.take(8)
    with pytest.raises(pkv.PkvError) as e:
        arena.take(3)
    assert e.value.code == pkv.EAGAIN
    assert arena.info()[1] == 2          # nothing was taken by the refused call


def test_arena_refuses_foreign_or_double_give(arena):
    ids = arena.take(2)
    for bad in ([7], [0, 0], [-1], [10]):
        with pytest.raises(pkv.PkvError):
            arena.give(bad, defer=False)
    arena.give(ids, defer=False)
    with pytest.raises(pkv.PkvError):
        arena.give(ids, defer=False)


class FakeEvents:
    """Event operations whose completion the test controls."""

    def __init__(self):
        self.done = set()
        self.fail = set()
        self.live = set()
        self.n = 0

        def record(ctx, stream, ev):
            self.n += 1
            ev[0] = self.n
            self.live.add(self.n)
            return 0

        def query(ctx, ev):
            if ev in self.fail:
                return -1
            return 0 if ev in self.done else 1

        def destroy(ctx, ev):
            self.live.discard(ev)

        self.ops = pkv.EventOps(pkv.EventOps.RECORD(record), pkv.EventOps.QUERY(query),
                                pkv.EventOps.DESTROY(destroy), None)


def test_given_pages_return_only_after_the_stream_drains(arena):
    ev = FakeEvents()
    arena.set_event_ops(ev.ops)
    ids = arena.take(10)
    arena.give(ids[:4], stream=0x1234, defer=True)
    assert arena.info()[1] == 0                # still in flight on the stream
    with pytest.raises(pkv.PkvError) as e:
        arena.take(1)
    assert e.value.code == pkv.EAGAIN
    with pytest.raises(pkv.PkvError):
        arena.give(ids[:1], stream=0x1234)     # already pending: not held any more
    ev.done.add(1)
    assert arena.info()[1] == 4
    assert ev.live == set()                    # the event was destroyed once done
    assert arena.take(4).tolist() == [0, 1, 2, 3]


def test_failed_event_query_is_reported_and_pages_stay_out(arena):
    ev = FakeEvents()
    arena.set_event_ops(ev.ops)
    ids = arena.take(3)
    arena.give(ids, stream=0x1, defer=True)
    ev.fail.add(1)
    with pytest.raises(pkv.PkvError) as e:
        arena.take(1)
    assert e.value.code == pkv.ECUDA
    ev.fail.clear(); ev.done.add(1)
    assert arena.take(1).tolist() == [0]


def test_arena_pg_describes_the_pool(arena):
    g = arena.pg(0x5000, n_table=3)
    n, _, ps = arena.info()
    assert (g.base, g.table, g.page_elems, g.page_pos, g.n_pages, g.n_table) == \
        (0x100000, 0x5000, ps, 16, n, 3)


# ---- runs (#1170, commit 1ac2075: findRun / claimRun / releaseRun; commit
# 51f8354: mapRun refuses a run shorter than its parts) ------------------------

def test_runs_come_from_the_top_and_pages_from_the_bottom(arena):
    assert arena.run_take(3) == 7                 # pages 7, 8, 9
    assert arena.take(2).tolist() == [0, 1]
    assert arena.run_take(2) == 5                 # the next window down
    assert arena.info()[1] == 3
    assert arena.take(3).tolist() == [2, 3, 4]    # run pages are never handed out
    with pytest.raises(pkv.PkvError) as e:
        arena.take(1)
    assert e.value.code == pkv.EAGAIN


def test_fragmented_pool_makes_a_run_wait(arena):
    ids = arena.take(10)
    arena.give(ids[1::2], defer=False)            # pages 1, 3, 5, 7, 9 free
    assert arena.info()[1] == 5
    with pytest.raises(pkv.PkvError) as e:
        arena.run_take(2)
    assert e.value.code == pkv.EAGAIN
    assert arena.info()[1] == 5                   # nothing was taken
    assert arena.run_take(1) == 9
    arena.give([6], defer=False)                  # 5, 6, 7 free now
    assert arena.run_take(3) == 5


def test_run_give_takes_back_exactly_a_run_held(arena):
    first = arena.run_take(4)                     # 6 .. 9
    for f, k in ((first, 3), (first + 1, 3), (first, 5), (0, 1)):
        with pytest.raises(pkv.PkvError):
            arena.run_give(f, k, defer=False)
    with pytest.raises(pkv.PkvError):
        arena.give([first], defer=False)          # a run's page is not a KV page
    ids = arena.take(2)
    with pytest.raises(pkv.PkvError):
        arena.run_give(int(ids[0]), 2, defer=False)   # KV pages are not a run
    arena.run_give(first, 4, defer=False)
    with pytest.raises(pkv.PkvError):
        arena.run_give(first, 4, defer=False)     # not held any more
    assert arena.info()[1] == 8
    assert arena.run_take(8) == 2


def test_run_returns_only_after_the_stream_drains(arena):
    ev = FakeEvents()
    arena.set_event_ops(ev.ops)
    first = arena.run_take(10)
    assert first == 0
    arena.run_give(first, 10, stream=0x77, defer=True)
    with pytest.raises(pkv.PkvError) as e:
        arena.run_take(1)
    assert e.value.code == pkv.EAGAIN
    with pytest.raises(pkv.PkvError):
        arena.run_give(first, 10, defer=False)    # pending: not held
    ev.done.add(1)
    assert arena.info()[1] == 10
    assert ev.live == set()
    assert arena.take(1).tolist() == [0]


def test_run_pages_round_up_to_whole_pages(arena):
    _, _, ps = arena.info()
    page_bytes = 2 * ps
    for nbytes, k in ((0, 0), (1, 1), (page_bytes, 1), (page_bytes + 1, 2), (5 * page_bytes, 5)):
        assert arena.run_pages(nbytes) == k


def test_run_map_lays_parts_in_order_and_refuses_a_short_run(arena):
    _, _, ps = arena.info()
    page_bytes = 2 * ps
    first = arena.run_take(2)
    lo = 0x100000 + first * page_bytes
    parts = [100, 1000, 7, page_bytes]
    ptrs = arena.run_map(first, 2, parts, align=256)
    expect, cur = [], lo
    for b in parts:
        cur = -(-cur // 256) * 256
        expect.append(cur)
        cur += b
    assert ptrs == expect
    assert all(p % 256 == 0 for p in ptrs)
    assert ptrs[-1] + parts[-1] <= lo + 2 * page_bytes
    # exactly filling the run is fine; one byte more is refused
    assert arena.run_map(first, 2, [2 * page_bytes], align=16) == [lo]
    with pytest.raises(pkv.PkvError):
        arena.run_map(first, 2, [2 * page_bytes + 1], align=16)
    with pytest.raises(pkv.PkvError):
        arena.run_map(first, 2, [page_bytes, page_bytes], align=4096)   # padding pushes it out
    for align in (8, 24, 8192):
        with pytest.raises(pkv.PkvError):
            arena.run_map(first, 2, [16], align=align)
    with pytest.raises(pkv.PkvError):
        arena.run_map(first, 1, [16])             # not the run as taken


class PoolModel:
    """Brute-force model of the pool: a set of free ids.  KV pages: the n
    lowest free ids.  A run: the largest first id whose k pages are all
    free.  Releases take effect at once (no deferral)."""

    def __init__(self, n):
        self.n = n
        self.free = set(range(n))
        self.runs = {}

    def take(self, k):
        if k > len(self.free):
            return None
        ids = sorted(self.free)[:k]
        self.free -= set(ids)
        return ids

    def run_take(self, k):
        for first in range(self.n - k, -1, -1):
            if all(i in self.free for i in range(first, first + k)):
                self.free -= set(range(first, first + k))
                self.runs[first] = k
                return first
        return None


def test_pool_follows_the_brute_force_model_over_random_operations(lib):
    lay = pkv.layout(1, 1, 256, 0)
    ps = pkv.page_elems(lay, 4)
    rng = np.random.default_rng(5)
    for trial in range(6):
        n = int(rng.integers(5, 60))
        a = pkv.Arena(lay, 4, 0x200000, nbytes=ps * 2 * n)
        m = PoolModel(n)
        held_pages, held_runs = [], []
        try:
            for _ in range(400):
                op = rng.integers(0, 4)
                if op == 0:
                    k = int(rng.integers(1, 6))
                    want = m.take(k)
                    if want is None:
                        with pytest.raises(pkv.PkvError) as e:
                            a.take(k)
                        assert e.value.code == pkv.EAGAIN
                    else:
                        assert a.take(k).tolist() == want
                        held_pages += want
                elif op == 1:
                    k = int(rng.integers(1, 8))
                    want = m.run_take(k)
                    if want is None:
                        with pytest.raises(pkv.PkvError) as e:
                            a.run_take(k)
                        assert e.value.code == pkv.EAGAIN
                    else:
                        assert a.run_take(k) == want
                        held_runs.append((want, k))
                elif op == 2 and held_pages:
                    pick = rng.permutation(len(held_pages))[: int(rng.integers(1, len(held_pages) + 1))]
                    ids = [held_pages[i] for i in pick]
                    a.give(ids, defer=False)
                    m.free |= set(ids)
                    held_pages = [x for i, x in enumerate(held_pages) if i not in set(pick.tolist())]
                elif op == 3 and held_runs:
                    first, k = held_runs.pop(int(rng.integers(0, len(held_runs))))
                    a.run_give(first, k, defer=False)
                    m.free |= set(range(first, first + k))
                    del m.runs[first]
                assert a.info()[1] == len(m.free)
        finally:
            a.close()


# ---- e4m3 K/V format (#1170, commit 5c09685) -------------------------------

def test_e4m3_page_elems_match_oracle(lib, orc):
    for hkv, di, ptok in [(2, 128, 256), (4, 0, 256), (1, 128, 16), (2, 128, 4)]:
        lay = pkv.layout(13, hkv, 256, di, pkv.KV_E4M3)
        assert pkv.page_elems(lay, ptok) == \
            orc.page_elems(orc.Shape(13, hkv, 256, di, orc.E4M3), ptok)


@pytest.mark.parametrize("ptok", [4, 16, 48, 256])
def test_host_pg_at_gives_e4m3_byte_offsets_of_the_oracle(lib, orc, ptok):
    lay = pkv.layout(3, 2, 256, 128, pkv.KV_E4M3)
    shape = orc.Shape(3, 2, 256, 128, orc.E4M3)
    ps = pkv.page_elems(lay, ptok)
    n_pages = 40
    table = synth.shuffled_tables(ptok + 1, n_pages, [7])[0]
    oc = orc.Cache(np.zeros(1, np.uint16), ptok, ps, table, n_pages)
    g = pkv.pg(0x10000, 0x20000, ps, ptok, n_pages, table.size)
    rng = np.random.default_rng(ptok + 1)
    for _ in range(400):
        layer = int(rng.integers(3)); kind = int(rng.integers(6)); head = int(rng.integers(2))
        if kind in (pkv.IK, pkv.P):
            head = 0
        pos = int(rng.integers(7 * ptok // 4 if kind == pkv.P else 7 * ptok))
        assert pkv.pg_row(lay, g, table, layer, kind, head, pos) == \
            orc.row8(shape, oc, layer, kind, head, pos)


def test_e4m3_refusals_before_launch(lib):
    lay8 = pkv.layout(1, 2, 256, 128, pkv.KV_E4M3)
    with pytest.raises(pkv.PkvError) as e:     # the tensor-core prefill reads bf16 rows
        pkv.prefill_ws_size(lay8, [_seq(lay8, length=64, n_new=8)], 16)
    assert e.value.code == pkv.EINVAL
    with pytest.raises(pkv.PkvError) as e:     # scales exist only in the e4m3 format
        pkv.pg_row(pkv.layout(1, 2), pkv.pg(0x10000, None, pkv.page_elems(pkv.layout(1, 2), 16), 16),
                   None, 0, pkv.KS, 0, 0)
    assert e.value.code == pkv.EINVAL
    with pytest.raises(pkv.PkvError) as e:     # an unknown format
        pkv.page_elems(pkv.layout(1, 2, 256, 128, 2), 16)
    assert e.value.code == pkv.EINVAL
