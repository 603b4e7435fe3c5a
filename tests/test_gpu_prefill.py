"""GPU parity: chunked prefill on the tensor cores against the oracle.

A chunk of new positions is stored (pkv_store) and its queries attend the
cached context plus the chunk, causally.  Every row is checked against the
float64 oracle where the oracle finishes in seconds; the pages' chunk (512
queries appended to 31,000 cached positions, pages of 256) is checked on
sampled rows.  Paged output must equal contiguous output bit for bit, and a
chunk of a few queries must agree with the decode kernel.
"""
import numpy as np
import pytest

import oracle as orc
from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import dev_u16, host_u16, oracle_decode, place, torch, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def _prefill(pl, lens, n_new, layer, hq, q_list):
    t = torch()
    seqs = pl.seqs(lens, n_new)
    q = dev_u16(np.concatenate(q_list))
    out = t.zeros_like(q)
    ws = t.zeros(max(64, pkv.prefill_ws_size(pl.lay, seqs, hq) // 4 + 64), dtype=t.float32,
                 device="cuda")
    status = t.zeros(1, dtype=t.int32, device="cuda")
    pkv.prefill(pl.lay, seqs, layer, hq, q, out, ws, status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    return host_u16(out)


@pytest.mark.parametrize("ptok", [16, 48, 256, None, 20])
def test_small_chunks_match_oracle_and_contiguous(ptok):
    lay = pkv.layout(2, 2, 256, 128)
    lens = [140, 77]            # cached + chunk
    n_new = [40, 77]            # the second stream is all chunk (a prompt from scratch)
    streams = [synth.make_stream(1200 + i, 2, T, 2, 256, 128) for i, T in enumerate(lens)]
    q = [synth.queries(1300 + i, n, 16, 256) for i, n in enumerate(n_new)]
    if ptok is None:
        pl = place(lay, streams, None)
    else:
        pl = place(lay, streams, ptok, seed=ptok)
    got = _prefill(pl, lens, n_new, 1, 16, q)
    ok, report = within_tol(got, oracle_decode(pl, 1, 16, q))
    assert ok, report
    cont = place(lay, streams, None)
    assert np.array_equal(_prefill(cont, lens, n_new, 1, 16, q), got)


@pytest.mark.parametrize("ptok", [4, 8])
def test_small_pages_many_pages_a_tile(ptok):
    # Pages of 4 and 8 positions: a 64-key tile spans 9 to 17 pages, so the
    # producers' 64-page window of ids slides within the split, and every
    # tile goes key by key.  Lengths give splits and a ragged tail.
    lay = pkv.layout(1, 2, 256, 128)
    lens = [1500, 644]
    n_new = [36, 100]
    streams = [synth.make_stream(1800 + i, 1, T, 2, 256, 128) for i, T in enumerate(lens)]
    q = [synth.queries(1900 + i, n, 16, 256) for i, n in enumerate(n_new)]
    pl = place(lay, streams, ptok, seed=ptok)
    got = _prefill(pl, lens, n_new, 0, 16, q)
    ok, report = within_tol(got, oracle_decode(pl, 0, 16, q))
    assert ok, report
    cont = place(lay, streams, None)
    assert np.array_equal(_prefill(cont, lens, n_new, 0, 16, q), got)


def test_prefill_of_a_short_window_agrees_with_decode():
    t = torch()
    lay = pkv.layout(1, 2, 256, 128)
    lens = [300, 1000]
    streams = [synth.make_stream(1400 + i, 1, T, 2, 256, 128) for i, T in enumerate(lens)]
    q = [synth.queries(1500 + i, 4, 16, 256) for i in range(2)]
    pl = place(lay, streams, 128, seed=3)
    a = _prefill(pl, lens, [4, 4], 0, 16, q)
    seqs = pl.seqs(lens, [4, 4])
    dq = dev_u16(np.concatenate(q))
    out = t.zeros_like(dq)
    ws = t.zeros(pkv.decode_ws_size(lay, seqs, 16) // 4 + 64, dtype=t.float32, device="cuda")
    pkv.decode(lay, seqs, 0, 16, dq, out, ws)
    t.cuda.synchronize()
    b = host_u16(out)
    ref = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok, report = within_tol(a, ref)
    assert ok, report
    ok, report = within_tol(a, oracle_decode(pl, 0, 16, q))
    assert ok, report


def test_group_sizes_other_than_eight():
    lay = pkv.layout(1, 4, 256, 0)
    T, C = 96, 96
    streams = [synth.Stream(T, synth.normal_bf16(1600, (1, T, 4, 256)),
                            synth.normal_bf16(1601, (1, T, 4, 256)), np.zeros((1, T, 0), np.uint16))]
    q = [synth.queries(1602, C, 8, 256)]   # G = 2
    pl = place(lay, streams, 32, seed=5)
    got = _prefill(pl, [T], [C], 0, 8, q)
    ok, report = within_tol(got, oracle_decode(pl, 0, 8, q))
    assert ok, report


def test_pages_chunk_31000_plus_512_sampled():
    # 1 stream, 512 queries appended to 31,000 cached positions, pages of 256
    lay = pkv.layout(1, 2, 256, 128)
    P0, C = 31000, 512
    T = P0 + C
    s = synth.make_stream(1700, 1, T, 2, 256, 128)
    q = synth.queries(1701, C, 16, 256)
    pl = place(lay, [s], 256, seed=6)
    got = _prefill(pl, [T], [C], 0, 16, [q]).reshape(C, 16, 256)
    rng = np.random.default_rng(7)
    picks = [(0, 0), (C - 1, 15), (255, 7), (256, 8)] + \
        [(int(rng.integers(C)), int(rng.integers(16))) for _ in range(12)]
    for j, h in picks:
        ref = orc.attend_row(pl.shape, pl.ocaches[0], 0, 16, h, P0 + j, q[j, h])
        ok, report = within_tol(got[j, h], ref)
        assert ok, (j, h, report)
    cont = place(lay, [s], None)
    assert np.array_equal(_prefill(cont, [T], [C], 0, 16, [q]).reshape(C, 16, 256), got)



def _bf16_bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0] >> 16)


def _prefill_status(pl, lens, n_new, layer, hq, q_list):
    t = torch()
    seqs = pl.seqs(lens, n_new)
    q = dev_u16(np.concatenate(q_list))
    out = t.zeros_like(q)
    ws = t.zeros(max(64, pkv.prefill_ws_size(pl.lay, seqs, hq) // 4 + 64), dtype=t.float32,
                 device="cuda")
    status = t.zeros(1, dtype=t.int32, device="cuda")
    pkv.prefill(pl.lay, seqs, layer, hq, q, out, ws, status=status)
    t.cuda.synchronize()
    return host_u16(out), int(status.item())


@pytest.mark.parametrize("ptok", [16, 48, 256, None, 20])
def test_fp16_v_chunks_match_oracle_and_contiguous(ptok):
    # chunks of more than 32 queries and at least 8 M-tiles a KV head in
    # every stream: the PV product runs in fp16 on V rows converted once
    lay = pkv.layout(2, 2, 256, 128)
    lens = [460, 150]
    n_new = [130, 150]          # 1,040 and 1,200 query columns a KV head
    streams = [synth.make_stream(1900 + i, 2, T, 2, 256, 128) for i, T in enumerate(lens)]
    q = [synth.queries(1910 + i, n, 16, 256) for i, n in enumerate(n_new)]
    pl = place(lay, streams, ptok, seed=9) if ptok else place(lay, streams, None)
    got = _prefill(pl, lens, n_new, 1, 16, q)
    ok, report = within_tol(got, oracle_decode(pl, 1, 16, q))
    assert ok, report
    cont = place(lay, streams, None)
    assert np.array_equal(_prefill(cont, lens, n_new, 1, 16, q), got)


@pytest.mark.parametrize("big, n_new, reported", [(65280.0, 128, False), (131072.0, 128, True),
                                                  (131072.0, 60, False)])
def test_v_at_and_beyond_fp16_range(big, n_new, reported):
    # A chunk of 128 queries (8 M-tiles a KV head) runs the PV product in
    # fp16.  65,280 is the largest bf16 value fp16 holds exactly: the rows
    # stay within tolerance and nothing is reported.  2^17 overflows fp16:
    # the kernel reports a non-finite accumulator.  A chunk of 60 queries
    # keeps bf16 V: 2^17 is an ordinary value there.
    lay = pkv.layout(1, 2, 256, 128)
    T = 400
    s = synth.make_stream(1800, 1, T, 2, 256, 128)
    v = s.v.copy()
    v[0, 37, 1, 5] = _bf16_bits(big)
    v[0, 350, 0, 200] = _bf16_bits(-big)
    s = synth.Stream(T, s.k, v, s.ik)
    q = synth.queries(1801, n_new, 16, 256)
    pl = place(lay, [s], 48, seed=8)
    got, st = _prefill_status(pl, [T], [n_new], 0, 16, [q])
    assert bool(st & pkv.DEV_RANGE) == reported, st
    assert st & ~pkv.DEV_RANGE == 0, st
    if not reported:
        ok, report = within_tol(got, oracle_decode(pl, 0, 16, [q]))
        assert ok, report


def test_fp16_v_mode_starts_at_eight_m_tiles():
    # 250 positions: one split, so the workspace holds no partials, only the
    # fp16 V mode's converted rows (2 KV heads x 256 padded keys x 512 B).
    # 113 queries are 904 query columns a KV head (8 M-tiles): the mode
    # applies; 112 are 896 (7 M-tiles): bf16 V, no workspace.  Both match
    # the oracle.
    lay = pkv.layout(1, 2, 256, 128)
    T = 250
    s = synth.make_stream(2000, 1, T, 2, 256, 128)
    pl = place(lay, [s], 48, seed=10)
    assert pkv.prefill_ws_size(pl.lay, pl.seqs([T], [113]), 16) == 2 * 256 * 512
    assert pkv.prefill_ws_size(pl.lay, pl.seqs([T], [112]), 16) == 0
    for n in (112, 113):
        q = synth.queries(2001, n, 16, 256)
        got = _prefill(pl, [T], [n], 0, 16, [q])
        ok, report = within_tol(got, oracle_decode(pl, 0, 16, [q]))
        assert ok, (n, report)
