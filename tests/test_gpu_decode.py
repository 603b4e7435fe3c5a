"""GPU parity: decode attention (split-KV partials + combine) against the oracle.

Bars: every output row within |gpu - ref| <= 1e-3 + 2e-3 |ref| of the
float64 oracle; paged output bit-identical to contiguous output at every
page size and over three repeats; a stream's output in a batch
bit-identical to its output alone; red controls go red.
"""
import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import decode, dev_u16, host_u16, oracle_decode, place, torch, within_tol

pytestmark = pytest.mark.gpu

PAGES = [16, 48, 128, 256, 512]
MULTI_LENS = [1000, 3000, 6000, 9000]    # cached before the new token


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def _streams(lens, n_layers, hkv, seed=0):
    return [synth.make_stream(seed + i, n_layers, T, hkv, 256, 128) for i, T in enumerate(lens)]


def test_tiny_reversed_table_decode():
    # 1 layer, 1 stream, 4 query / 1 KV head, 64 cached positions, pages of 16
    # read through a reversed table; one query token attends all 64 keys.
    lay = pkv.layout(1, 1, 256, 128)
    s = _streams([64], 1, 1)
    q = [synth.queries(0, 1, 4, 256)]
    paged = place(lay, s, 16, tables=[synth.reversed_table(4)], spare_pages=0)
    cont = place(lay, s, None)
    a = decode(paged, 0, 4, q, n_new=[1])
    b = decode(cont, 0, 4, q, n_new=[1])
    assert np.array_equal(a, b)
    ok, worst = within_tol(a, oracle_decode(cont, 0, 4, q))
    assert ok, worst


@pytest.fixture(scope="module")
def multi():
    """Config of the benchmark: 4 streams, 16/2 heads, the new token stored then read."""
    lay = pkv.layout(2, 2, 256, 128)
    lens = [L + 1 for L in MULTI_LENS]
    streams = _streams(lens, 2, 2, seed=100)
    q = [synth.queries(200 + i, 1, 16, 256) for i in range(4)]
    cont = place(lay, streams, None)
    ref = oracle_decode(cont, 1, 16, q)
    base = decode(cont, 1, 16, q)
    return lay, streams, q, ref, base


def test_multi_stream_contiguous_within_oracle_bound(multi):
    lay, streams, q, ref, base = multi
    ok, worst = within_tol(base, ref)
    assert ok, worst


@pytest.mark.parametrize("ptok", PAGES)
def test_multi_stream_paged_bit_identical_to_contiguous(multi, ptok):
    lay, streams, q, ref, base = multi
    pl = place(lay, streams, ptok, seed=ptok)
    for _ in range(3):
        assert np.array_equal(decode(pl, 1, 16, q), base)
    assert pl.guards_intact()


def test_stream_alone_equals_stream_in_batch(multi):
    lay, streams, q, ref, base = multi
    pl = place(lay, streams, 48, seed=1)
    rows = np.split(base, 4)
    for i in range(4):
        sub = place(lay, [streams[i]], 48, seed=50 + i)
        assert np.array_equal(decode(sub, 1, 16, [q[i]]), rows[i])


def test_red_every_stream_given_stream_zeros_table(multi):
    lay, streams, q, ref, base = multi
    pl = place(lay, [streams[0], streams[0]], 128, seed=3)
    # both entries carry stream 0's table while the second query is stream 1's
    out = decode(pl, 1, 16, [q[0], q[1]], lens=[streams[0].length] * 2)
    ok, _ = within_tol(out[1], ref[1])
    assert not ok
    ok0, worst = within_tol(out[0], ref[0])
    assert ok0, worst


@pytest.mark.parametrize("nq,hq,hkv", [(4, 16, 2), (2, 16, 2), (4, 8, 2), (1, 2, 2),
                                       (3, 4, 1), (32, 2, 2)])
def test_draft_window_causal_decode(nq, hq, hkv):
    lay = pkv.layout(1, hkv, 256, 128)
    lens = [700 + nq, 97, 16 + nq, nq]
    streams = _streams(lens, 1, hkv, seed=300 + nq)
    q = [synth.queries(400 + i, nq, hq, 256) for i in range(len(lens))]
    cont = place(lay, streams, None)
    ref = oracle_decode(cont, 0, hq, q)
    a = decode(cont, 0, hq, q)
    ok, worst = within_tol(a, ref)
    assert ok, worst
    pl = place(lay, streams, 16, seed=nq)
    assert np.array_equal(decode(pl, 0, hq, q), a)


def test_draft_windows_alone_equal_windows_in_batch():
    # Windows of 4 queries x 8 heads (32 columns a unit) run on the tensor
    # cores, with the work items of the longest splits launched first across
    # streams: a stream's output must not depend on the streams beside it.
    lay = pkv.layout(1, 2, 256, 128)
    lens = [900 + 4, 5000 + 4, 2600 + 4]
    streams = _streams(lens, 1, 2, seed=700)
    q = [synth.queries(710 + i, 4, 16, 256) for i in range(3)]
    pl = place(lay, streams, 48, seed=7)
    both = decode(pl, 0, 16, q)
    ok, worst = within_tol(both, oracle_decode(place(lay, streams, None), 0, 16, q))
    assert ok, worst
    rows = np.split(both, 3)
    for i in range(3):
        sub = place(lay, [streams[i]], 48, seed=720 + i)
        assert np.array_equal(decode(sub, 0, 16, [q[i]]), rows[i])


@pytest.mark.parametrize("length", [1, 2, 15, 16, 17, 127, 128, 129, 4095, 40960])
def test_ragged_lengths(length):
    lay = pkv.layout(1, 2, 256, 0)
    streams = [synth.Stream(length, synth.normal_bf16(length, (1, length, 2, 256)),
                            synth.normal_bf16(length + 1, (1, length, 2, 256)),
                            np.zeros((1, length, 0), np.uint16))]
    q = [synth.queries(length, 1, 16, 256)]
    pl = place(lay, streams, 256 if length > 1000 else 16, seed=length)
    a = decode(pl, 0, 16, q)
    if length <= 4095:
        ok, worst = within_tol(a, oracle_decode(pl, 0, 16, q))
        assert ok, worst
    else:
        # 40,960 keys: sample rows the oracle computes one at a time
        import oracle as orc
        for h in (0, 7, 8, 15):
            ref = orc.attend_row(pl.shape, pl.ocaches[0], 0, 16, h, length - 1, q[0][0, h])
            ok, worst = within_tol(a[0, h], ref)
            assert ok, worst


def test_sixty_four_streams_in_one_launch():
    # The most streams a launch takes, every one with its own table and
    # length (ragged, 1 to 300 positions), pages of 16 through one arena:
    # each row within the oracle's bound, paged bits equal to contiguous.
    lay = pkv.layout(1, 2, 256, 128)
    lens = [1 + (37 * i) % 300 for i in range(64)]
    streams = _streams(lens, 1, 2, seed=2000)
    q = [synth.queries(2100 + i, 1, 16, 256) for i in range(64)]
    paged = place(lay, streams, 16, seed=5)
    cont = place(lay, streams, None)
    a = decode(paged, 0, 16, q)
    assert np.array_equal(a, decode(cont, 0, 16, q))
    ok, worst = within_tol(a, oracle_decode(cont, 0, 16, q))
    assert ok, worst
    assert paged.guards_intact()


def test_empty_batch_and_no_query_streams_launch_nothing():
    import oracle as orc
    t = torch()
    lay = pkv.layout(1, 2, 256, 128)
    streams = _streams([50, 60], 1, 2, seed=9)
    pl = place(lay, streams, 16)
    qh = synth.queries(1, 1, 16, 256)
    q = dev_u16(qh)
    out = t.zeros_like(q)
    ws = t.zeros(1 << 16, dtype=t.float32, device="cuda")
    pkv.decode(lay, [], 0, 16, q, out, ws)
    t.cuda.synchronize()
    assert int(t.count_nonzero(out)) == 0
    # the first stream has no new token: only the second one's query is answered
    pkv.decode(lay, pl.seqs([50, 60], [0, 1]), 0, 16, q, out, ws)
    t.cuda.synchronize()
    ok, worst = within_tol(host_u16(out), orc.attend(pl.shape, pl.ocaches[1], 0, 16, 60, qh))
    assert ok, worst


def test_status_word_stays_clear_on_good_input(multi):
    t = torch()
    lay, streams, q, ref, base = multi
    pl = place(lay, streams, 256, seed=2)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    out = decode(pl, 1, 16, q, status=status)
    assert int(status.item()) == 0
    assert np.array_equal(out, base)


@pytest.mark.parametrize("ptok", [4, 16, 48, None])
def test_fused_store_decode_equals_store_then_decode(ptok):
    # Lengths put a split boundary (multiples of 256 keys) inside the 4-token
    # window of the first stream; the second stream's window starts a split.
    from gpu_setup import CANARY
    t = torch()
    lay = pkv.layout(2, 2, 256, 128)
    lens = [258, 516, 1000, 37]
    nq, layer = 4, 1
    full = _streams(lens, 2, 2, seed=900)
    q = [synth.queries(950 + i, nq, 16, 256) for i in range(len(lens))]
    kn = dev_u16(np.concatenate([s.k[layer][-nq:] for s in full]))
    vn = dev_u16(np.concatenate([s.v[layer][-nq:] for s in full]))
    ikn = dev_u16(np.concatenate([s.ik[layer][-nq:] for s in full]))
    dq = dev_u16(np.concatenate(q))
    canary = int(np.array([CANARY], np.uint16).view(np.int16)[0])
    outs, bodies = [], []
    for fused in (False, True):
        pl = place(lay, full, ptok, seed=7)
        # blank the window rows: the call itself must write them
        for i, T in enumerate(lens):
            body = pl.body(0 if ptok else i)
            tab = pl.tables[i] if ptok else None
            for p in range(T - nq, T):
                for kind, heads, width in ((pkv.K, 2, 256), (pkv.V, 2, 256), (pkv.IK, 1, 128)):
                    for h in range(heads):
                        off = pkv.pg_row(lay, pl.pgs[i], tab, layer, kind, h, p)
                        body[off:off + width] = canary
        seqs = pl.seqs(lens, [nq] * len(lens))
        out = t.zeros_like(dq)
        ws = t.zeros(pkv.decode_ws_size(lay, seqs, 16) // 4 + 64, dtype=t.float32, device="cuda")
        if fused:
            pkv.decode(lay, seqs, layer, 16, dq, out, ws, k_new=kn, v_new=vn, ik_new=ikn)
        else:
            pkv.store(lay, seqs, layer, kn, vn, ikn)
            pkv.decode(lay, seqs, layer, 16, dq, out, ws)
        t.cuda.synchronize()
        outs.append(host_u16(out))
        bodies.append([host_u16(pl.body(i)) for i in range(len(pl.buffers))])
        # the stored bytes are the oracle's placement of the full streams
        for i in range(len(pl.buffers)):
            assert np.array_equal(bodies[-1][i], pl.oarenas[i])
        assert pl.guards_intact()
    assert np.array_equal(outs[0], outs[1])
    ref_pl = place(lay, full, None)
    ok, worst = within_tol(outs[1], oracle_decode(ref_pl, layer, 16, q))
    assert ok, worst


@pytest.mark.parametrize("ptok", [16, 256, None])
def test_token_by_token_decode_of_one_stream_and_layer(ptok):
    # Decoding in order: each call stores its token (fused) and attends it, the
    # calls queued back to back on one stream with nothing between them, so
    # each call's early reads of cached rows overlap the previous call's
    # store of the row just below its own token.  Every step's output is
    # checked against the oracle, and the cache ends as the oracle's placement.
    from gpu_setup import CANARY
    t = torch()
    lay = pkv.layout(1, 2, 256, 128)
    T0, steps, layer = 3000, 48, 0
    full = _streams([T0 + steps], 1, 2, seed=960)
    pl = place(lay, full, ptok, seed=8)
    canary = int(np.array([CANARY], np.uint16).view(np.int16)[0])
    body = pl.body(0)
    tab = pl.tables[0] if ptok else None
    for p in range(T0, T0 + steps):
        for kind, heads, width in ((pkv.K, 2, 256), (pkv.V, 2, 256), (pkv.IK, 1, 128)):
            for h in range(heads):
                off = pkv.pg_row(lay, pl.pgs[0], tab, layer, kind, h, p)
                body[off:off + width] = canary
    s = full[0]
    qs = [synth.queries(970 + j, 1, 16, 256) for j in range(steps)]
    outs = []
    ws = t.zeros(pkv.decode_ws_size(lay, pl.seqs([T0 + steps], [1]), 16) // 4 + 64,
                 dtype=t.float32, device="cuda")
    ins = [(dev_u16(s.k[layer][p:p + 1]), dev_u16(s.v[layer][p:p + 1]), dev_u16(s.ik[layer][p:p + 1]),
            dev_u16(qs[p - T0])) for p in range(T0, T0 + steps)]
    t.cuda.synchronize()
    for j, (kn, vn, ikn, dq) in enumerate(ins):
        out = t.zeros_like(dq)
        pkv.decode(lay, pl.seqs([T0 + j + 1], [1]), layer, 16, dq, out, ws, k_new=kn, v_new=vn,
                   ik_new=ikn)
        outs.append(out)
    t.cuda.synchronize()
    assert np.array_equal(host_u16(pl.body(0)), pl.oarenas[0])
    for j in range(steps):
        ref = oracle_decode(pl, layer, 16, [qs[j]], lens=[T0 + j + 1])
        ok, worst = within_tol(host_u16(outs[j]), ref)
        assert ok, (j, worst)


@pytest.mark.parametrize("ptok", [16, 256, None])
def test_decode_right_after_a_store_of_its_cached_rows(ptok):
    # A store of every row of the streams and a decode that reads those rows
    # as cached positions, back to back on one stream: the decode stages
    # cached rows before its grid-dependency wait, so the store must make its
    # rows visible before letting the decode start.  The caches are blanked
    # before each layer's store, so a row read too early shows.
    from gpu_setup import CANARY
    t = torch()
    lay = pkv.layout(4, 2, 256, 128)
    lens = [L + 1 for L in MULTI_LENS]
    streams = _streams(lens, 4, 2, seed=1300)
    q = [synth.queries(1350 + i, 1, 16, 256) for i in range(4)]
    pl = place(lay, streams, ptok, seed=3)
    canary = int(np.array([CANARY], np.uint16).view(np.int16)[0])
    seqs_all = [pkv.seq(g, L, L) for g, L in zip(pl.pgs, lens)]
    seqs = pl.seqs(lens, [1] * 4)
    dq = dev_u16(np.concatenate(q))
    ws = t.zeros(pkv.decode_ws_size(lay, seqs, 16) // 4 + 64, dtype=t.float32, device="cuda")
    for layer in range(4):
        k, v, ik = (dev_u16(np.concatenate([getattr(s, f)[layer] for s in streams]))
                    for f in ("k", "v", "ik"))
        out = t.zeros_like(dq)
        for i in range(len(pl.buffers)):
            pl.body(i).fill_(canary)
        pkv.store(lay, seqs_all, layer, k, v, ik)
        pkv.decode(lay, seqs, layer, 16, dq, out, ws)
        t.cuda.synchronize()
        ok, worst = within_tol(host_u16(out), oracle_decode(pl, layer, 16, q))
        assert ok, (layer, worst)
    assert pl.guards_intact()


def test_one_workspace_serves_calls_of_different_shapes(multi):
    # A workspace holds no state between calls: one workspace serves batches
    # of different shapes back to back (single tokens, 4-query windows, a
    # smaller batch) with the bits a fresh workspace gives.
    t = torch()
    lay, streams, q, ref, base = multi
    pl = place(lay, streams, 48, seed=11)
    lens = [s.length for s in streams]
    win = [synth.queries(300 + i, 4, 16, 256) for i in range(4)]
    calls = [(pl.seqs(lens, [1] * 4), q, 1),
             (pl.seqs(lens, [4] * 4), win, 0),
             (pl.seqs(lens[:2], [1, 1]), q[:2], 1)]
    sizes = [pkv.decode_ws_size(lay, sq, 16) for sq, _, _ in calls]
    shared = t.full((max(sizes) // 4 + 64,), float("nan"), dtype=t.float32, device="cuda")
    for _ in range(2):
        for (sq, ql, layer), size in zip(calls, sizes):
            dq = dev_u16(np.concatenate(ql))
            fresh = t.empty(size // 4 + 64, dtype=t.float32, device="cuda")
            a, b = t.zeros_like(dq), t.zeros_like(dq)
            pkv.decode(lay, sq, layer, 16, dq, a, shared)
            pkv.decode(lay, sq, layer, 16, dq, b, fresh)
            t.cuda.synchronize()
            assert t.equal(a, b)
