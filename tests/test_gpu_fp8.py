"""GPU parity for the e4m3 K/V format (TensorFold #1170, commit 5c09685:
each K and V row is its e4m3 codes and a float32 scale, found through the
page table; the reference dequantizes code x scale in float64).

Bars: the store's bytes (codes, scales, indexer rows) equal the oracle's
quantization bit for bit; gathered codes and scales equal the oracle's;
decode rows are within |gpu - ref| <= 1e-3 + 2e-3 |ref| (+ half a bf16 ulp)
of the float64 dequantizing oracle; paged output equals contiguous output
bit for bit; a decode that stores its new rows itself leaves the bytes of
the store and gives the outputs of a store and a decode; pooling and block
scores on an e4m3 layout equal the oracle's bits; calls the format does not
support refuse it.
"""
import numpy as np
import pytest

import oracle as orc
from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import decode, dev_u16, host_u16, oracle_decode, place, torch, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def _lay(n_layers=2, hkv=2, di=128):
    return pkv.layout(n_layers, hkv, 256, di, pkv.KV_E4M3)


def _streams(lens, n_layers=2, hkv=2, seed=0, di=128):
    return [synth.make_stream(seed + i, n_layers, T, hkv, 256, di) for i, T in enumerate(lens)]


@pytest.mark.parametrize("ptok", [16, 48, 256, None, 20])
def test_e4m3_store_bytes_equal_oracle(ptok):
    lay = _lay()
    streams = _streams([140, 77, 300], seed=2000)
    pl = place(lay, streams, ptok, seed=3)
    for i in range(len(pl.buffers)):
        assert np.array_equal(host_u16(pl.body(i)), pl.oarenas[i])
    assert pl.guards_intact()


@pytest.mark.parametrize("hkv", [2, 3, 8])
def test_e4m3_gather_codes_and_scales_equal_oracle(hkv):
    # 3 and 8 KV heads: a gather lane takes several heads (16 lanes a head's
    # 256 code bytes, heads two apart)
    t = torch()
    lay = _lay(hkv=hkv)
    lens = [300, 77]
    streams = _streams(lens, hkv=hkv, seed=2100 + hkv)
    pl = place(lay, streams, 48, seed=4)
    seqs = pl.seqs(lens, [0, 0])
    for layer in range(2):
        for kind in (pkv.K, pkv.V):
            out = t.empty((sum(lens), hkv, 256), dtype=t.uint8, device="cuda")
            pkv.gather(lay, seqs, layer, kind, out)
            want = np.concatenate([orc.get_rows8(pl.shape, oc, layer, kind, 0, T)
                                   for oc, T in zip(pl.ocaches, lens)])
            assert np.array_equal(out.cpu().numpy(), want)
        for kind in (pkv.KS, pkv.VS):
            out = t.empty((sum(lens), hkv), dtype=t.float32, device="cuda")
            pkv.gather(lay, seqs, layer, kind, out)
            want = np.concatenate([orc.get_rows8(pl.shape, oc, layer, kind, 0, T)
                                   for oc, T in zip(pl.ocaches, lens)])
            assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


MULTI = [L + 1 for L in (1000, 3000, 6000, 9000)]


@pytest.fixture(scope="module")
def multi8():
    lay = _lay(2, 2, 128)
    streams = _streams(MULTI, seed=2200)
    q = [synth.queries(2300 + i, 1, 16, 256) for i in range(4)]
    cont = place(lay, streams, None)
    return lay, streams, q, oracle_decode(cont, 1, 16, q), decode(cont, 1, 16, q)


def test_e4m3_multi_stream_decode_within_oracle_bound(multi8):
    lay, streams, q, ref, base = multi8
    ok, report = within_tol(base, ref)
    assert ok, report


@pytest.mark.parametrize("ptok", [16, 48, 128, 256, 512])
def test_e4m3_paged_decode_bit_identical_to_contiguous(multi8, ptok):
    lay, streams, q, ref, base = multi8
    pl = place(lay, streams, ptok, seed=ptok)
    assert np.array_equal(decode(pl, 1, 16, q), base)


def test_e4m3_stream_alone_equals_stream_in_batch(multi8):
    lay, streams, q, ref, base = multi8
    rows = np.split(base, 4)
    for i in (0, 3):
        pl = place(lay, streams[i:i + 1], 48, seed=9 + i)
        assert np.array_equal(decode(pl, 1, 16, q[i:i + 1]), rows[i])


@pytest.mark.parametrize("nq,hq,hkv", [(4, 16, 2), (2, 8, 4), (1, 4, 1), (3, 16, 2)])
def test_e4m3_draft_windows_and_group_sizes(nq, hq, hkv):
    lay = _lay(1, hkv, 0)
    lens = [700, 1501, 33]
    streams = _streams(lens, 1, hkv, seed=2400 + nq, di=0)
    q = [synth.queries(2500 + i, nq, hq, 256) for i in range(len(lens))]
    pl = place(lay, streams, 16, seed=nq)
    got = decode(pl, 0, hq, q)
    ok, report = within_tol(got, oracle_decode(pl, 0, hq, q))
    assert ok, report
    cont = place(lay, streams, None)
    assert np.array_equal(decode(cont, 0, hq, q), got)


@pytest.mark.parametrize("length", [1, 2, 15, 16, 17, 255, 257, 1023])
def test_e4m3_ragged_lengths(length):
    lay = _lay(1, 2, 128)
    streams = _streams([length], 1, seed=2600 + length)
    q = [synth.queries(2700 + length, 1, 16, 256)]
    pl = place(lay, streams, 48, seed=length)
    ok, report = within_tol(decode(pl, 0, 16, q), oracle_decode(pl, 0, 16, q))
    assert ok, report


def test_e4m3_pool_and_scores_bit_identical_to_oracle():
    t = torch()
    lay = _lay(1, 2, 128)
    lens = [9000, 1001]
    streams = _streams(lens, 1, seed=2800)
    pl = place(lay, streams, 128, seed=1)
    pkv.pool(lay, pl.seqs(lens, lens), 0)
    for oc, T in zip(pl.ocaches, lens):
        orc.pool(pl.shape, oc, 0, 0, T // 4)
    t.cuda.synchronize()
    assert np.array_equal(host_u16(pl.body(0)), pl.oarenas[0])
    qi = [synth.queries(2900 + i, 1, 16, 128) for i in range(2)]
    ld = 2250
    sc = t.empty((2, 16, ld), dtype=t.float32, device="cuda")
    pkv.block_scores(lay, pl.seqs(lens, [1, 1]), 0, 16, dev_u16(np.concatenate(qi)), sc, ld)
    t.cuda.synchronize()
    got = sc.cpu().numpy()
    for i, (oc, T) in enumerate(zip(pl.ocaches, lens)):
        ref = orc.scores(pl.shape, oc, 0, 16, T, qi[i][0])
        assert np.array_equal(got[i, :, :T // 4].view(np.uint32), ref.view(np.uint32))


def test_e4m3_decode_static_matches_decode(multi8):
    t = torch()
    lay, streams, q, ref, base = multi8
    pl = place(lay, streams, 256, seed=2)
    dq = dev_u16(np.concatenate(q))
    out = t.zeros_like(dq)
    pkv.decode_static(lay, pl.seqs(MULTI, [1] * 4), 1, 16, dq, out)
    t.cuda.synchronize()
    assert np.array_equal(host_u16(out), base)


@pytest.mark.parametrize("ptok", [16, 48, None])
def test_e4m3_fused_store_decode_equals_store_then_decode(ptok):
    # The decode call quantizes and stores its new rows itself: the cache
    # bytes equal the oracle's placement (so pkv_store's quantization, bit for
    # bit) and the outputs equal a pkv_store followed by a pkv_decode.
    # Lengths put a split boundary (multiples of 256 keys) inside the
    # 4-token window of the first stream.
    t = torch()
    lay = _lay()
    lens = [258, 516, 1000, 37]
    nq, layer = 4, 1
    full = _streams(lens, seed=3100)
    q = [synth.queries(3150 + i, nq, 16, 256) for i in range(len(lens))]
    kn = dev_u16(np.concatenate([s.k[layer][-nq:] for s in full]))
    vn = dev_u16(np.concatenate([s.v[layer][-nq:] for s in full]))
    ikn = dev_u16(np.concatenate([s.ik[layer][-nq:] for s in full]))
    dq = dev_u16(np.concatenate(q))
    outs = []
    for fused in (False, True):
        pl = place(lay, full, ptok, seed=9)
        # blank the window's K/V codes, scales and indexer rows (0x7f: an
        # e4m3 NaN code, a huge scale)
        for i, T in enumerate(lens):
            body = pl.body(0 if ptok else i)
            tab = pl.tables[i] if ptok else None
            b8 = body.view(t.uint8)
            for p in range(T - nq, T):
                for kind, heads, nbytes in ((pkv.K, 2, 256), (pkv.V, 2, 256), (pkv.KS, 2, 4),
                                            (pkv.VS, 2, 4)):
                    for h in range(heads):
                        off = pkv.pg_row(lay, pl.pgs[i], tab, layer, kind, h, p)
                        b8[off:off + nbytes] = 0x7f
                off = pkv.pg_row(lay, pl.pgs[i], tab, layer, pkv.IK, 0, p)
                b8[off:off + 256] = 0x7f
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
        for i in range(len(pl.buffers)):
            assert np.array_equal(host_u16(pl.body(i)), pl.oarenas[i])
        assert pl.guards_intact()
    assert np.array_equal(outs[0], outs[1])
    ref_pl = place(lay, full, None)
    ok, worst = within_tol(outs[1], oracle_decode(ref_pl, layer, 16, q))
    assert ok, worst


def test_e4m3_refuses_sparse():
    t = torch()
    lay = _lay(1, 2, 128)
    streams = _streams([64], 1, seed=3000)
    pl = place(lay, streams, 16, seed=1)
    seqs = pl.seqs([64], [1])
    q = t.zeros((1, 16, 256), dtype=t.int16, device="cuda")
    ws = t.zeros(1 << 16, dtype=t.float32, device="cuda")
    ids = t.zeros((1, 16, 4), dtype=t.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.sparse_decode(lay, seqs, 0, 16, q, ids, 4, t.zeros_like(q), ws)
    assert e.value.code == pkv.EINVAL
