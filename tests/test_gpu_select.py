"""GPU parity: block scores and top-k (bit for bit) and block-sparse decode.

The sparse case of the benchmark: 2 streams of 9,000 cached positions in
pages of 128, 16 query / 2 KV heads, indexer keys of 128 pooled in blocks
of 4, block score = indexer query . pooled row, top-64 blocks per head,
attention over the selected blocks only.
"""
import numpy as np
import pytest

import oracle as orc
from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import dev_u16, host_u16, place, torch, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def _pooled(lens, ptok, seed=0, hkv=2):
    lay = pkv.layout(1, hkv, 256, 128)
    streams = [synth.make_stream(seed + i, 1, T, hkv, 256, 128) for i, T in enumerate(lens)]
    pl = place(lay, streams, ptok, seed=seed)
    pkv.pool(lay, pl.seqs(lens, lens), 0)
    for oc, T in zip(pl.ocaches, lens):
        orc.pool(pl.shape, oc, 0, 0, T // 4)
    torch().cuda.synchronize()
    return lay, pl


def _scores(lay, pl, lens, hq, seed, ld=None):
    t = torch()
    qi = [synth.queries(seed + i, 1, hq, 128) for i in range(len(lens))]
    ld = ld or max(T // 4 for T in lens)
    sc = t.empty((len(lens), hq, ld), dtype=t.float32, device="cuda")
    pkv.block_scores(lay, pl.seqs(lens, [1] * len(lens)), 0, hq, dev_u16(np.concatenate(qi)), sc, ld)
    t.cuda.synchronize()
    ref = [orc.scores(pl.shape, oc, 0, hq, T, q[0]) for oc, T, q in zip(pl.ocaches, lens, qi)]
    return sc.cpu().numpy(), ref, qi


@pytest.mark.parametrize("ptok", [16, 48, 128])
def test_block_scores_bit_identical_to_oracle(ptok):
    lens = [9000, 1001, 7]
    lay, pl = _pooled(lens, ptok, seed=ptok)
    sc, ref, _ = _scores(lay, pl, lens, 16, seed=ptok + 1, ld=2300)
    for i, T in enumerate(lens):
        nb = T // 4
        assert np.array_equal(sc[i, :, :nb].view(np.uint32), ref[i].view(np.uint32))
        assert np.isneginf(sc[i, :, nb:]).all()


def _topk(sc, lens, hq, k):
    t = torch()
    ld = sc.shape[2]
    dsc = t.from_numpy(np.ascontiguousarray(sc)).cuda()
    ids = t.empty((len(lens), hq, k), dtype=t.int32, device="cuda")
    seqs = [pkv.seq(pkv.pg(0x100, None, 0, 4), L, 1) for L in lens]
    pkv.topk(seqs, hq, dsc, ld, k, ids)
    t.cuda.synchronize()
    return ids.cpu().numpy()


@pytest.mark.parametrize("k", [1, 8, 64, 256])
def test_topk_ids_bit_identical_to_oracle(k):
    rng = np.random.default_rng(k)
    lens = [9000, 2001, 64, 3, 900]
    hq = 4
    ld = 2250
    sc = rng.standard_normal((len(lens), hq, ld)).astype(np.float32)
    sc[1] = np.round(sc[1] * 2)            # heavy exact ties
    sc[4, 0, :] = 0.0                      # all equal
    sc[4, 1, ::2] = -0.0                   # signed zeros tie with +0
    # more than 512 keys in the threshold's top-11-bit bin: the kernel's
    # radix path instead of ranking the bin's keys directly
    sc[0, 1, :] = 1.0                      # 2,250 equal keys
    sc[0, 2, :] = 1.0
    sc[0, 2, rng.choice(2250, 30, replace=False)] = 5.0   # 30 above, the rest tie at 1.0
    got = _topk(sc, lens, hq, k)
    for i, T in enumerate(lens):
        want = orc.topk(sc[i], k, nb=T // 4)
        assert np.array_equal(got[i], want), (i, T)


@pytest.mark.parametrize("m", [63, 64, 65])
def test_topk_threshold_bin_of_63_64_65_keys(m):
    """m keys in [3, 3.5), one top-11-bit bin, above every other key: a
    threshold inside that bin takes the one-warp sort up to 64 keys and the
    direct ranking past it."""
    rng = np.random.default_rng(900 + m)
    sc = rng.uniform(-1.9, 1.9, (1, 2, 2250)).astype(np.float32)
    for h in range(2):
        pos = rng.choice(2250, m, replace=False)
        sc[0, h, pos] = rng.uniform(3.01, 3.49, m).astype(np.float32)
    sc[0, 1, pos[: m // 2]] = 3.25  # exact ties inside the bin
    for k in (1, 10, m - 1, m):
        got = _topk(sc, [9000], 2, k)
        assert np.array_equal(got[0], orc.topk(sc[0], k, nb=2250)), k


def test_sparse_config_scores_topk_and_attention():
    t = torch()
    lens = [9000, 9000]
    hq, k = 16, 64
    lay, pl = _pooled(lens, 128, seed=500)
    sc, ref, _ = _scores(lay, pl, lens, hq, seed=600)
    for i in range(2):
        assert np.array_equal(sc[i].view(np.uint32), ref[i].view(np.uint32))
    ids = _topk(sc, lens, hq, k)
    for i in range(2):
        assert np.array_equal(ids[i], orc.topk(ref[i], k))
    q = [synth.queries(700 + i, 1, hq, 256) for i in range(2)]
    seqs = pl.seqs(lens, [1, 1])
    dq = dev_u16(np.concatenate(q))
    out = t.zeros_like(dq)
    ws = t.zeros(pkv.sparse_ws_size(lay, seqs, hq, k) // 4 + 64, dtype=t.float32, device="cuda")
    dids = t.from_numpy(ids).cuda()
    pkv.sparse_decode(lay, seqs, 0, hq, dq, dids, k, out, ws)
    t.cuda.synchronize()
    got = host_u16(out).reshape(2, hq, 256)
    for i in range(2):
        want = orc.sparse_attend(pl.shape, pl.ocaches[i], 0, hq, 9000, q[i][0], ids[i])
        ok, worst = within_tol(got[i], want)
        assert ok, worst
    # paged == contiguous for the whole sparse path
    cont = place(lay, pl.streams, None)
    pkv.pool(lay, cont.seqs(lens, lens), 0)
    out2 = t.zeros_like(dq)
    pkv.sparse_decode(lay, cont.seqs(lens, [1, 1]), 0, hq, dq, dids, k, out2, ws)
    t.cuda.synchronize()
    assert t.equal(out, out2)


def test_sparse_with_all_blocks_equals_dense_and_padding_is_skipped():
    t = torch()
    lens = [256, 40]
    hq = 8
    lay, pl = _pooled(lens, 16, seed=800)
    k = 64
    ids = np.full((2, hq, k), -1, np.int32)
    ids[0, :, :] = np.arange(64)            # every block of stream 0
    ids[1, :, :10] = np.arange(10)          # every block of stream 1, then padding
    q = [synth.queries(900 + i, 1, hq, 256) for i in range(2)]
    seqs = pl.seqs(lens, [1, 1])
    dq = dev_u16(np.concatenate(q))
    out = t.zeros_like(dq)
    ws = t.zeros(pkv.sparse_ws_size(lay, seqs, hq, k) // 4 + 64, dtype=t.float32, device="cuda")
    pkv.sparse_decode(lay, seqs, 0, hq, dq, t.from_numpy(ids).cuda(), k, out, ws)
    t.cuda.synchronize()
    got = host_u16(out).reshape(2, hq, 256)
    for i, T in enumerate(lens):
        dense = orc.attend(pl.shape, pl.ocaches[i], 0, hq, T, q[i])[0]
        ok, worst = within_tol(got[i], dense)
        assert ok, worst
