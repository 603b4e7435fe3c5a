"""GPU parity: the serving-shaped mix at its full size, in the launch shape the
benchmark times.

One arena of 792 pages of 256 positions holds four streams on random
non-overlapping page tables.  Three decode 4-query draft windows (causal
within the window) over 9,000, 24,000 and 40,956 cached positions, the
windows' rows stored by the decode call itself; the fourth appends a
2,048-query chunk at 16,384 (store, pool, tensor-core prefill).  Every
draft-window row is checked against the float64 oracle, the chunk on sampled
rows, and paged outputs must equal the outputs on contiguous caches bit for
bit.
"""
import numpy as np
import pytest

import oracle as orc
from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import dev_u16, host_u16, place, torch, within_tol

pytestmark = pytest.mark.gpu

DEC = [9000, 24000, 40956]      # cached positions of the draft-window streams
P0, C, W = 16384, 2048, 4       # the chunk's start and length, the window
ARENA = 792


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def _run(pl, streams, lay, qd_list, qp):
    """The two launches of a mix step on placed caches: the draft windows'
    decode (rows stored by the call), then the chunk's store, pool and
    prefill."""
    t = torch()
    totals = [L + W for L in DEC] + [P0 + C]
    status = t.zeros(1, dtype=t.int32, device="cuda")
    dsq = pl.seqs(totals[:3], [W] * 3)
    kn, vn, ikn = (dev_u16(np.concatenate([getattr(s, f)[0][L:] for s, L in zip(streams[:3], DEC)]))
                   for f in ("k", "v", "ik"))
    dq = dev_u16(np.concatenate(qd_list))
    od = t.zeros_like(dq)
    wsd = t.zeros(pkv.decode_ws_size(lay, dsq, 16) // 4 + 64, dtype=t.float32, device="cuda")
    pkv.decode(lay, dsq, 0, 16, dq, od, wsd, status=status, k_new=kn, v_new=vn, ik_new=ikn)
    psq = [pkv.seq(pl.pgs[3], P0 + C, C)]
    kc, vc, ic = (dev_u16(getattr(streams[3], f)[0][P0:]) for f in ("k", "v", "ik"))
    dqp = dev_u16(qp)
    op = t.zeros_like(dqp)
    wsp = t.zeros(pkv.prefill_ws_size(lay, psq, 16) // 4 + 64, dtype=t.float32, device="cuda")
    pkv.store(lay, psq, 0, kc, vc, ic, status=status)
    pkv.pool(lay, psq, 0, status=status)
    pkv.prefill(lay, psq, 0, 16, dqp, op, wsp, status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    return host_u16(od), host_u16(op).reshape(C, 16, 256)


def test_serving_mix_full_size():
    lay = pkv.layout(1, 2, 256, 128)
    totals = [L + W for L in DEC] + [P0 + C]
    streams = [synth.make_stream(2500 + i, 1, T, 2, 256, 128) for i, T in enumerate(totals)]
    spare = ARENA - sum(synth.pages_for(T, 256) for T in totals)
    pl = place(lay, streams, 256, seed=11, spare_pages=spare)
    qd_list = [synth.queries(2600 + i, W, 16, 256) for i in range(3)]
    qp = synth.queries(2700, C, 16, 256)
    dec, pre = _run(pl, streams, lay, qd_list, qp)
    # every draft-window row against the oracle
    ref = np.concatenate([orc.attend(pl.shape, pl.ocaches[i], 0, 16, totals[i], qd_list[i])
                          for i in range(3)])
    ok, worst = within_tol(dec, ref)
    assert ok, worst
    # sampled chunk rows, including its first and last query and both ends of a 128-row tile
    rng = np.random.default_rng(12)
    picks = [(0, 0), (C - 1, 15), (127, 3), (128, 12)] + \
        [(int(rng.integers(C)), int(rng.integers(16))) for _ in range(12)]
    for j, h in picks:
        r = orc.attend_row(pl.shape, pl.ocaches[3], 0, 16, h, P0 + j, qp[j, h])
        ok, worst = within_tol(pre[j, h], r)
        assert ok, (j, h, worst)
    assert pl.guards_intact()
    # the same launches on contiguous caches give the same bits
    cont = place(lay, streams, None)
    dec_c, pre_c = _run(cont, streams, lay, qd_list, qp)
    assert np.array_equal(dec, dec_c)
    assert np.array_equal(pre, pre_c)
