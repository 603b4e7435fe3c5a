"""The workspace-free decode entry point, checked against pkv_decode.

Some callers cannot allocate device memory: a plugin running inside a host
framework that owns every device allocation, or a serving loop that must not
call cudaMalloc because it can synchronize the whole device and take an
unbounded time.  pkv_decode_static serves them: it takes the same arguments
as pkv_decode minus the workspace, and keeps its split partials in a fixed
array inside the library.

This test calls it through the C ABI twice in a row, with different queries
and layers (so a stale partial left in the shared array would show).  Both
entry points run the same kernels with the same split plan, so each output
must equal pkv_decode's on the same inputs bit for bit; each is also checked
against the oracle within the bound the other parity tests use.  A batch
whose partials would not fit the fixed array must be refused.  The file is
named to run last.
"""
import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import dev_u16, host_u16, oracle_decode, place, torch, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def test_static_scratch_decode_matches_workspace_decode_twice():
    t = torch()
    lay = pkv.layout(2, 2, 256, 128)
    lens = [1001, 3001, 6001, 9001]   # the multi-stream workload, new token included
    streams = [synth.make_stream(700 + i, 2, T, 2, 256, 128) for i, T in enumerate(lens)]
    pl = place(lay, streams, 48, seed=4)
    seqs = pl.seqs(lens, [1] * 4)
    ws = t.zeros(pkv.decode_ws_size(lay, seqs, 16) // 4 + 64, dtype=t.float32, device="cuda")
    assert pkv.decode_ws_size(lay, seqs, 16) <= pkv.STATIC_SCRATCH_BYTES
    for call, layer in enumerate((1, 0)):
        q_list = [synth.queries(800 + 10 * call + i, 1, 16, 256) for i in range(4)]
        q = dev_u16(np.concatenate(q_list))
        want = t.zeros_like(q)
        got = t.zeros_like(q)
        pkv.decode(lay, seqs, layer, 16, q, want, ws)
        pkv.decode_static(lay, seqs, layer, 16, q, got)
        t.cuda.synchronize()
        assert np.array_equal(host_u16(got), host_u16(want)), f"call {call}: outputs differ"
        ok, report = within_tol(host_u16(got), oracle_decode(pl, layer, 16, q_list, lens))
        assert ok, f"call {call}: {report}"


def test_batch_too_large_for_the_fixed_array_is_refused():
    t = torch()
    lay = pkv.layout(1, 2, 256, 128)
    cap = 40960
    ps = pkv.page_elems(lay, cap)
    base = t.empty(1024, dtype=t.int16, device="cuda")   # never read: the call stops first
    # a 4-token window over 40,960 positions: 32 query columns x ~151 splits x 2 heads
    seqs = [pkv.seq(pkv.pg(base, None, ps, cap), cap, 4)]
    assert pkv.decode_ws_size(lay, seqs, 16) > pkv.STATIC_SCRATCH_BYTES
    q = t.zeros((4, 16, 256), dtype=t.int16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.decode_static(lay, seqs, 0, 16, q, t.zeros_like(q))
    assert e.value.code == pkv.EINVAL
