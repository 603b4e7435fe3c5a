"""GPU: a pipeline wait that runs out ends with a status bit, not a hang.

Every barrier wait in the kernels is bounded (about a second); when it runs
out the kernel ORs PKV_DEV_TIMEOUT into the caller's status word and
returns.  The diagnostic launch waits on a barrier nothing arrives on; the
test checks the bit, the time it took, and that the context still runs a
decode that matches the oracle afterwards.  Nothing faults or hangs.
"""
import time

import numpy as np
import pytest

from paged_kv_cache_pg_gb300 import pkv, synth

from gpu_setup import decode, oracle_decode, place, torch, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_pg_gb300 import build
    build.build()
    pkv.load()


def test_a_wait_that_runs_out_reports_and_returns():
    t = torch()
    status = t.zeros(1, dtype=t.int32, device="cuda")
    t.cuda.synchronize()
    t0 = time.perf_counter()
    pkv.diag_wait_runs_out(status)
    t.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & pkv.DEV_TIMEOUT
    assert 0.5 < elapsed < 20.0
    # the context is intact: a decode right after still matches the oracle
    lay = pkv.layout(1, 1, 256, 128)
    s = [synth.make_stream(3000, 1, 64, 1, 256, 128)]
    q = [synth.queries(3001, 1, 4, 256)]
    pl = place(lay, s, 16, tables=[synth.reversed_table(4)], spare_pages=0)
    ok, worst = within_tol(decode(pl, 0, 4, q), oracle_decode(pl, 0, 4, q))
    assert ok, worst


@pytest.mark.parametrize("withheld", [0, 2])
def test_a_cta_whose_stage_never_lands_returns_as_a_whole(withheld):
    # eight warps in the decode's barrier structure; one slice's stage never
    # lands: its two warps time out and abort, the other slices finish, the
    # CTA meets at its barrier and the launch ends within a few limits
    t = torch()
    status = t.zeros(1, dtype=t.int32, device="cuda")
    t.cuda.synchronize()
    t0 = time.perf_counter()
    pkv.diag_cta_wait_runs_out(status, withheld)
    t.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & pkv.DEV_TIMEOUT
    assert 0.5 < elapsed < 10.0
    # the context is intact
    lay = pkv.layout(1, 1, 256, 128)
    s = [synth.make_stream(3002, 1, 300, 1, 256, 128)]
    q = [synth.queries(3003, 1, 4, 256)]
    pl = place(lay, s, 16, seed=3)
    ok, worst = within_tol(decode(pl, 0, 4, q), oracle_decode(pl, 0, 4, q))
    assert ok, worst


def test_cta_diagnostic_refuses_a_slice_out_of_range():
    t = torch()
    status = t.zeros(1, dtype=t.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.diag_cta_wait_runs_out(status, 4)
    assert e.value.code == pkv.EINVAL
