#!/usr/bin/env python
"""Benchmark of the paged decode-attention step on GB300.

Workload (multi-stream paged decode): 4 streams with cached lengths
{1000, 3000, 6000, 9000}, shuffled through one arena by random permutation
page tables; 16 query / 2 KV heads of 256, indexer keys of 128; one new
token per stream is stored, then its query attends the stream's keys
(split-KV partials and their combine).  A step runs 13 layer slots (the
pages' Flash Next pool: 12 attention layers plus the MTP head's cache) at
each swept page size {16, 48, 128, 256, 512}; each page size's 13 layers
stream ~506 MB of K/V, well above the 129 MB L2, so no flush is needed.
The same streams in contiguous buffers are timed beside it for the
paged/contiguous ratio.

Metric: algorithmic HBM bytes / device time, in GB/s, and query-heads/s.
Every other row of the hot path is measured after the timed region and
reported beside the headline (`rows`): the chunked prefill of 512 queries on
31,000 cached positions (store, pool, tensor-core attention), the
block-sparse decode (block scores, top-64, sparse attention), the serving
mix (three 4-query draft windows and a 2048-query prefill chunk in one
arena), and a single decode layer with L2 flushed.  `--only ROW` runs one of
those alone inside the profiler's capture range (for ncu), `--pages` limits
the decode sweep.

`--impl reference` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from paged_kv_cache_pg_gb300 import synth  # noqa: E402

METRIC = ("paged decode attn HBM GB/s (% of peak) & query-heads/s at 9k ctx; "
          "paged/contig ratio")
LENS = [1000, 3000, 6000, 9000]          # cached before the new token
N_LAYERS, HQ, HKV, D, DI = 13, 16, 2, 256, 128
PAGES = [16, 48, 128, 256, 512]
NOMINAL_HBM = 8000.0
ROWS = ["prefill", "sparse", "mix", "decode_layer", "prompt_cache", "decode_e4m3", "page_runs",
        "allocator"]
# DRAM bytes (read + write) of one pkv_decode call of the workload (partial +
# combine kernels), from one ncu capture of the decode kernels (summary under
# profiles/), valid while the decode sources hash to the value the capture
# was taken with; reported as null, with the capture date, otherwise.
DECODE_TRAFFIC = {"bytes": 40379904, "captured": "2026-12-02",
                  "sources": ["pkv_decode.cu", "pkv_dev.cuh", "pkv_internal.h", "pkv_host.cu"],
                  "sha256": "3d0c281022d012bc7f95eec7324822942159e464c695fbcdf299834a54e6561d"}
FLUSH_BYTES = 256 << 20                  # written between timed calls: twice the L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the other hot-path rows")
    ap.add_argument("--only", choices=ROWS, help="run one hot-path row alone (profiling)")
    ap.add_argument("--pages", type=str, default=None,
                    help="comma-separated page sizes to sweep (default: all five)")
    args = ap.parse_args()
    if args.pages:
        args.page_list = [int(x) for x in args.pages.split(",")]
        if any(p not in PAGES for p in args.page_list):
            ap.error(f"page sizes must be among {PAGES}")
    else:
        args.page_list = list(PAGES)
    return args


def config_desc(pages=PAGES):
    return {"workload": "multi-stream paged decode", "streams": len(LENS),
            "cached_lengths": LENS, "new_tokens_per_stream": 1, "layers": N_LAYERS,
            "q_heads": HQ, "kv_heads": HKV, "head_dim": D, "idx_dim": DI,
            "page_sizes": list(pages), "tables": "random permutations of one arena",
            "l2": "inputs larger than L2 (about 506 MB of K/V per page size per step)",
            "step": "13 layer slots x (split-KV decode with the new token's store fused + combine) at every page size"}


# ---- accounting ------------------------------------------------------------------

def layer_bytes(lens_after, n_pages_used):
    """Algorithmic HBM bytes of one layer's store + decode for the batch."""
    kv = sum(lens_after) * HKV * D * 2 * 2          # every K and V row read once
    qo = len(lens_after) * HQ * D * 2 * 2           # queries read, outputs written
    store = len(lens_after) * (2 * HKV * D + DI) * 2 * 2  # new rows read and written
    tables = n_pages_used * 4
    return kv + qo + store + tables


def decode_bytes(lens_after):
    """Bytes one decode call must move: K/V rows, queries, outputs."""
    return sum(lens_after) * HKV * D * 2 * 2 + len(lens_after) * HQ * D * 2 * 2


def row_credit_bytes(length):
    """Algorithmic bytes credited to one (stream, query head) row: its share of
    the stream's K/V read (the G heads of a KV head share each row)."""
    return length * HKV * D * 2 * 2 / HQ


def decode_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, "paged_kv_cache_pg_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return DECODE_TRAFFIC["bytes"] if h.hexdigest() == DECODE_TRAFFIC["sha256"] else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---- clocks ----------------------------------------------------------------------

class Clocks:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- distributed -------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(step_bytes: float, steps: int, local_ms: float, world: int, device=None):
    """Whole-job throughput (GB/s) of `world` replicas that each moved
    step_bytes per step for `steps` steps: every rank's bytes over the slowest
    rank's time.  Returns (value, max_ms)."""
    max_ms = max_over_ranks(local_ms, world, device)
    return world * step_bytes * steps / (max_ms / 1e3) / 1e9, max_ms


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- the CPU oracle (baseline and reference arm) ------------------------------------

def oracle_rows(seconds: float, max_rows: int = 1 << 30, part: int = 0, parts: int = 1):
    """Time oracle rows of the workload's layer 0 round-robin over (stream, head)
    (this worker's share `part` of `parts`) until `seconds` pass; returns
    (credited bytes, rows, elapsed)."""
    import oracle as orc
    orc.build()
    shape = orc.Shape(1, HKV, D, DI)
    caches, qs = [], []
    for i, L in enumerate(LENS):
        s = synth.make_stream(i, 1, L + 1, HKV, D, DI)
        c = orc.contiguous(shape, -(-(L + 1) // 4) * 4)
        orc.put_rows(shape, c, 0, orc.K, 0, s.k[0])
        orc.put_rows(shape, c, 0, orc.V, 0, s.v[0])
        caches.append(c)
        qs.append(synth.queries(100 + i, 1, HQ, D))
    credited, rows = 0.0, 0
    order = [(i, h) for h in range(HQ) for i in range(len(LENS))][part::parts]
    t0 = time.perf_counter()
    while rows < max_rows:
        i, h = order[rows % len(order)]
        orc.attend_row(shape, caches[i], 0, HQ, h, LENS[i], qs[i][0, h])
        credited += row_credit_bytes(LENS[i] + 1)
        rows += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return credited, rows, el


def oracle_row_rates(seconds: float):
    """The oracle as it stands, one thread, on a bounded sample of each other
    hot-path row's workload, each for about `seconds`: the CPU figure beside
    the row's GPU figure, in the row's own units."""
    import oracle as orc
    orc.build()
    out = {}
    shape = orc.Shape(1, HKV, D, DI)
    # chunked prefill: (query, head) rows of the 512-query chunk at 31,000
    P0, C = 31000, 512
    st = synth.make_stream(200, 1, P0 + C, HKV, D, DI)
    cache = orc.contiguous(shape, P0 + C)
    orc.put_rows(shape, cache, 0, orc.K, 0, st.k[0])
    orc.put_rows(shape, cache, 0, orc.V, 0, st.v[0])
    q = synth.queries(201, C, HQ, D)
    rng = np.random.default_rng(0)
    flop, rows, t0 = 0.0, 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        j, h = int(rng.integers(C)), int(rng.integers(HQ))
        orc.attend_row(shape, cache, 0, HQ, h, P0 + j, q[j, h])
        flop += 4.0 * (P0 + j + 1) * D
        rows += 1
    el = time.perf_counter() - t0
    out["prefill"] = {"value": round(flop / el / 1e12, 6), "unit": "TFLOP/s",
                      "query_heads_per_s": round(rows / el, 1),
                      "sample": f"{rows} random (query, head) rows of the chunk ({el:.1f} s)"}
    del cache, st
    # block-sparse step: pool, scores, top-64 and sparse attention of whole streams of 9,000
    T = 9000
    st = synth.make_stream(210, 1, T, HKV, D, DI)
    cache = orc.contiguous(shape, T)
    for kind, arr in ((orc.K, st.k[0]), (orc.V, st.v[0]), (orc.IK, st.ik[0])):
        orc.put_rows(shape, cache, 0, kind, 0, arr)
    qi = synth.normal_bf16(211, (HQ, DI))
    qs = synth.queries(212, 1, HQ, D)[0]
    n, t0 = 0, time.perf_counter()
    while True:
        orc.pool(shape, cache, 0, 0, T // 4)
        sc = orc.scores(shape, cache, 0, HQ, T, qi)
        ids = orc.topk(sc, 64)
        orc.sparse_attend(shape, cache, 0, HQ, T, qs, ids)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    out["sparse"] = {"value": round(n / el, 2), "unit": "streams a second",
                     "us_per_stream": round(el / n * 1e6, 1),
                     "query_heads_per_s": round(n * HQ / el, 1),
                     "sample": f"{n} streams of 9,000 positions, 16 heads each ({el:.1f} s)"}
    del cache, st
    # e4m3 decode: one query token, 16 heads, over e4m3 rows of 9,001 positions
    T = 9001
    shape8 = orc.Shape(1, HKV, D, DI, orc.E4M3)
    st = synth.make_stream(220, 1, T, HKV, D, DI)
    cache = orc.contiguous(shape8, -(-T // 4) * 4)
    orc.put_rows8(shape8, cache, 0, orc.K, 0, st.k[0])
    orc.put_rows8(shape8, cache, 0, orc.V, 0, st.v[0])
    q8 = synth.queries(221, 1, HQ, D)
    n, t0 = 0, time.perf_counter()
    while True:
        orc.attend(shape8, cache, 0, HQ, T, q8)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    b8 = T * HKV * 2 * (D + 4) + HQ * D * 2 * 2
    out["decode_e4m3"] = {"value": round(n * b8 / el / 1e9, 4), "unit": "GB/s",
                          "query_heads_per_s": round(n * HQ / el, 1),
                          "sample": f"{n} decodes of one token, 16 heads, 9,001 e4m3 positions "
                                    f"({el:.1f} s)"}
    del cache, st
    # prompt-cache save: a 31,512-position stream in pages of 256 gathered to the contiguous form
    T = 31512
    st = synth.make_stream(230, 1, T, HKV, D, DI)
    ptok = 256
    npg = synth.pages_for(T, ptok)
    table = np.ascontiguousarray(synth.shuffled_tables(231, npg, [npg])[0], dtype=np.int32)
    arena = np.zeros(npg * orc.page_elems(shape, ptok), np.uint16)
    cache = orc.paged(shape, arena, ptok, table)
    for kind, arr in ((orc.K, st.k[0]), (orc.V, st.v[0]), (orc.IK, st.ik[0])):
        orc.put_rows(shape, cache, 0, kind, 0, arr)
    n, t0 = 0, time.perf_counter()
    while True:
        for kind in (orc.K, orc.V, orc.IK):
            orc.get_rows(shape, cache, 0, kind, 0, T)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    gb = 2 * T * (2 * HKV * D + DI) * 2
    out["prompt_cache"] = {"value": round(n * gb / el / 1e9, 4), "unit": "GB/s",
                           "sample": f"{n} gathers of K, V and indexer rows of one layer "
                                     f"({el:.1f} s)"}
    return out


def _oracle_worker(args):
    seconds, part, parts = args
    return oracle_rows(seconds, part=part, parts=parts)


def oracle_rows_all_cores(seconds: float):
    """The oracle's independent (stream, head) rows split across every host core,
    one process each (started by spawn, so no CUDA state is inherited)."""
    import multiprocessing as mp
    import oracle as orc
    orc.build()
    n = max(1, min(os.cpu_count() or 1, len(LENS) * HQ))
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_worker, [(seconds, i, n) for i in range(n)])
    credited = sum(r[0] for r in res)
    rows = sum(r[1] for r in res)
    el = max(r[2] for r in res)
    return credited, rows, el, n


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # each step: one (stream, head) row of the workload, a bounded sample
    import oracle as orc
    orc.build()
    for _ in range(args.warmup):
        oracle_rows(0.0, max_rows=1)
    credited, rows, el = oracle_rows(1e9, max_rows=args.steps)
    gbs = credited / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / rows * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_desc(),
            "query_heads_per_s": rows / el,
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"{rows} (stream, query head) rows of layer 0, one a step, "
                                       "round-robin over the 4 streams and 16 heads"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---- the other rows of the hot path ------------------------------------------------

def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except Exception:
        return 1900.0, "fallback"


GRAPH_TIMING = "the row's calls captured once in a CUDA graph, each timed repetition a replay, L2 flushed before it"


class FlushTimer:
    """Median CUDA-event time of a call on the current stream, with a buffer
    twice the L2 written and then read back before every timed call (not
    timed): the read writes back the dirty lines the fill left in L2, so that
    their write-back is not charged to the timed call."""

    def __init__(self, torch, dev, profile=False):
        self.torch = torch
        self.buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.profile = profile

    def flush(self):
        self.buf.zero_()
        self.sink = self.buf.sum()

    def ms(self, fn, reps=20, warm=3, graph=False):
        """With `graph`, the calls of `fn` are captured once into a CUDA graph
        and each timed repetition replays it (as a serving loop would), so the
        host's time to issue the calls stays out of the timed region."""
        t = self.torch
        for _ in range(warm):
            self.flush()
            fn()
        t.cuda.synchronize()
        run = fn
        if graph:
            g = t.cuda.CUDAGraph()
            with t.cuda.graph(g):
                fn()
            g.replay()
            t.cuda.synchronize()
            run = g.replay
        e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        out = []
        if self.profile:
            t.cuda.profiler.start()
        for _ in range(reps):
            self.flush()
            e0.record()
            run()
            e1.record()
            e1.synchronize()
            out.append(e0.elapsed_time(e1))
        if self.profile:
            t.cuda.profiler.stop()
        return statistics.median(out)


def _paged(torch, pkv, lay, dev, ptok, lens_total, n_pages, seed):
    """One arena of n_pages, streams placed by random permutation tables."""
    ps = pkv.page_elems(lay, ptok)
    counts = [synth.pages_for(T, ptok) for T in lens_total]
    tabs = synth.shuffled_tables(seed, n_pages, counts)
    mem = torch.empty(n_pages * ps, dtype=torch.int16, device=dev)
    tables = [torch.from_numpy(t).to(dev) for t in tabs]
    return mem, tables, [pkv.pg(mem, t, ps, ptok, n_pages, t.numel()) for t in tables]


def _up(torch, dev, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def _place(torch, pkv, lay, dev, pg, stream, upto):
    """Store positions 0 .. upto-1 of a synthetic stream and pool their blocks."""
    sq = [pkv.seq(pg, upto, upto)]
    pkv.store(lay, sq, 0, _up(torch, dev, stream.k[0][:upto]), _up(torch, dev, stream.v[0][:upto]),
              _up(torch, dev, stream.ik[0][:upto]))
    pkv.pool(lay, sq, 0)


PREFILL_P0, PREFILL_C = 31000, 512


def _prefill_chunk(torch, pkv, dev, ptok):
    """The 512-query chunk on 31,000 cached positions in an arena of
    `ptok`-position pages: (store, pool, attend, status, buffers), each call
    on the current stream; the caller holds `buffers` (the arena and its
    table) while it calls them."""
    P0, C = PREFILL_P0, PREFILL_C
    T = P0 + C
    lay = pkv.layout(1, HKV, D, DI)
    mem, tables, pgs = _paged(torch, pkv, lay, dev, ptok, [T], synth.pages_for(T, ptok) + 4, 4)
    s = synth.make_stream(40, 1, T, HKV, D, DI)
    _place(torch, pkv, lay, dev, pgs[0], s, P0)
    kc, vc, ic = (_up(torch, dev, x[0][P0:]) for x in (s.k, s.v, s.ik))
    sq = [pkv.seq(pgs[0], T, C)]
    q = _up(torch, dev, synth.queries(41, C, HQ, D))
    out = torch.empty_like(q)
    ws = torch.zeros(pkv.prefill_ws_size(lay, sq, HQ) // 4 + 64, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def store():
        pkv.store(lay, sq, 0, kc, vc, ic, status=status)

    def pool():
        pkv.pool(lay, sq, 0, status=status)

    def attend():
        pkv.prefill(lay, sq, 0, HQ, q, out, ws, status=status)

    return store, pool, attend, status, (mem, tables)


def row_prefill(torch, pkv, dev, timer):
    """512-query chunk on 31,000 cached positions, pages of 256: the chunk's
    store, its pooled blocks, then the tensor-core attention."""
    P0, C = PREFILL_P0, PREFILL_C
    store, pool, attend, status, buffers = _prefill_chunk(torch, pkv, dev, 256)

    def step():
        store(), pool(), attend()

    t = {"store": timer.ms(store, graph=True), "pool": timer.ms(pool, graph=True),
         "prefill": timer.ms(attend, graph=True), "step": timer.ms(step, graph=True)}
    if int(status.item()) != 0:
        raise RuntimeError(f"prefill row: device status {int(status.item())}")
    flop = 4.0 * sum(P0 + j + 1 for j in range(C)) * HQ * D
    peak, kind = bf16_peak()
    tf = flop / (t["prefill"] / 1e3) / 1e12
    return {"timing": GRAPH_TIMING,
            "workload": "chunked prefill: 512 queries on 31,000 cached positions, pages of 256, "
                        "16/2 heads", "us": {k: round(v * 1e3, 2) for k, v in t.items()},
            "flop": flop, "TFLOPs": round(tf, 1),
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tf / peak, 4), "peak_kind": kind},
            "query_heads_per_s": round(C * HQ / (t["step"] / 1e3), 1)}


def row_sparse(torch, pkv, dev, timer):
    """2 streams of 9,000 positions in pages of 128: block scores of the pooled
    indexer keys, top-64 blocks per head, attention over those blocks."""
    T, K_SEL = 9000, 64
    lay = pkv.layout(1, HKV, D, DI)
    n_pages = 2 * synth.pages_for(T, 128) + 8
    mem, tables, pgs = _paged(torch, pkv, lay, dev, 128, [T, T], n_pages, 3)
    for i in range(2):
        _place(torch, pkv, lay, dev, pgs[i], synth.make_stream(30 + i, 1, T, HKV, D, DI), T)
    sq = [pkv.seq(g, T, 1) for g in pgs]
    nb = T // 4
    qi = _up(torch, dev, np.concatenate([synth.queries(32 + i, 1, HQ, DI) for i in range(2)]))
    q = _up(torch, dev, np.concatenate([synth.queries(34 + i, 1, HQ, D) for i in range(2)]))
    scores = torch.empty((2, HQ, nb), dtype=torch.float32, device=dev)
    ids = torch.empty((2, HQ, K_SEL), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    ws = torch.zeros(pkv.sparse_ws_size(lay, sq, HQ, K_SEL) // 4 + 64, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def sc():
        pkv.block_scores(lay, sq, 0, HQ, qi, scores, nb, status=status)

    def tk():
        pkv.topk(sq, HQ, scores, nb, K_SEL, ids)

    def att():
        pkv.sparse_decode(lay, sq, 0, HQ, q, ids, K_SEL, out, ws, status=status)

    def step():
        sc(), tk(), att()

    t = {"block_scores": timer.ms(sc, graph=True), "topk": timer.ms(tk, graph=True),
         "sparse_decode": timer.ms(att, graph=True), "step": timer.ms(step, graph=True)}
    step_direct = timer.ms(step)
    if int(status.item()) != 0:
        raise RuntimeError(f"sparse row: device status {int(status.item())}")
    # algorithmic bytes: pooled rows, scores written and read back, the selected
    # K and V rows of every query head, queries and outputs
    b_scores = 2 * (nb * DI * 2 + HQ * DI * 2 + HQ * nb * 4)
    b_topk = 2 * (HQ * nb * 4 + HQ * K_SEL * 4)
    b_att = 2 * (HQ * K_SEL * 4 * 2 * D * 2 + 2 * HQ * D * 2 + HQ * K_SEL * 4)
    peak, kind = peaks()
    gbs = (b_scores + b_topk + b_att) / (t["step"] / 1e3) / 1e9
    att_gbs = b_att / (t["sparse_decode"] / 1e3) / 1e9
    return {"timing": GRAPH_TIMING,
            "workload": "block-sparse decode: 2 streams of 9,000, pages of 128, top-64 blocks",
            "us": {k: round(v * 1e3, 2) for k, v in t.items()},
            "bytes": {"block_scores": b_scores, "topk": b_topk, "sparse_decode": b_att},
            "step_us_direct_calls": round(step_direct * 1e3, 2),
            "GBps_step": round(gbs, 1), "GBps_sparse_decode": round(att_gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind},
            "query_heads_per_s": round(2 * HQ / (t["step"] / 1e3), 1)}


def row_mix(torch, pkv, dev, timer):
    """Serving mix in one arena of 792 pages of 256: three streams decoding
    4-query draft windows (the window's rows stored by the call) and one
    2048-query prefill chunk (store, pool, attention)."""
    dec_cached = [9000, 24000, 40956]
    P0, C, W = 16384, 2048, 4
    totals = [L + W for L in dec_cached] + [P0 + C]
    lay = pkv.layout(1, HKV, D, DI)
    mem, tables, pgs = _paged(torch, pkv, lay, dev, 256, totals, 792, 5)
    streams = [synth.make_stream(50 + i, 1, T, HKV, D, DI) for i, T in enumerate(totals)]
    for i, L in enumerate(dec_cached + [P0]):
        _place(torch, pkv, lay, dev, pgs[i], streams[i], L)
    dsq = [pkv.seq(pgs[i], totals[i], W) for i in range(3)]
    win = [np.concatenate([getattr(streams[i], f)[0][dec_cached[i]:] for i in range(3)])
           for f in ("k", "v", "ik")]
    kn, vn, ikn = (_up(torch, dev, x) for x in win)
    qd = _up(torch, dev, np.concatenate([synth.queries(60 + i, W, HQ, D) for i in range(3)]))
    od = torch.empty_like(qd)
    wsd = torch.zeros(pkv.decode_ws_size(lay, dsq, HQ) // 4 + 64, dtype=torch.float32, device=dev)
    psq = [pkv.seq(pgs[3], P0 + C, C)]
    kc, vc, ic = (_up(torch, dev, x[0][P0:]) for x in (streams[3].k, streams[3].v, streams[3].ik))
    qp = _up(torch, dev, synth.queries(64, C, HQ, D))
    op = torch.empty_like(qp)
    wsp = torch.zeros(pkv.prefill_ws_size(lay, psq, HQ) // 4 + 64, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    del streams

    def dec():
        pkv.decode(lay, dsq, 0, HQ, qd, od, wsd, status=status, k_new=kn, v_new=vn, ik_new=ikn)

    def pre():
        pkv.store(lay, psq, 0, kc, vc, ic, status=status)
        pkv.pool(lay, psq, 0, status=status)
        pkv.prefill(lay, psq, 0, HQ, qp, op, wsp, status=status)

    def step():
        dec(), pre()

    t = {"draft_window_decode": timer.ms(dec, graph=True), "prefill_lane": timer.ms(pre, graph=True),
         "step": timer.ms(step, graph=True)}
    if int(status.item()) != 0:
        raise RuntimeError(f"mix row: device status {int(status.item())}")
    dec_bytes = sum(totals[:3]) * HKV * D * 2 * 2 + 2 * 3 * W * HQ * D * 2
    flop = 4.0 * sum(P0 + j + 1 for j in range(C)) * HQ * D
    peak, kind = peaks()
    dgbs = dec_bytes / (t["draft_window_decode"] / 1e3) / 1e9
    return {"timing": GRAPH_TIMING,
            "workload": "serving mix: 792 x 256 arena; 3 streams {9000, 24000, 40956} with 4-query "
                        "draft windows; 1 stream with a 2048-query chunk at 16,384",
            "us": {k: round(v * 1e3, 2) for k, v in t.items()},
            "draft_window_GBps": round(dgbs, 1), "draft_window_frac": round(dgbs / peak, 4),
            "prefill_lane_TFLOPs": round(flop / (t["prefill_lane"] / 1e3) / 1e12, 1),
            "query_heads_per_s": round((3 * W + C) * HQ / (t["step"] / 1e3), 1)}


def row_decode_layer(torch, pkv, dev, timer):
    """One decode layer of the multi-stream workload at pages of 256, L2 flushed."""
    lens_after = [L + 1 for L in LENS]
    lay = pkv.layout(1, HKV, D, DI)
    n_pages = sum(synth.pages_for(L, 256) for L in lens_after) + 8
    mem, tables, pgs = _paged(torch, pkv, lay, dev, 256, lens_after, n_pages, 6)
    streams = [synth.make_stream(70 + i, 1, L, HKV, D, DI) for i, L in enumerate(lens_after)]
    for g, st, L in zip(pgs, streams, LENS):
        _place(torch, pkv, lay, dev, g, st, L)
    sq = [pkv.seq(g, L, 1) for g, L in zip(pgs, lens_after)]
    kn, vn, ikn = (_up(torch, dev, np.concatenate([getattr(st, f)[0][-1:] for st in streams]))
                   for f in ("k", "v", "ik"))
    q = _up(torch, dev, np.concatenate([synth.queries(80 + i, 1, HQ, D) for i in range(len(LENS))]))
    out = torch.empty_like(q)
    ws = torch.zeros(pkv.decode_ws_size(lay, sq, HQ) // 4 + 64, dtype=torch.float32, device=dev)

    def dec():
        pkv.decode(lay, sq, 0, HQ, q, out, ws, k_new=kn, v_new=vn, ik_new=ikn)

    ms = timer.ms(dec, reps=50, graph=True)
    peak, kind = peaks()
    gbs = decode_bytes(lens_after) / (ms / 1e3) / 1e9
    return {"timing": GRAPH_TIMING,
            "workload": "one layer of the multi-stream decode at pages of 256, L2 flushed "
                        "before every call", "us": round(ms * 1e3, 2), "GBps": round(gbs, 1),
            "frac": round(gbs / peak, 4), "peak_kind": kind}


def row_prompt_cache(torch, pkv, dev, timer):
    """Prompt-cache save and restore of one 31,512-position stream in pages of
    256 (one layer): save gathers its K, V, indexer and pooled rows through
    the table into the contiguous layout; restore stores K, V and indexer rows
    back into another stream's pages and pools its blocks."""
    T = 31512
    lay = pkv.layout(1, HKV, D, DI)
    n_pages = 2 * synth.pages_for(T, 256) + 4
    mem, tables, pgs = _paged(torch, pkv, lay, dev, 256, [T, T], n_pages, 7)
    s = synth.make_stream(90, 1, T, HKV, D, DI)
    _place(torch, pkv, lay, dev, pgs[0], s, T)
    del s
    src, dst = [pkv.seq(pgs[0], T, T)], [pkv.seq(pgs[1], T, T)]
    k = torch.empty((T, HKV, D), dtype=torch.int16, device=dev)
    v = torch.empty_like(k)
    ik = torch.empty((T, DI), dtype=torch.int16, device=dev)
    pooled = torch.empty((T // 4, DI), dtype=torch.int16, device=dev)

    def save():
        pkv.gather(lay, src, 0, pkv.K, k)
        pkv.gather(lay, src, 0, pkv.V, v)
        pkv.gather(lay, src, 0, pkv.IK, ik)
        pkv.gather(lay, src, 0, pkv.P, pooled)

    def restore():
        pkv.store(lay, dst, 0, k, v, ik)
        pkv.pool(lay, dst, 0)

    t = {"save": timer.ms(save, graph=True), "restore": timer.ms(restore, graph=True)}
    torch.cuda.synchronize()
    same = all(torch.equal(a, b) for a, b in zip(_gather_all(torch, pkv, lay, dst, T, dev), (k, v, ik, pooled)))
    row = T * (2 * HKV * D + DI) * 2 + (T // 4) * DI * 2   # bytes of one copy of the stream
    b_save = 2 * row                                       # read through the table, written packed
    b_restore = 2 * (T * (2 * HKV * D + DI) * 2) + (T * DI * 2 + (T // 4) * DI * 2)
    peak, kind = peaks()
    g_save = b_save / (t["save"] / 1e3) / 1e9
    g_restore = b_restore / (t["restore"] / 1e3) / 1e9
    return {"timing": GRAPH_TIMING,
            "workload": "prompt-cache save/restore: 1 stream of 31,512 positions, pages of 256, "
                        "one layer (K, V, indexer, pooled rows)",
            "us": {k_: round(v_ * 1e3, 2) for k_, v_ in t.items()},
            "GBps": {"save": round(g_save, 1), "restore": round(g_restore, 1)},
            "frac": {"save": round(g_save / peak, 4), "restore": round(g_restore / peak, 4)},
            "restored_equals_saved": bool(same)}


def row_decode_e4m3(torch, pkv, dev, timer):
    """The multi-stream decode with e4m3 K/V (codes + a float32 scale per head
    and row): 13 layer slots at pages of 256, each one decode call that also
    quantizes and stores the new token's rows, replayed as one CUDA graph."""
    lens_after = [L + 1 for L in LENS]
    lay8 = pkv.layout(N_LAYERS, HKV, D, DI, pkv.KV_E4M3)
    n_pages = sum(synth.pages_for(L, 256) for L in lens_after) + 8
    mem, tables, pgs = _paged(torch, pkv, lay8, dev, 256, lens_after, n_pages, 8)
    streams = [synth.make_stream(110 + i, N_LAYERS, L, HKV, D, DI) for i, L in enumerate(lens_after)]
    for l in range(N_LAYERS):
        pkv.store(lay8, [pkv.seq(g, L, L) for g, L in zip(pgs, LENS)], l,
                  *(_up(torch, dev, np.concatenate([getattr(st, f)[l][:-1] for st in streams]))
                    for f in ("k", "v", "ik")))
    new = [[_up(torch, dev, np.concatenate([getattr(st, f)[l][-1:] for st in streams]))
            for f in ("k", "v", "ik")] for l in range(N_LAYERS)]
    del streams
    sq = [pkv.seq(g, L, 1) for g, L in zip(pgs, lens_after)]
    q = [_up(torch, dev, np.concatenate([synth.queries(120 + l * 4 + i, 1, HQ, D) for i in range(4)]))
         for l in range(N_LAYERS)]
    out = [torch.empty_like(x) for x in q]
    ws = torch.zeros(pkv.decode_ws_size(lay8, sq, HQ) // 4 + 64, dtype=torch.float32, device=dev)

    def step():
        for l in range(N_LAYERS):
            k_, v_, ik_ = new[l]
            pkv.decode(lay8, sq, l, HQ, q[l], out[l], ws, k_new=k_, v_new=v_, ik_new=ik_)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    ms = timer.ms(g.replay, reps=30)
    row8 = HKV * 2 * (D + 4)                            # K and V codes + scales of a position
    b_layer = sum(lens_after) * row8 + len(LENS) * HQ * D * 2 * 2 + len(LENS) * (2 * HKV * D + DI) * 2 * 2
    gbs = N_LAYERS * b_layer / (ms / 1e3) / 1e9
    peak, kind = peaks()
    bf16_bytes = N_LAYERS * layer_bytes(lens_after, 0)
    return {"workload": "multi-stream decode, e4m3 K/V: 4 streams {1000, 3000, 6000, 9000} + 1 new "
                        "token, 16/2 heads, 13 layer slots, pages of 256 (decode with the store fused)",
            "us_13_layers": round(ms * 1e3, 2), "us_per_layer": round(ms * 1e3 / N_LAYERS, 2),
            "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
            "bf16_equivalent_GBps": round(bf16_bytes / (ms / 1e3) / 1e9, 1),
            "query_heads_per_s": round(N_LAYERS * len(LENS) * HQ / (ms / 1e3), 1)}


def row_page_runs(torch, pkv, dev, timer):
    """The page-run path against key-by-key copies: the multi-stream decode
    (13 layer slots, the new token stored by the call) at pages of 16, whose
    16-row page runs load as 2D TMA tiles, and at pages of 20, whose rows load
    key by key with cp.async.  Each page size is one CUDA graph."""
    lens_after = [L + 1 for L in LENS]
    lay = pkv.layout(N_LAYERS, HKV, D, DI)
    streams = [synth.make_stream(140 + i, N_LAYERS, L, HKV, D, DI) for i, L in enumerate(lens_after)]
    new = [[_up(torch, dev, np.concatenate([getattr(st, f)[l][-1:] for st in streams]))
            for f in ("k", "v", "ik")] for l in range(N_LAYERS)]
    q = [_up(torch, dev, np.concatenate([synth.queries(160 + l * 4 + i, 1, HQ, D) for i in range(4)]))
         for l in range(N_LAYERS)]
    out = [torch.empty_like(x) for x in q]
    res = {}
    for ptok in (16, 20):
        n_pages = sum(synth.pages_for(L, ptok) for L in lens_after) + 8
        mem, tables, pgs = _paged(torch, pkv, lay, dev, ptok, lens_after, n_pages, 9)
        for l in range(N_LAYERS):
            pkv.store(lay, [pkv.seq(g, L, L) for g, L in zip(pgs, LENS)], l,
                      *(_up(torch, dev, np.concatenate([getattr(st, f)[l][:-1] for st in streams]))
                        for f in ("k", "v", "ik")))
        sq = [pkv.seq(g, L, 1) for g, L in zip(pgs, lens_after)]
        ws = torch.zeros(pkv.decode_ws_size(lay, sq, HQ) // 4 + 64, dtype=torch.float32, device=dev)

        def step():
            for l in range(N_LAYERS):
                k_, v_, ik_ = new[l]
                pkv.decode(lay, sq, l, HQ, q[l], out[l], ws, k_new=k_, v_new=v_, ik_new=ik_)

        for _ in range(2):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        ms = timer.ms(g.replay, reps=30)
        res[ptok] = ms * 1e3 / N_LAYERS
        del g, mem, tables, pgs, ws
        torch.cuda.empty_cache()
    # the chunked prefill, whose one producer warp a K or V ring issues a
    # tile's copies: 8 TMA boxes a 32-key tile of 16-row runs, or 32
    # cp.async a lane key by key
    pre = {}
    for ptok in (16, 20):
        store, pool, attend, status, buffers = _prefill_chunk(torch, pkv, dev, ptok)
        pre[ptok] = timer.ms(attend, graph=True) * 1e3
        if int(status.item()) != 0:
            raise RuntimeError(f"page-run row: device status {int(status.item())}")
        del store, pool, attend, status, buffers
        torch.cuda.empty_cache()
    peak, kind = peaks()
    b = decode_bytes(lens_after)
    return {"workload": "multi-stream decode, 13 layer slots, new token stored by the call, and the "
                        "512-query prefill chunk on 31,000 positions: pages of 16 (16-row page runs "
                        "by TMA) against pages of 20 (rows key by key)",
            "us_per_layer": {"page_runs_p16": round(res[16], 2), "key_by_key_p20": round(res[20], 2)},
            "GBps": {"page_runs_p16": round(b / res[16] / 1e3, 1),
                     "key_by_key_p20": round(b / res[20] / 1e3, 1)},
            "key_by_key_over_page_runs": round(res[20] / res[16], 4),
            "prefill_us": {"page_runs_p16": round(pre[16], 2), "key_by_key_p20": round(pre[20], 2)},
            "prefill_key_by_key_over_page_runs": round(pre[20] / pre[16], 4)}


def row_allocator(torch, pkv, dev, timer):
    """Host cost of the page pool on the serving-mix arena (792 pages of 256,
    13 layers): a lane opens (a run of state pages claimed from the top, the
    KV pages of a 40,960-position stream from the bottom) and closes (both
    given back, deferred on the stream by an event).  Host work only, timed
    with the host clock through the Python binding."""
    import time
    lay = pkv.layout(N_LAYERS, HKV, D, DI)
    ps = pkv.page_elems(lay, 256)
    n_pages = 792
    mem = torch.empty(n_pages * ps, dtype=torch.int16, device=dev)
    arena = pkv.Arena(lay, 256, mem)
    stream = torch.cuda.current_stream(dev)
    k_run = arena.run_pages(64 << 20)          # 64 MiB of per-stream state
    n_kv = 40960 // 256
    busy = arena.take(300)                     # other lanes' pages: the scan starts mid-pool
    cycles = 2000

    def cycle():
        first = arena.run_take(k_run)
        ids = arena.take(n_kv)
        arena.give(ids, stream=stream, defer=True)
        arena.run_give(first, k_run, stream=stream, defer=True)

    for _ in range(50):
        cycle()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(cycles):
        cycle()
    us = (time.perf_counter() - t0) / cycles * 1e6
    torch.cuda.synchronize()
    ok = arena.info()[1] == n_pages - busy.size
    arena.close()
    return {"workload": "page pool: lane open + close on a 792 x 256 arena (run of %d pages from "
                        "the top, %d KV pages from the bottom, deferred release)" % (k_run, n_kv),
            "us_per_open_close": round(us, 2), "cycles": cycles, "pages_all_returned": bool(ok),
            "clock": "host (time.perf_counter), no kernels"}


def _gather_all(torch, pkv, lay, seqs, T, dev):
    outs = [torch.empty((T, HKV, D), dtype=torch.int16, device=dev),
            torch.empty((T, HKV, D), dtype=torch.int16, device=dev),
            torch.empty((T, DI), dtype=torch.int16, device=dev),
            torch.empty((T // 4, DI), dtype=torch.int16, device=dev)]
    for kind, o in zip((pkv.K, pkv.V, pkv.IK, pkv.P), outs):
        pkv.gather(lay, seqs, 0, kind, o)
    return outs


ROW_FNS = {"prefill": row_prefill, "sparse": row_sparse, "mix": row_mix,
           "decode_layer": row_decode_layer, "prompt_cache": row_prompt_cache,
           "decode_e4m3": row_decode_e4m3, "page_runs": row_page_runs, "allocator": row_allocator}


def hot_path_rows(torch, pkv, dev, names, profile=False):
    timer = FlushTimer(torch, dev, profile=profile)
    out = {}
    for n in names:
        out[n] = ROW_FNS[n](torch, pkv, dev, timer)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


# ---- our arm -----------------------------------------------------------------------

def main_ours(args):
    import torch
    from paged_kv_cache_pg_gb300 import build, pkv

    rank, world, local = dist_env()
    pages = args.page_list
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    pkv.load()

    if args.only:
        # one hot-path row alone, its timed calls inside the profiler's capture range
        res = hot_path_rows(torch, pkv, dev, [args.only], profile=True)
        if rank == 0:
            print(json.dumps({"only": args.only, "row": res[args.only]}))
        return 0

    lay = pkv.layout(N_LAYERS, HKV, D, DI)
    lens_after = [L + 1 for L in LENS]
    S = len(LENS)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    # data: per layer, every stream's positions 0..L (the last one is the new token)
    streams = [synth.make_stream(rank * 100 + i, N_LAYERS, L + 1, HKV, D, DI)
               for i, L in enumerate(LENS)]
    q_host = [np.concatenate([synth.queries(rank * 100 + 50 + l * S + i, 1, HQ, D)
                              for i in range(S)]) for l in range(N_LAYERS)]
    k_new = [up(np.concatenate([s.k[l][-1:] for s in streams])) for l in range(N_LAYERS)]
    v_new = [up(np.concatenate([s.v[l][-1:] for s in streams])) for l in range(N_LAYERS)]
    ik_new = [up(np.concatenate([s.ik[l][-1:] for s in streams])) for l in range(N_LAYERS)]
    q_dev = [up(q) for q in q_host]
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # caches: one arena per page size, and contiguous buffers
    confs = {}
    for p in pages + [None]:
        if p is None:
            pgs, mems = [], []
            for L in lens_after:
                cap = -(-L // 256) * 256   # a reserved window, rounded to 256 positions
                ps = pkv.page_elems(lay, cap)
                m = torch.empty(ps, dtype=torch.int16, device=dev)
                mems.append(m)
                pgs.append(pkv.pg(m, None, ps, cap))
            tables, used = [], 0
        else:
            ps = pkv.page_elems(lay, p)
            counts = [synth.pages_for(L, p) for L in lens_after]
            n_pages = sum(counts) + 8
            tabs = synth.shuffled_tables(rank * 1000 + p, n_pages, counts)
            m = torch.empty(n_pages * ps, dtype=torch.int16, device=dev)
            mems = [m]
            tables = [torch.from_numpy(t).to(dev) for t in tabs]
            pgs = [pkv.pg(m, t, ps, p, n_pages, t.numel()) for t in tables]
            used = sum(counts)
        confs[p] = {"mems": mems, "tables": tables, "pgs": pgs, "pages_used": used}

    for l in range(N_LAYERS):
        kc = up(np.concatenate([s.k[l][:-1] for s in streams]))
        vc = up(np.concatenate([s.v[l][:-1] for s in streams]))
        ic = up(np.concatenate([s.ik[l][:-1] for s in streams]))
        for p, cf in confs.items():
            pkv.store(lay, [pkv.seq(g, L, L) for g, L in zip(cf["pgs"], LENS)], l, kc, vc, ic,
                      status=status)
        del kc, vc, ic
    torch.cuda.synchronize()
    del streams

    step_seqs = {p: [pkv.seq(g, L, 1) for g, L in zip(cf["pgs"], lens_after)]
                 for p, cf in confs.items()}
    for p, cf in confs.items():
        n = pkv.decode_ws_size(lay, step_seqs[p], HQ)
        cf["ws"] = torch.zeros(max(64, n // 4 + 64), dtype=torch.float32, device=dev)
        cf["launches_per_layer"] = 1 + (1 if n > 0 else 0)
        cf["out"] = [torch.empty_like(q_dev[0]) for _ in range(N_LAYERS)]

    def capture(p):
        cf = confs[p]
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):  # settle lazy set-up before capture
                for l in range(N_LAYERS):
                    pkv.decode(lay, step_seqs[p], l, HQ, q_dev[l], cf["out"][l], cf["ws"],
                               status=status, k_new=k_new[l], v_new=v_new[l], ik_new=ik_new[l])
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for l in range(N_LAYERS):
                # the new token's store is fused into the decode call
                pkv.decode(lay, step_seqs[p], l, HQ, q_dev[l], cf["out"][l], cf["ws"],
                           status=status, k_new=k_new[l], v_new=v_new[l], ik_new=ik_new[l])
        return g

    graphs = {p: capture(p) for p in confs}

    # correctness guard: paged outputs equal contiguous outputs bit for bit
    for p in confs:
        graphs[p].replay()
    torch.cuda.synchronize()
    same = all(torch.equal(confs[p]["out"][l], confs[None]["out"][l])
               for p in pages for l in range(N_LAYERS))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status word {int(status.item())}")

    for _ in range(args.warmup):
        for p in confs:
            graphs[p].replay()
    torch.cuda.synchronize()

    clocks = Clocks(local)
    step_ms = {p: [] for p in confs}
    ev0 = {p: torch.cuda.Event(enable_timing=True) for p in confs}
    ev1 = {p: torch.cuda.Event(enable_timing=True) for p in confs}
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    torch.cuda.profiler.start()   # the profiler's capture range is the timed region
    for _ in range(args.steps):
        for p in pages:
            ev0[p].record()
            graphs[p].replay()
            ev1[p].record()
        ev1[pages[-1]].synchronize()
        for p in pages:
            step_ms[p].append(ev0[p].elapsed_time(ev1[p]))
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    wall = time.perf_counter() - t_wall
    barrier(world)
    clk = clocks.stop()

    # paging overhead: the contiguous baseline (same workload, own buffers) in
    # one rotation with every paged graph, each timed alone, so that both sides
    # start their steps from the same cache state
    rot_ms = {p: [] for p in confs}
    for _ in range(args.steps):
        for p in list(pages) + [None]:
            ev0[p].record()
            graphs[p].replay()
            ev1[p].record()
        ev1[None].synchronize()
        for p in confs:
            rot_ms[p].append(ev0[p].elapsed_time(ev1[p]))
    torch.cuda.synchronize()
    cont_ms = rot_ms[None]

    # ---- results ----
    per_step_ms = sum(statistics.fmean(step_ms[p]) for p in pages)
    step_bytes = sum(N_LAYERS * layer_bytes(lens_after, confs[p]["pages_used"]) for p in pages)
    value, max_ms = aggregate(step_bytes, args.steps, per_step_ms * args.steps, world, dev)
    qh_per_step = len(pages) * N_LAYERS * S * HQ
    per_page = {}
    for p in pages:
        ms = statistics.fmean(step_ms[p])
        per_page[str(p)] = {
            "GBps": round(N_LAYERS * layer_bytes(lens_after, confs[p]["pages_used"]) / ms / 1e6, 1),
            "ms_13_layers": round(ms, 4),
            "paged_over_contig": round(statistics.fmean(rot_ms[p]) / statistics.fmean(cont_ms), 4)}
    cont_gbs = N_LAYERS * layer_bytes(lens_after, 0) / statistics.fmean(cont_ms) / 1e6
    peak, peak_kind = peaks()

    # one pkv_decode call (partial kernel with the fused store + combine kernel) per
    # layer; its average duration is the timed graph time over its 13 calls
    dur = statistics.fmean(x for p in pages for x in step_ms[p]) / N_LAYERS / 1e3
    achieved = decode_bytes(lens_after) / dur / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": decode_traffic(),
            "traffic_captured": DECODE_TRAFFIC["captured"],
            "traffic_valid": decode_traffic() is not None,
            "algorithmic_bytes": decode_bytes(lens_after),
            "kernel": "pkv_decode (split-KV partial with fused store + combine), one layer, 4 streams",
            "avg_launch_us": round(dur * 1e6, 3), "peak_kind": peak_kind,
            "frac_of_nominal_8TBs": round(achieved / NOMINAL_HBM, 4)}

    rows = None if args.no_rows else hot_path_rows(torch, pkv, dev, ROWS)

    # end to end through the public API with host buffers
    e2e = e2e_arm(torch, pkv, lay, confs, step_seqs, q_host, k_new, v_new, ik_new, status,
                  lens_after, dev, args)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        credited, n_rows, el = oracle_rows(args.cpu_seconds)
        cpu = {"value": round(credited / el / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{n_rows} (stream, query head) rows of layer 0 of the workload "
                         f"({el:.1f} s, one thread)"}
        c_all, r_all, el_all, n_all = oracle_rows_all_cores(args.cpu_seconds)
        cpu["all_cores"] = {"value": round(c_all / el_all / 1e9, 4), "unit": "GB/s", "cores": n_all,
                            "sample": f"{r_all} rows, the (stream, head) rows split across "
                                      f"{n_all} processes ({el_all:.1f} s)"}
        if rows is not None:
            cpu["rows"] = oracle_row_rates(args.cpu_seconds / 5)

    launches = args.steps * sum(N_LAYERS * confs[p]["launches_per_layer"] for p in pages)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_desc(pages),
            "pct_of_measured_peak": round(100 * value / world / peak, 2),
            "pct_of_nominal_8TBs": round(100 * value / world / NOMINAL_HBM, 2),
            "query_heads_per_s": round(world * qh_per_step * args.steps / (max_ms / 1e3), 1),
            "per_page_size": per_page,
            "contiguous": {"GBps": round(cont_gbs, 1), "ms_13_layers": round(statistics.fmean(cont_ms), 4)},
            "paged_contig_ratio_worst": max(v["paged_over_contig"] for v in per_page.values()),
            "paged_equals_contiguous": bool(same),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "rows": rows,
            "clocks": clk, "timed_wall_s": round(wall, 3)}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def e2e_arm(torch, pkv, lay, confs, step_seqs, q_host, k_new, v_new, ik_new, status, lens_after,
            dev, args):
    """Same step through the public calls, inputs from pinned host memory and
    outputs back to it, copies inside the timed region."""
    pages = args.page_list
    h_q = torch.from_numpy(np.stack(q_host).view(np.int16))
    kv_rows = torch.stack([torch.stack([k.cpu(), v.cpu()]) for k, v in zip(k_new, v_new)])
    ik_rows = torch.stack([i.cpu() for i in ik_new])
    # the step's inputs, queries then new K/V rows then indexer rows, in one
    # pinned buffer: one host-to-device copy a graph (every part starts on a
    # 16-byte boundary)
    nq, nkv, nik = h_q.numel(), kv_rows.numel(), ik_rows.numel()
    assert (nq * 2) % 16 == 0 and ((nq + nkv) * 2) % 16 == 0
    h_in = torch.empty(nq + nkv + nik, dtype=torch.int16).pin_memory()
    h_in[:nq].copy_(h_q.reshape(-1))
    h_in[nq:nq + nkv].copy_(kv_rows.reshape(-1))
    h_in[nq + nkv:].copy_(ik_rows.reshape(-1))
    # per page size its own device inputs and outputs and host outputs, so
    # that one graph's copies can run while another graph computes
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    bufs, graphs = {}, {}
    for p in pages:
        cf = confs[p]
        d_in = torch.empty(h_in.shape, dtype=torch.int16, device=dev)
        d_q = d_in[:nq].view(h_q.shape)
        d_kv = d_in[nq:nq + nkv].view(kv_rows.shape)
        d_ik = d_in[nq + nkv:].view(ik_rows.shape)
        d_out = torch.empty(h_q.shape, dtype=torch.int16, device=dev)
        h_out = torch.empty(h_q.shape, dtype=torch.int16).pin_memory()
        d_in.copy_(h_in)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for l in range(N_LAYERS):
                pkv.decode(lay, step_seqs[p], l, HQ, d_q[l], d_out[l], cf["ws"], status=status,
                           k_new=d_kv[l, 0], v_new=d_kv[l, 1], ik_new=d_ik[l])
        graphs[p] = g
        ev = lambda: torch.cuda.Event()
        bufs[p] = {"d_in": d_in, "d_out": d_out, "h_out": h_out,
                   "in": ev(), "comp": ev(), "out": ev()}
    torch.cuda.synchronize()

    def step(first):
        # inputs: once the previous step's graph of the same page size has read
        # them; compute: once its inputs are in and its previous outputs are
        # out; outputs: once the graph has written them
        for p in pages:
            b = bufs[p]
            if not first:
                s_in.wait_event(b["comp"])
            with torch.cuda.stream(s_in):
                b["d_in"].copy_(h_in, non_blocking=True)
                b["in"].record(s_in)
        for p in pages:
            b = bufs[p]
            cur.wait_event(b["in"])
            if not first:
                cur.wait_event(b["out"])
            graphs[p].replay()
            b["comp"].record(cur)
            s_out.wait_event(b["comp"])
            with torch.cuda.stream(s_out):
                b["h_out"].copy_(b["d_out"], non_blocking=True)
                b["out"].record(s_out)

    for i in range(max(3, args.warmup)):
        step(i == 0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(10, args.steps // 4)
    e0.record(cur)
    s_in.wait_event(e0)
    for _ in range(n):
        step(False)
    cur.wait_stream(s_out)
    e1.record(cur)
    e1.synchronize()
    total = e0.elapsed_time(e1)
    for p in pages:
        if not torch.equal(bufs[p]["h_out"], bufs[pages[0]]["h_out"]):
            raise RuntimeError("end-to-end outputs differ between page sizes")
    step_bytes = sum(N_LAYERS * layer_bytes(lens_after, confs[p]["pages_used"]) for p in pages)
    h2d = len(pages) * h_in.numel() * 2
    d2h = len(pages) * h_q.numel() * 2
    return {"value": round(step_bytes / (total / n / 1e3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": n, "ms_per_step": round(total / n, 4),
            "copies": "every step copies each page size's inputs in and outputs out "
                      "(pinned host memory) on two copy streams, overlapping other "
                      "graphs' compute"}


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    return main_ours(args)


if __name__ == "__main__":
    sys.exit(main())
