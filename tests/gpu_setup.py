"""Shared set-up for the GPU parity tests.

The same synthetic streams are placed twice: into a device arena through the
library's own store kernel, and into a host arena through the oracle.  The
two arenas are then compared byte for byte, and the kernels' outputs are
compared with the oracle's.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

import oracle as orc
from paged_kv_cache_pg_gb300 import pkv, synth

CANARY = 0x7FC1      # bf16 NaN: a read of an unplaced row poisons the result
GUARD = 8192         # canary elements before and after every device buffer
ATOL, RTOL = 1e-3, 2e-3


def torch():
    import torch as t
    return t


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |ref| (8 significant bits): the representation
    error of a correctly rounded bf16 output."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def bound(ref: np.ndarray) -> np.ndarray:
    """Accumulation tolerance 1e-3 + 2e-3|ref| for float32-accumulated results,
    plus the half-ulp of the bf16 output format they are written in."""
    return ATOL + RTOL * np.abs(ref) + half_ulp_bf16(ref)


# Totals over every within_tol call of the session: elements checked,
# elements inside the bound only thanks to its half-ulp term, and the worst
# error of a passing check as a fraction of its bound (printed in the pytest
# summary by conftest.py).
TOL_STATS = {"calls": 0, "checked": 0, "needed_half_ulp": 0, "worst_frac_of_bound": 0.0}


def within_tol(gpu_bf16_bits: np.ndarray, ref: np.ndarray):
    """|gpu - ref| <= bound(ref) elementwise.

    Returns (ok, report); the report names the worst element, its index,
    the GPU value and the oracle value, how many elements fail, and how
    many pass only through the half-ulp term of the bound."""
    g = (gpu_bf16_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g = g.reshape(ref.shape)
    diff = np.abs(g - ref)
    err = diff - bound(ref)
    ok = bool((err <= 0).all() and np.isfinite(g).all())
    half = int(((diff > ATOL + RTOL * np.abs(ref)) & (err <= 0)).sum())
    frac = float(np.nanmax(np.where(np.isfinite(diff), diff / bound(ref), np.inf))) if ref.size else 0.0
    TOL_STATS["calls"] += 1
    TOL_STATS["checked"] += int(ref.size)
    TOL_STATS["needed_half_ulp"] += half
    if ok:   # red controls, which must fail, do not count
        TOL_STATS["worst_frac_of_bound"] = max(TOL_STATS["worst_frac_of_bound"], frac)
    i = np.unravel_index(int(np.nanargmax(np.where(np.isfinite(err), err, np.inf))), ref.shape)
    report = (f"worst excess {float(err[i]):.3g} at {tuple(int(x) for x in i)}: gpu {g[i]!r} "
              f"oracle {ref[i]!r}; {int((err > 0).sum())} of {err.size} outside; "
              f"{half} inside only through the half-ulp term; "
              f"non-finite {int((~np.isfinite(g)).sum())}")
    return ok, report


def dev_u16(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def host_u16(x) -> np.ndarray:
    return x.cpu().numpy().view(np.uint16)


@dataclass
class Placed:
    """Streams placed in device memory, and the same placement by the oracle."""
    lay: pkv.Layout
    shape: orc.Shape
    streams: List[synth.Stream]
    ptok: Optional[int]                 # None: each stream in its own contiguous buffer
    buffers: list = field(default_factory=list)     # device tensors with guards
    tables: list = field(default_factory=list)      # numpy tables (paged)
    dev_tables: list = field(default_factory=list)
    pgs: list = field(default_factory=list)
    ocaches: list = field(default_factory=list)
    oarenas: list = field(default_factory=list)

    def seqs(self, lens=None, n_new=None):
        lens = lens or [s.length for s in self.streams]
        n_new = n_new or [0] * len(lens)
        return [pkv.seq(g, L, n) for g, L, n in zip(self.pgs, lens, n_new)]

    def body(self, i=0):
        """The device buffer without its guards."""
        b = self.buffers[i]
        return b[GUARD:b.numel() - GUARD]

    def guards_intact(self) -> bool:
        for b in self.buffers:
            h = host_u16(b)
            if not ((h[:GUARD] == CANARY).all() and (h[-GUARD:] == CANARY).all()):
                return False
        return True


def _guarded(n_elems: int):
    t = torch()
    fill = int(np.array([CANARY], np.uint16).view(np.int16)[0])
    return t.full((n_elems + 2 * GUARD,), fill, dtype=t.int16, device="cuda")


def place(lay: pkv.Layout, streams: List[synth.Stream], ptok: Optional[int], seed: int = 0,
          spare_pages: int = 3, tables: Optional[list] = None, status=None) -> Placed:
    """Store every position of every stream, on the GPU and in the oracle."""
    t = torch()
    shape = orc.Shape(lay.n_layers, lay.n_kv_heads, lay.head_dim, lay.idx_dim, lay.kv_format)
    pl = Placed(lay, shape, streams, ptok)
    if ptok is None:
        for s in streams:
            cap = max(4, -(-s.length // 4) * 4)
            ps = pkv.page_elems(lay, cap)
            buf = _guarded(ps)
            pl.buffers.append(buf)
            body = buf[GUARD:GUARD + ps]
            pl.pgs.append(pkv.pg(body, None, ps, cap))
            oc = orc.contiguous(shape, cap, CANARY)
            pl.ocaches.append(oc)
            pl.oarenas.append(oc.base)
    else:
        ps = pkv.page_elems(lay, ptok)
        counts = [synth.pages_for(s.length, ptok) for s in streams]
        n_pages = sum(counts) + spare_pages
        if tables is None:
            tables = synth.shuffled_tables(seed, n_pages, counts)
        buf = _guarded(n_pages * ps)
        pl.buffers.append(buf)
        body = buf[GUARD:GUARD + n_pages * ps]
        oarena = np.full(n_pages * ps, CANARY, np.uint16)
        pl.oarenas.append(oarena)
        for tab in tables:
            dt = t.from_numpy(np.ascontiguousarray(tab, np.int32)).cuda()
            pl.tables.append(tab)
            pl.dev_tables.append(dt)
            pl.pgs.append(pkv.pg(body, dt, ps, ptok, n_pages, tab.size))
            pl.ocaches.append(orc.paged(shape, oarena, ptok, tab))
    # device: one store per layer of all positions of all streams
    seqs = [pkv.seq(g, s.length, s.length) for g, s in zip(pl.pgs, streams)]
    for layer in range(lay.n_layers):
        k = dev_u16(np.concatenate([s.k[layer] for s in streams]))
        v = dev_u16(np.concatenate([s.v[layer] for s in streams]))
        ik = dev_u16(np.concatenate([s.ik[layer] for s in streams])) if lay.idx_dim else None
        pkv.store(lay, seqs, layer, k, v, ik, status=status)
    # oracle: the same rows through its own translation
    put_kv = orc.put_rows8 if lay.kv_format == pkv.KV_E4M3 else orc.put_rows
    for oc, s in zip(pl.ocaches, streams):
        for layer in range(lay.n_layers):
            put_kv(shape, oc, layer, orc.K, 0, s.k[layer])
            put_kv(shape, oc, layer, orc.V, 0, s.v[layer])
            if lay.idx_dim:
                orc.put_rows(shape, oc, layer, orc.IK, 0, s.ik[layer])
    t.cuda.synchronize()
    return pl


def decode(pl: Placed, layer: int, n_q_heads: int, q_list: List[np.ndarray], lens=None,
           n_new=None, status=None):
    """Run pkv.decode; q_list[i] is stream i's [n_new][Hq][D] queries."""
    t = torch()
    n_new = n_new or [q.shape[0] for q in q_list]
    seqs = pl.seqs(lens, n_new)
    q = dev_u16(np.concatenate(q_list))
    out = t.zeros_like(q)
    ws_bytes = pkv.decode_ws_size(pl.lay, seqs, n_q_heads)
    ws = t.zeros(max(1, ws_bytes // 4 + 64), dtype=t.float32, device="cuda")
    pkv.decode(pl.lay, seqs, layer, n_q_heads, q, out, ws, status=status)
    t.cuda.synchronize()
    return host_u16(out)


def oracle_decode(pl: Placed, layer: int, n_q_heads: int, q_list, lens=None) -> np.ndarray:
    lens = lens or [s.length for s in pl.streams]
    outs = [orc.attend(pl.shape, oc, layer, n_q_heads, L, q)
            for oc, L, q in zip(pl.ocaches, lens, q_list)]
    return np.concatenate(outs)
