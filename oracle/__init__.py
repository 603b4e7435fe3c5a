"""CPU oracle for the paged KV-cache attention path.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library and its binding never
do.  It wraps ``pkv_oracle.c`` (plain single-threaded C, float64 attention)
through ctypes and shares no code with the CUDA path.

Caches are numpy ``uint16`` arrays (bf16 bit patterns; an e4m3-format
cache keeps its K and V codes and float32 scales in the same buffer, read as
bytes).  A :class:`Cache`
says where one stream's rows live: page 0 of an arena plus an int page table,
or a contiguous buffer of ``cap`` rows a head (``table=None``).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, the pages' printed pool sizes, invariants and brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_HDR = os.path.join(_HERE, "pkv_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

K, V, IK, P, KS, VS = 0, 1, 2, 3, 4, 5
BF16, E4M3 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-adds, no fast math)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Shape(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
                ("kv_format", ctypes.c_int32)]


class _Cache(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("n_table", ctypes.c_int32), ("ptok", ctypes.c_int32),
                ("ps", ctypes.c_int64), ("n_pages", ctypes.c_int32),
                ("pad_", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P_ = ctypes.POINTER
            sh, ca = P_(_Shape), P_(_Cache)
            i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            sig = {
                "orc_layer_elems": (i64, [sh, i32]),
                "orc_page_elems": (i64, [sh, i32]),
                "orc_row": (i64, [sh, ca, i32, i32, i32, i32]),
                "orc_put_rows": (ctypes.c_int, [sh, ca, i32, i32, i32, i32, vp]),
                "orc_get_rows": (ctypes.c_int, [sh, ca, i32, i32, i32, i32, vp]),
                "orc_bf16_round": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
                "orc_pool": (ctypes.c_int, [sh, ca, i32, i32, i32]),
                "orc_attend": (ctypes.c_int, [sh, ca, i32, i32, i32, i32, vp, vp]),
                "orc_attend_row": (ctypes.c_int, [sh, ca, i32, i32, i32, i32, vp, vp]),
                "orc_scores": (ctypes.c_int, [sh, ca, i32, i32, i32, vp, vp]),
                "orc_topk": (ctypes.c_int, [i32, i32, vp, i32, i32, vp]),
                "orc_sparse_attend": (ctypes.c_int, [sh, ca, i32, i32, i32, vp, vp, i32, vp]),
                "orc_e4m3_to_double": (ctypes.c_double, [ctypes.c_uint8]),
                "orc_e4m3_from_float": (ctypes.c_uint8, [ctypes.c_float]),
                "orc_e4m3_decode_n": (None, [vp, i64, vp]),
                "orc_e4m3_encode_n": (None, [vp, i64, vp]),
                "orc_quantize_row": (None, [vp, i32, vp, vp]),
                "orc_row8": (i64, [sh, ca, i32, i32, i32, i32]),
                "orc_put_rows8": (ctypes.c_int, [sh, ca, i32, i32, i32, i32, vp]),
                "orc_get_rows8": (ctypes.c_int, [sh, ca, i32, i32, i32, i32, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


@dataclass(frozen=True)
class Shape:
    n_layers: int
    n_kv_heads: int
    head_dim: int = 256
    idx_dim: int = 128
    kv_format: int = BF16

    def c(self) -> _Shape:
        return _Shape(self.n_layers, self.n_kv_heads, self.head_dim, self.idx_dim,
                      self.kv_format)


@dataclass
class Cache:
    """One stream's caches: ``base`` is the arena (or the stream's own buffer)."""
    base: np.ndarray                 # uint16, writable
    ptok: int                        # positions a page (cap when contiguous)
    ps: int                          # elements a page
    table: Optional[np.ndarray] = None   # int32 page ids, or None
    n_pages: int = 1

    def c(self) -> _Cache:
        assert self.base.dtype == np.uint16 and self.base.flags.c_contiguous
        tab = None
        n_table = 0
        if self.table is not None:
            assert self.table.dtype == np.int32 and self.table.flags.c_contiguous
            tab = self.table.ctypes.data
            n_table = int(self.table.size)
        return _Cache(self.base.ctypes.data, tab, n_table, self.ptok, self.ps,
                      self.n_pages, 0)


def _chk(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: a row falls outside the cache")


def layer_elems(shape: Shape, ptok: int) -> int:
    return int(_load().orc_layer_elems(ctypes.byref(shape.c()), ptok))


def page_elems(shape: Shape, ptok: int) -> int:
    return int(_load().orc_page_elems(ctypes.byref(shape.c()), ptok))


def contiguous(shape: Shape, cap: int, fill: int = 0) -> Cache:
    """A stream's own buffer of cap rows a head (one page with ptok = cap)."""
    ps = page_elems(shape, cap)
    return Cache(np.full(ps, fill, dtype=np.uint16), cap, ps, None, 1)


def paged(shape: Shape, arena: np.ndarray, ptok: int, table: np.ndarray) -> Cache:
    ps = page_elems(shape, ptok)
    assert arena.size % ps == 0
    return Cache(arena, ptok, ps, np.ascontiguousarray(table, dtype=np.int32),
                 arena.size // ps)


def row(shape: Shape, cache: Cache, layer: int, kind: int, head: int, pos: int) -> int:
    """Element offset of a row from the cache's base (-1: outside)."""
    return int(_load().orc_row(ctypes.byref(shape.c()), ctypes.byref(cache.c()),
                               layer, kind, head, pos))


def _row_len(shape: Shape, kind: int) -> int:
    return shape.head_dim if kind in (K, V) else shape.idx_dim


def _heads(shape: Shape, kind: int) -> int:
    return shape.n_kv_heads if kind in (K, V) else 1


def put_rows(shape: Shape, cache: Cache, layer: int, kind: int, pos0: int,
             rows: np.ndarray) -> None:
    """Store rows ([n][heads][row] for K/V, [n][row] otherwise) at pos0.."""
    rows = np.ascontiguousarray(rows, dtype=np.uint16)
    n = rows.size // (_heads(shape, kind) * _row_len(shape, kind))
    _chk(_load().orc_put_rows(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                              kind, pos0, n, rows.ctypes.data), "put_rows")


def get_rows(shape: Shape, cache: Cache, layer: int, kind: int, pos0: int, n: int) -> np.ndarray:
    h, r = _heads(shape, kind), _row_len(shape, kind)
    out = np.zeros((n, h, r) if kind in (K, V) else (n, r), dtype=np.uint16)
    _chk(_load().orc_get_rows(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                              kind, pos0, n, out.ctypes.data), "get_rows")
    return out


def bf16_round(x: float) -> int:
    return int(_load().orc_bf16_round(ctypes.c_float(x)))


def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly (a bit shift; no arithmetic)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def pool(shape: Shape, cache: Cache, layer: int, block0: int, n_blocks: int) -> None:
    _chk(_load().orc_pool(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                          block0, n_blocks), "pool")


def attend(shape: Shape, cache: Cache, layer: int, n_q_heads: int, length: int,
           q: np.ndarray) -> np.ndarray:
    """Causal attention of the last nq positions; q bf16 [nq][Hq][D] -> float64."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    nq = q.shape[0]
    out = np.zeros((nq, n_q_heads, shape.head_dim), dtype=np.float64)
    _chk(_load().orc_attend(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                            n_q_heads, length, nq, q.ctypes.data, out.ctypes.data), "attend")
    return out


def attend_row(shape: Shape, cache: Cache, layer: int, n_q_heads: int, head: int,
               pos: int, q_row: np.ndarray) -> np.ndarray:
    q_row = np.ascontiguousarray(q_row, dtype=np.uint16)
    out = np.zeros(shape.head_dim, dtype=np.float64)
    _chk(_load().orc_attend_row(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                                n_q_heads, head, pos, q_row.ctypes.data, out.ctypes.data),
         "attend_row")
    return out


def scores(shape: Shape, cache: Cache, layer: int, n_q_heads: int, length: int,
           qi: np.ndarray) -> np.ndarray:
    qi = np.ascontiguousarray(qi, dtype=np.uint16)
    nb = length // 4
    out = np.zeros((n_q_heads, nb), dtype=np.float32)
    _chk(_load().orc_scores(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                            n_q_heads, length, qi.ctypes.data, out.ctypes.data), "scores")
    return out


def topk(scores_: np.ndarray, k: int, nb: Optional[int] = None) -> np.ndarray:
    s = np.ascontiguousarray(scores_, dtype=np.float32)
    rows, ld = s.shape
    nb = ld if nb is None else nb
    ids = np.zeros((rows, k), dtype=np.int32)
    _chk(_load().orc_topk(rows, nb, s.ctypes.data, ld, k, ids.ctypes.data), "topk")
    return ids


def sparse_attend(shape: Shape, cache: Cache, layer: int, n_q_heads: int, length: int,
                  q: np.ndarray, ids: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    k = ids.shape[1]
    out = np.zeros((n_q_heads, shape.head_dim), dtype=np.float64)
    _chk(_load().orc_sparse_attend(ctypes.byref(shape.c()), ctypes.byref(cache.c()),
                                   layer, n_q_heads, length, q.ctypes.data,
                                   ids.ctypes.data, k, out.ctypes.data), "sparse_attend")
    return out


# ---- e4m3 K/V (codes + float32 scale per head and row) ---------------------

def e4m3_to_double(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(c.shape, dtype=np.float64)
    _load().orc_e4m3_decode_n(c.ctypes.data, c.size, out.ctypes.data)
    return out


def e4m3_from_float(x) -> np.ndarray:
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(f.shape, dtype=np.uint8)
    _load().orc_e4m3_encode_n(f.ctypes.data, f.size, out.ctypes.data)
    return out


def quantize_row(row_bf16: np.ndarray):
    """(codes uint8 [n], scale float32) of one bf16 row."""
    r = np.ascontiguousarray(row_bf16, dtype=np.uint16)
    codes = np.zeros(r.size, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.float32)
    _load().orc_quantize_row(r.ctypes.data, r.size, codes.ctypes.data, sc.ctypes.data)
    return codes, sc[0]


def row8(shape: Shape, cache: Cache, layer: int, kind: int, head: int, pos: int) -> int:
    """Byte offset of a row of an e4m3-format cache from its base (-1: outside)."""
    return int(_load().orc_row8(ctypes.byref(shape.c()), ctypes.byref(cache.c()),
                                layer, kind, head, pos))


def put_rows8(shape: Shape, cache: Cache, layer: int, kind: int, pos0: int,
              rows: np.ndarray) -> None:
    """Quantize and store bf16 K or V rows [n][heads][head_dim] at pos0.."""
    rows = np.ascontiguousarray(rows, dtype=np.uint16)
    n = rows.size // (shape.n_kv_heads * shape.head_dim)
    _chk(_load().orc_put_rows8(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                               kind, pos0, n, rows.ctypes.data), "put_rows8")


def get_rows8(shape: Shape, cache: Cache, layer: int, kind: int, pos0: int, n: int) -> np.ndarray:
    """Codes (K, V: uint8 [n][heads][head_dim]) or scales (KS, VS: float32 [n][heads])."""
    if kind in (KS, VS):
        out = np.zeros((n, shape.n_kv_heads), dtype=np.float32)
    else:
        out = np.zeros((n, shape.n_kv_heads, shape.head_dim), dtype=np.uint8)
    _chk(_load().orc_get_rows8(ctypes.byref(shape.c()), ctypes.byref(cache.c()), layer,
                               kind, pos0, n, out.ctypes.data), "get_rows8")
    return out
