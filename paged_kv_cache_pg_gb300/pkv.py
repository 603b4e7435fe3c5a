"""Thin ctypes binding of ``libpkv.so`` (the C ABI in ``include/pkv.h``).

Argument marshalling only: tensors become device pointers, lists of streams
become ``pkv_seq`` arrays, and the current torch CUDA stream is passed as the
launch stream.  Every step of the computation runs in the library's CUDA
kernels; there is no other path.  If the library is missing this module
raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import build as _build

K, V, IK, P, KS, VS = 0, 1, 2, 3, 4, 5
KV_BF16, KV_E4M3 = 0, 1
OK, EINVAL, EAGAIN, ECUDA, EDEVICE = 0, 1, 2, 3, 4
DEV_BAD_PAGE, DEV_TIMEOUT, DEV_SMEM, DEV_RANGE = 1, 2, 4, 8
MAX_SEQS = 64
_NAMES = {EINVAL: "PKV_EINVAL", EAGAIN: "PKV_EAGAIN", ECUDA: "PKV_ECUDA", EDEVICE: "PKV_EDEVICE"}


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {_NAMES.get(code, code)}")
        self.code = code


class Layout(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
                ("kv_format", ctypes.c_int32)]


class Pg(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("table", ctypes.c_void_p),
                ("page_elems", ctypes.c_int64), ("page_pos", ctypes.c_int32),
                ("n_pages", ctypes.c_int32), ("n_table", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class Seq(ctypes.Structure):
    _fields_ = [("pg", Pg), ("len", ctypes.c_int32), ("n_new", ctypes.c_int32)]


class EventOps(ctypes.Structure):
    RECORD = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.POINTER(ctypes.c_void_p))
    QUERY = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p)
    DESTROY = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)
    _fields_ = [("record", RECORD), ("query", QUERY), ("destroy", DESTROY),
                ("ctx", ctypes.c_void_p)]


_lib = None

EXPORTS = [
    "pkv_layout_page_elems", "pkv_pg_row", "pkv_arena_create", "pkv_arena_destroy",
    "pkv_arena_info", "pkv_pages_take", "pkv_pages_give", "pkv_arena_pg",
    "pkv_arena_set_event_ops", "pkv_run_pages", "pkv_run_take", "pkv_run_give", "pkv_run_map",
    "pkv_store", "pkv_gather", "pkv_pool", "pkv_decode_ws_size",
    "pkv_decode", "pkv_decode_static", "pkv_block_scores", "pkv_topk", "pkv_sparse_ws_size",
    "pkv_sparse_decode", "pkv_prefill_ws_size", "pkv_prefill", "pkv_diag_wait_runs_out",
    "pkv_diag_cta_wait_runs_out",
]


def library_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load the CUDA library (built in-tree by ``build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with paged_kv_cache_pg_gb300.build.build()")
    lib = ctypes.CDLL(p)
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    LP, PP, SP = ctypes.POINTER(Layout), ctypes.POINTER(Pg), ctypes.POINTER(Seq)
    sig = {
        "pkv_layout_page_elems": [LP, i32, ctypes.POINTER(i64)],
        "pkv_pg_row": [LP, PP, vp, i32, i32, i32, i32, ctypes.POINTER(i64)],
        "pkv_arena_create": [LP, i32, vp, sz, ctypes.POINTER(vp)],
        "pkv_arena_destroy": [vp],
        "pkv_arena_info": [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i64)],
        "pkv_pages_take": [vp, i32, vp],
        "pkv_pages_give": [vp, vp, i32, vp, i32],
        "pkv_arena_pg": [vp, vp, i32, PP],
        "pkv_arena_set_event_ops": [vp, ctypes.POINTER(EventOps)],
        "pkv_run_pages": [vp, ctypes.c_uint64, ctypes.POINTER(i32)],
        "pkv_run_take": [vp, i32, ctypes.POINTER(i32)],
        "pkv_run_give": [vp, i32, i32, vp, i32],
        "pkv_run_map": [vp, i32, i32, vp, i32, ctypes.c_uint64, vp],
        "pkv_store": [LP, SP, i32, i32, vp, vp, vp, vp, vp],
        "pkv_gather": [LP, SP, i32, i32, i32, vp, vp, vp],
        "pkv_pool": [LP, SP, i32, i32, vp, vp],
        "pkv_decode_ws_size": [LP, SP, i32, i32, ctypes.POINTER(sz)],
        "pkv_decode": [LP, SP, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp],
        "pkv_decode_static": [LP, SP, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp],
        "pkv_prefill_ws_size": [LP, SP, i32, i32, ctypes.POINTER(sz)],
        "pkv_prefill": [LP, SP, i32, i32, i32, vp, vp, vp, sz, vp, vp],
        "pkv_block_scores": [LP, SP, i32, i32, i32, vp, vp, i32, vp, vp],
        "pkv_topk": [SP, i32, i32, vp, i32, i32, vp, vp],
        "pkv_sparse_ws_size": [LP, SP, i32, i32, i32, ctypes.POINTER(sz)],
        "pkv_sparse_decode": [LP, SP, i32, i32, i32, vp, vp, i32, vp, vp, sz, vp, vp],
        "pkv_diag_wait_runs_out": [vp, vp],
        "pkv_diag_cta_wait_runs_out": [vp, i32, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise PkvError(rc, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _seqs(seqs: Sequence[Seq]):
    arr = (Seq * max(1, len(seqs)))(*seqs)
    return arr, len(seqs)


# ---- descriptors ------------------------------------------------------------

def layout(n_layers: int, n_kv_heads: int, head_dim: int = 256, idx_dim: int = 128,
           kv_format: int = KV_BF16) -> Layout:
    """kv_format KV_E4M3: K and V rows are e4m3 codes + a float32 scale each."""
    return Layout(n_layers, n_kv_heads, head_dim, idx_dim, kv_format)


def page_elems(lay: Layout, page_pos: int) -> int:
    out = ctypes.c_int64()
    _check(load().pkv_layout_page_elems(ctypes.byref(lay), page_pos, ctypes.byref(out)),
           "pkv_layout_page_elems")
    return out.value


def pg(base, table, page_elems_: int, page_pos: int, n_pages: int = 1,
       n_table: Optional[int] = None) -> Pg:
    """A stream's Pg: table None means a contiguous buffer of page_pos rows a head."""
    if table is None:
        return Pg(_ptr(base), None, page_elems_, page_pos, 1, 1, 0)
    nt = int(table.numel()) if n_table is None else n_table
    return Pg(_ptr(base), _ptr(table), page_elems_, page_pos, n_pages, nt, 0)


def seq(pg_: Pg, length: int, n_new: int) -> Seq:
    return Seq(pg_, length, n_new)


def pg_row(lay: Layout, pg_: Pg, host_table, layer: int, kind: int, head: int, pos: int) -> int:
    """Host pg_at: element offset of a row from pg.base; host_table is a numpy int32 array."""
    out = ctypes.c_int64()
    tab = None if host_table is None else host_table.ctypes.data
    _check(load().pkv_pg_row(ctypes.byref(lay), ctypes.byref(pg_), tab, layer, kind, head, pos,
                             ctypes.byref(out)), "pkv_pg_row")
    return out.value


class Arena:
    """The page pool over caller-owned device memory (a torch tensor)."""

    def __init__(self, lay: Layout, page_pos: int, memory, nbytes: Optional[int] = None):
        self._lib = load()
        self._h = ctypes.c_void_p()
        self.memory = memory
        n = nbytes if nbytes is not None else memory.numel() * memory.element_size()
        _check(self._lib.pkv_arena_create(ctypes.byref(lay), page_pos, _ptr(memory), n,
                                          ctypes.byref(self._h)), "pkv_arena_create")
        self._ops = None

    def close(self):
        if self._h:
            self._lib.pkv_arena_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self):
        n, f, e = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        _check(self._lib.pkv_arena_info(self._h, ctypes.byref(n), ctypes.byref(f),
                                        ctypes.byref(e)), "pkv_arena_info")
        return n.value, f.value, e.value

    def take(self, n: int):
        import numpy as np
        ids = np.zeros(max(1, n), dtype=np.int32)
        _check(self._lib.pkv_pages_take(self._h, n, ids.ctypes.data), "pkv_pages_take")
        return ids[:n]

    def give(self, ids, stream=None, defer: bool = True):
        import numpy as np
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        st = _stream(stream) if defer else (stream or 0)
        _check(self._lib.pkv_pages_give(self._h, ids.ctypes.data, ids.size, st, int(defer)),
               "pkv_pages_give")

    def run_pages(self, run_bytes: int) -> int:
        k = ctypes.c_int32()
        _check(self._lib.pkv_run_pages(self._h, run_bytes, ctypes.byref(k)), "pkv_run_pages")
        return k.value

    def run_take(self, k: int) -> int:
        first = ctypes.c_int32()
        _check(self._lib.pkv_run_take(self._h, k, ctypes.byref(first)), "pkv_run_take")
        return first.value

    def run_give(self, first: int, k: int, stream=None, defer: bool = True):
        st = _stream(stream) if defer else (stream or 0)
        _check(self._lib.pkv_run_give(self._h, first, k, st, int(defer)), "pkv_run_give")

    def run_map(self, first: int, k: int, part_bytes, align: int = 256):
        """Device addresses of the parts laid one after another in the run."""
        import numpy as np
        parts = np.ascontiguousarray(part_bytes, dtype=np.uint64)
        out = (ctypes.c_void_p * max(1, parts.size))()
        _check(self._lib.pkv_run_map(self._h, first, k, parts.ctypes.data, parts.size, align,
                                     out), "pkv_run_map")
        return [int(out[i] or 0) for i in range(parts.size)]

    def pg(self, dev_table, n_table: Optional[int] = None) -> Pg:
        out = Pg()
        nt = int(dev_table.numel()) if n_table is None else n_table
        _check(self._lib.pkv_arena_pg(self._h, _ptr(dev_table), nt, ctypes.byref(out)),
               "pkv_arena_pg")
        return out

    def set_event_ops(self, ops: Optional[EventOps]):
        self._ops = ops
        _check(self._lib.pkv_arena_set_event_ops(self._h, ctypes.byref(ops) if ops else None),
               "pkv_arena_set_event_ops")


# ---- kernels ------------------------------------------------------------------

def store(lay, seqs, layer, k_new, v_new, ik_new=None, status=None, stream=None):
    arr, n = _seqs(seqs)
    _check(load().pkv_store(ctypes.byref(lay), arr, n, layer, _ptr(k_new), _ptr(v_new),
                            _ptr(ik_new), _ptr(status), _stream(stream)), "pkv_store")


def gather(lay, seqs, layer, kind, out, status=None, stream=None):
    arr, n = _seqs(seqs)
    _check(load().pkv_gather(ctypes.byref(lay), arr, n, layer, kind, _ptr(out), _ptr(status),
                             _stream(stream)), "pkv_gather")


def pool(lay, seqs, layer, status=None, stream=None):
    arr, n = _seqs(seqs)
    _check(load().pkv_pool(ctypes.byref(lay), arr, n, layer, _ptr(status), _stream(stream)),
           "pkv_pool")


def decode_ws_size(lay, seqs, n_q_heads) -> int:
    arr, n = _seqs(seqs)
    out = ctypes.c_size_t()
    _check(load().pkv_decode_ws_size(ctypes.byref(lay), arr, n, n_q_heads, ctypes.byref(out)),
           "pkv_decode_ws_size")
    return out.value


def decode(lay, seqs, layer, n_q_heads, q, out, ws, status=None, stream=None, k_new=None,
           v_new=None, ik_new=None):
    """Decode attention; with k_new/v_new (and ik_new) the new rows are stored too."""
    arr, n = _seqs(seqs)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pkv_decode(ctypes.byref(lay), arr, n, layer, n_q_heads, _ptr(q), _ptr(k_new),
                             _ptr(v_new), _ptr(ik_new), _ptr(out), _ptr(ws), ws_bytes,
                             _ptr(status), _stream(stream)), "pkv_decode")


def prefill_ws_size(lay, seqs, n_q_heads) -> int:
    arr, n = _seqs(seqs)
    out = ctypes.c_size_t()
    _check(load().pkv_prefill_ws_size(ctypes.byref(lay), arr, n, n_q_heads, ctypes.byref(out)),
           "pkv_prefill_ws_size")
    return out.value


def prefill(lay, seqs, layer, n_q_heads, q, out, ws, status=None, stream=None):
    """Chunked-prefill attention on the tensor cores (the chunk already stored)."""
    arr, n = _seqs(seqs)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pkv_prefill(ctypes.byref(lay), arr, n, layer, n_q_heads, _ptr(q), _ptr(out),
                              _ptr(ws), ws_bytes, _ptr(status), _stream(stream)), "pkv_prefill")


STATIC_SCRATCH_BYTES = 4 << 20


def decode_static(lay, seqs, layer, n_q_heads, q, out, status=None, stream=None, k_new=None,
                  v_new=None, ik_new=None):
    """pkv_decode without a workspace: for callers that cannot allocate device
    memory.  The partials go to a fixed 4 MiB array inside the library; calls
    that run at the same time on the GPU share it, so issue them in order."""
    arr, n = _seqs(seqs)
    _check(load().pkv_decode_static(ctypes.byref(lay), arr, n, layer, n_q_heads, _ptr(q),
                                    _ptr(k_new), _ptr(v_new), _ptr(ik_new), _ptr(out),
                                    _ptr(status), _stream(stream)), "pkv_decode_static")


def block_scores(lay, seqs, layer, n_q_heads, qi, scores, ld, status=None, stream=None):
    arr, n = _seqs(seqs)
    _check(load().pkv_block_scores(ctypes.byref(lay), arr, n, layer, n_q_heads, _ptr(qi),
                                   _ptr(scores), ld, _ptr(status), _stream(stream)),
           "pkv_block_scores")


def topk(seqs, n_q_heads, scores, ld, k, ids, stream=None):
    arr, n = _seqs(seqs)
    _check(load().pkv_topk(arr, n, n_q_heads, _ptr(scores), ld, k, _ptr(ids), _stream(stream)),
           "pkv_topk")


def sparse_ws_size(lay, seqs, n_q_heads, k) -> int:
    arr, n = _seqs(seqs)
    out = ctypes.c_size_t()
    _check(load().pkv_sparse_ws_size(ctypes.byref(lay), arr, n, n_q_heads, k,
                                     ctypes.byref(out)), "pkv_sparse_ws_size")
    return out.value


def sparse_decode(lay, seqs, layer, n_q_heads, q, ids, k, out, ws, status=None, stream=None):
    arr, n = _seqs(seqs)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pkv_sparse_decode(ctypes.byref(lay), arr, n, layer, n_q_heads, _ptr(q),
                                    _ptr(ids), k, _ptr(out), _ptr(ws), ws_bytes, _ptr(status),
                                    _stream(stream)), "pkv_sparse_decode")


def diag_wait_runs_out(status, stream=None):
    """One warp's wait on a barrier nothing arrives on: it gives up after about
    a second and sets PKV_DEV_TIMEOUT in `status` (a device int32)."""
    _check(load().pkv_diag_wait_runs_out(_ptr(status), _stream(stream)), "pkv_diag_wait_runs_out")


def diag_cta_wait_runs_out(status, withheld_slice=2, stream=None):
    """A decode-shaped CTA (eight warps, four key slices, twelve stage slots)
    in which one slice's stage never lands: that slice's waits give up after
    about a second, the CTA returns as a whole and PKV_DEV_TIMEOUT is set in
    `status` (a device int32)."""
    _check(load().pkv_diag_cta_wait_runs_out(_ptr(status), withheld_slice, _stream(stream)),
           "pkv_diag_cta_wait_runs_out")
