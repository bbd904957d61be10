"""Thin Python binding of libgdnspec (ctypes): argument marshalling only.

Every function has the name of its C entry point (``include/gdnspec.h``) and
takes the same arguments; device buffers may be given as torch tensors (their
``data_ptr()`` is passed) or as integer addresses.  Nothing here computes any
part of the method: every step runs in the library's CUDA kernels or in its
host planner.  A non-zero return code raises :class:`GdnError`.

The library must have been built (``python -m speculative_decoding_hybrid_gb300.build``
or ``__graft_entry__.build()``); importing this module without it fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdnspec.so")

GDN_OK, GDN_ERR_NULL, GDN_ERR_SHAPE, GDN_ERR_ARG = 0, -1, -2, -3
GDN_ERR_DUP_SLOT, GDN_ERR_NO_SLOT, GDN_ERR_CUDA, GDN_ERR_WORKSPACE, GDN_ERR_REFUSED = -4, -5, -6, -7, -8
DEV_SLOT_OOR, DEV_ROWS_BAD, DEV_TOKEN_OOR, DEV_CKPT_UNWRITTEN, DEV_ACCEPT_BAD, DEV_TIMEOUT = 1, 2, 4, 8, 16, 32
K_MAX = 15
MAX_ROWS = K_MAX + 1
REQ_DECODE, REQ_PREFILL = 0, 1
PLAN_RECURRENT, PLAN_CHUNKED = 0, 1

EXPORTS = ["gdn_decode_step", "gdn_verify", "mtp_accept_workspace_bytes", "mtp_greedy_accept",
           "mtp_greedy_accept_noalloc", "gdn_commit", "gdn_verify_at", "gdn_commit_at", "gdn_materialize",
           "gdn_verify_replay", "gdn_selftest_wait_timeout", "gdn_verify_layers", "gdn_verify_at_layers",
           "gdn_verify_replay_layers",
           "gdn_prefill_workspace_bytes", "gdn_chunked_prefill", "gdn_pool_init", "gdn_pool_alloc",
           "gdn_pool_share", "gdn_pool_release", "plan_transaction", "gdn_pool_apply", "gdn_pool_abort",
           "gdn_decode_transaction", "gdn_decode_transaction_at", "gdn_status_string",
           "gdn_selftest_prefill_timeout"]


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, status_string(status), status))


class gdn_dims(ctypes.Structure):
    _fields_ = [("h_qk", ctypes.c_int32), ("h_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("q_scale", ctypes.c_float)]


class mtp_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("proposed", "evaluated", "accepted", "emitted", "steps")]


class gdn_layer_rows(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "g", "beta")]


def layer_rows_array(rows) -> ctypes.Array:
    """Host array of gdn_layer_rows from objects with q, k, v, g, beta tensors."""
    arr = (gdn_layer_rows * max(len(rows), 1))()
    for i, r in enumerate(rows):
        arr[i] = gdn_layer_rows(_ptr(r.q), _ptr(r.k), _ptr(r.v), _ptr(r.g), _ptr(r.beta))
    return arr


class gdn_req(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kind", "k_draft", "n_tokens", "cur_len", "max_len", "slot")]


class gdn_plan_limits(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("max_rows", "max_reqs", "k_max")]


_I32P = ctypes.POINTER(ctypes.c_int32)


class gdn_pool(ctypes.Structure):
    _fields_ = [("num_slots", ctypes.c_int32), ("refcount", _I32P), ("free_fifo", _I32P),
                ("free_head", ctypes.c_int32), ("free_count", ctypes.c_int32)]


class gdn_plan(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int32) for n in ("n_selected", "plan", "deferred", "n_decode", "decode_rows",
                                                "n_prefill", "prefill_rows")] +
                [(n, _I32P) for n in ("k", "rows", "src", "dst", "dec_req", "dec_cu", "dec_src", "dec_dst",
                                      "pre_req", "pre_cu", "pre_src", "pre_dst")])


class gdn_decode_io(ctypes.Structure):
    _fields_ = [("tables", ctypes.c_void_p), ("rows", ctypes.c_void_p), ("pool", ctypes.c_void_p),
                ("slot_stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64), ("num_slots", ctypes.c_int32),
                ("ckpt", ctypes.c_void_p), ("ckpt_layer_stride", ctypes.c_int64), ("ckpt_tag", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("o_layer_stride", ctypes.c_int64), ("logits", ctypes.c_void_p),
                ("vocab", ctypes.c_int64), ("logit_row_stride", ctypes.c_int64), ("tokens", ctypes.c_void_p),
                ("argmax", ctypes.c_void_p), ("accept_len", ctypes.c_void_p), ("bonus", ctypes.c_void_p),
                ("out_tokens", ctypes.c_void_p), ("stats", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("dev_status", ctypes.c_void_p),
                ("host_tables", ctypes.c_void_p), ("host_out", ctypes.c_void_p)]


class gdn_arena_io(ctypes.Structure):
    _fields_ = [("arena", ctypes.c_void_p), ("elems_total", ctypes.c_int64), ("loc", ctypes.c_void_p),
                ("area_off", ctypes.c_int64 * 2)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libgdnspec.so is not built (expected at %s); run "
                          "`python -m speculative_decoding_hybrid_gb300.build`" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P, I32, I64, U32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    DP = ctypes.POINTER(gdn_dims)
    sig = {
        "gdn_decode_step": [DP, I32, P, P, P, P, P, P, I64, I32, P, P, P, P, P],
        "gdn_verify": [DP, I32, I32, P, P, P, P, P, P, P, I64, I32, P, P, P, U32, P, P, P],
        "mtp_accept_workspace_bytes": [I32, I64],
        "mtp_greedy_accept": [I32, I32, P, P, I64, I64, P, P, P, P, P, P, P, SZ, P, P],
        "mtp_greedy_accept_noalloc": [I32, I32, P, P, I64, I64, P, P, P, P, P, P, P, P],
        "gdn_commit": [DP, I32, I32, I32, P, P, P, I64, P, U32, P, I64, I64, I32, P, P, P],
        "gdn_verify_at": [DP, I32, I32, P, P, P, P, P, P, P, I64, P, P, P, U32, P, P, P],
        "gdn_commit_at": [DP, I32, I32, I32, P, P, I64, I64, P, U32, P, P, P],
        "gdn_materialize": [DP, I32, I32, P, I64, P, P, I64, I64, I32, P, P, P],
        "gdn_verify_replay": [DP, I32, I32, P, P, P, P, P, P, I32, P, P, P, P, P, P, P, I64, I32, P, P, P, P, P],
        "gdn_prefill_workspace_bytes": [DP, I32, I32],
        "gdn_chunked_prefill": [DP, I32, I32, P, I32, P, P, P, P, P, P, I64, I32, P, P, P, I32, P, SZ, P, P],
        "gdn_pool_init": [ctypes.POINTER(gdn_pool), I32, P, P, P],
        "gdn_pool_alloc": [ctypes.POINTER(gdn_pool), _I32P],
        "gdn_pool_share": [ctypes.POINTER(gdn_pool), I32],
        "gdn_pool_release": [ctypes.POINTER(gdn_pool), I32],
        "plan_transaction": [ctypes.POINTER(gdn_req), I32, ctypes.POINTER(gdn_plan_limits),
                             ctypes.POINTER(gdn_pool), ctypes.POINTER(gdn_plan)],
        "gdn_pool_apply": [ctypes.POINTER(gdn_pool), ctypes.POINTER(gdn_plan), I32],
        "gdn_pool_abort": [ctypes.POINTER(gdn_pool), ctypes.POINTER(gdn_plan), I32],
        "gdn_status_string": [ctypes.c_int],
        "gdn_verify_layers": [DP, I32, I32, I32, P, P, P, I64, I64, I32, P, P, I64, P, U32, P, I64, P, P],
        "gdn_verify_at_layers": [DP, I32, I32, I32, P, P, P, I64, P, P, I64, P, U32, P, I64, P, P],
        "gdn_verify_replay_layers": [DP, I32, I32, I32, P, P, I32, P, P, P, P, I64, I64, I32, P, P, P, I64, P, P],
        "gdn_selftest_wait_timeout": [P, ctypes.c_uint64, P],
        "gdn_selftest_prefill_timeout": [DP, I32, I32, P, P, P, P, P, P, P, I64, I32, P, P, P, P, SZ, P,
                                         ctypes.c_uint64, P],
        "gdn_decode_transaction": [DP, I32, I32, ctypes.POINTER(gdn_req), I32, ctypes.POINTER(gdn_plan_limits),
                                   ctypes.POINTER(gdn_pool), ctypes.POINTER(gdn_plan), ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.POINTER(gdn_decode_io), P, P],
        "gdn_decode_transaction_at": [DP, I32, I32, ctypes.POINTER(gdn_req), I32, ctypes.POINTER(gdn_plan_limits),
                                      ctypes.POINTER(gdn_pool), ctypes.POINTER(gdn_plan),
                                      ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(gdn_decode_io),
                                      ctypes.POINTER(gdn_arena_io), P, P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.mtp_accept_workspace_bytes.restype = SZ
    L.gdn_prefill_workspace_bytes.restype = SZ
    L.gdn_status_string.restype = ctypes.c_char_p
    return L


lib = _load()


def status_string(st: int) -> str:
    return lib.gdn_status_string(int(st)).decode()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError("expected a tensor, an array or an address, got %r" % type(x))


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, st: int) -> int:
    if st != GDN_OK:
        raise GdnError(fn, st)
    return st


def dims(h_qk: int, h_v: int, d_k: int, d_v: int, q_scale: float = 1.0) -> gdn_dims:
    return gdn_dims(h_qk, h_v, d_k, d_v, q_scale)


# ---------------------------------------------------------------------------
# Device entry points
# ---------------------------------------------------------------------------

def gdn_decode_step(d: gdn_dims, B, q, k, v, g, beta, pool_layer, slot_stride, num_slots, src_slot, dst_slot, o,
                    dev_status, stream=None):
    return _check("gdn_decode_step", lib.gdn_decode_step(
        ctypes.byref(d), B, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool_layer), slot_stride,
        num_slots, _ptr(src_slot), _ptr(dst_slot), _ptr(o), _ptr(dev_status), _stream(stream)))


def gdn_verify(d: gdn_dims, B, row_capacity, cu_rows, q, k, v, g, beta, pool_layer, slot_stride, num_slots,
               src_slot, ckpt_layer, ckpt_tag, txn, o, dev_status, stream=None):
    return _check("gdn_verify", lib.gdn_verify(
        ctypes.byref(d), B, row_capacity, _ptr(cu_rows), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(pool_layer), slot_stride, num_slots, _ptr(src_slot), _ptr(ckpt_layer), _ptr(ckpt_tag), txn, _ptr(o),
        _ptr(dev_status), _stream(stream)))


def mtp_accept_workspace_bytes(row_capacity: int, vocab: int) -> int:
    return int(lib.mtp_accept_workspace_bytes(row_capacity, vocab))


def mtp_greedy_accept(B, row_capacity, cu_rows, logits, vocab, row_stride, tokens, argmax, accept_len, bonus,
                      out_tokens, stats, workspace, workspace_bytes, dev_status, stream=None):
    return _check("mtp_greedy_accept", lib.mtp_greedy_accept(
        B, row_capacity, _ptr(cu_rows), _ptr(logits), vocab, row_stride, _ptr(tokens), _ptr(argmax),
        _ptr(accept_len), _ptr(bonus), _ptr(out_tokens), _ptr(stats), _ptr(workspace), workspace_bytes,
        _ptr(dev_status), _stream(stream)))


def mtp_greedy_accept_noalloc(B, row_capacity, cu_rows, logits, vocab, row_stride, tokens, argmax, accept_len,
                              bonus, out_tokens, stats, dev_status, stream=None):
    """mtp_greedy_accept with the library's fixed device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    return _check("mtp_greedy_accept_noalloc", lib.mtp_greedy_accept_noalloc(
        B, row_capacity, _ptr(cu_rows), _ptr(logits), vocab, row_stride, _ptr(tokens), _ptr(argmax),
        _ptr(accept_len), _ptr(bonus), _ptr(out_tokens), _ptr(stats), _ptr(dev_status), _stream(stream)))


def gdn_commit(d: gdn_dims, B, num_layers, row_capacity, cu_rows, accept_len, ckpt, ckpt_layer_stride, ckpt_tag,
               txn, pool, slot_stride, layer_stride, num_slots, dst_slot, dev_status, stream=None):
    return _check("gdn_commit", lib.gdn_commit(
        ctypes.byref(d), B, num_layers, row_capacity, _ptr(cu_rows), _ptr(accept_len), _ptr(ckpt),
        ckpt_layer_stride, _ptr(ckpt_tag), txn, _ptr(pool), slot_stride, layer_stride, num_slots, _ptr(dst_slot),
        _ptr(dev_status), _stream(stream)))


def gdn_verify_at(d: gdn_dims, B, row_capacity, cu_rows, q, k, v, g, beta, state_base, state_elems_total, src_off,
                  ckpt_layer, ckpt_tag, txn, o, dev_status, stream=None):
    return _check("gdn_verify_at", lib.gdn_verify_at(
        ctypes.byref(d), B, row_capacity, _ptr(cu_rows), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(state_base), state_elems_total, _ptr(src_off), _ptr(ckpt_layer), _ptr(ckpt_tag), txn, _ptr(o),
        _ptr(dev_status), _stream(stream)))


def gdn_commit_at(d: gdn_dims, B, num_layers, row_capacity, cu_rows, accept_len, ckpt_off, ckpt_layer_stride,
                  ckpt_tag, txn, loc, dev_status, stream=None):
    return _check("gdn_commit_at", lib.gdn_commit_at(
        ctypes.byref(d), B, num_layers, row_capacity, _ptr(cu_rows), _ptr(accept_len), ckpt_off, ckpt_layer_stride,
        _ptr(ckpt_tag), txn, _ptr(loc), _ptr(dev_status), _stream(stream)))


def gdn_materialize(d: gdn_dims, B, num_layers, state_base, state_elems_total, loc, pool, slot_stride, layer_stride,
                    num_slots, dst_slot, dev_status, stream=None):
    return _check("gdn_materialize", lib.gdn_materialize(
        ctypes.byref(d), B, num_layers, _ptr(state_base), state_elems_total, _ptr(loc), _ptr(pool), slot_stride,
        layer_stride, num_slots, _ptr(dst_slot), _ptr(dev_status), _stream(stream)))


def gdn_verify_replay(d: gdn_dims, B, row_capacity, cu_rows, q, k, v, g, beta, prev_capacity, prev_cu_rows,
                      prev_accept_len, prev_k, prev_v, prev_g, prev_beta, pool_layer, slot_stride, num_slots, src_slot,
                      dst_slot, o, dev_status, stream=None):
    return _check("gdn_verify_replay", lib.gdn_verify_replay(
        ctypes.byref(d), B, row_capacity, _ptr(cu_rows), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        prev_capacity, _ptr(prev_cu_rows), _ptr(prev_accept_len), _ptr(prev_k), _ptr(prev_v), _ptr(prev_g),
        _ptr(prev_beta), _ptr(pool_layer), slot_stride, num_slots, _ptr(src_slot), _ptr(dst_slot), _ptr(o),
        _ptr(dev_status), _stream(stream)))


def gdn_prefill_workspace_bytes(d: gdn_dims, nseq: int, row_capacity: int) -> int:
    return int(lib.gdn_prefill_workspace_bytes(ctypes.byref(d), nseq, row_capacity))


def gdn_chunked_prefill(d: gdn_dims, nseq, row_capacity, cu_seqlens, max_seqlen, q, k, v, g, beta, pool_layer,
                        slot_stride, num_slots, src_slot, dst_slot, o, chunk, workspace, workspace_bytes,
                        dev_status, stream=None):
    return _check("gdn_chunked_prefill", lib.gdn_chunked_prefill(
        ctypes.byref(d), nseq, row_capacity, _ptr(cu_seqlens), max_seqlen, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
        _ptr(beta), _ptr(pool_layer), slot_stride, num_slots, _ptr(src_slot), _ptr(dst_slot), _ptr(o), chunk,
        _ptr(workspace), workspace_bytes, _ptr(dev_status), _stream(stream)))


def gdn_verify_layers(d: gdn_dims, num_layers, B, row_capacity, cu_rows, rows, pool, slot_stride, layer_stride,
                      num_slots, src_slot, ckpt, ckpt_layer_stride, ckpt_tag, txn, o, o_layer_stride, dev_status,
                      stream=None):
    """``rows``: a ctypes array from layer_rows_array (kept alive by the caller)."""
    return _check("gdn_verify_layers", lib.gdn_verify_layers(
        ctypes.byref(d), num_layers, B, row_capacity, _ptr(cu_rows), ctypes.cast(rows, ctypes.c_void_p), _ptr(pool),
        slot_stride, layer_stride, num_slots, _ptr(src_slot), _ptr(ckpt), ckpt_layer_stride, _ptr(ckpt_tag), txn,
        _ptr(o), o_layer_stride, _ptr(dev_status), _stream(stream)))


def gdn_decode_transaction(d: gdn_dims, num_layers, row_capacity, reqs, n_reqs, lim, pool, plan, txn, io,
                           kernel_ms=None, stream=None):
    """``reqs``: a gdn_req array; ``lim``: gdn_plan_limits; ``pool``, ``plan``:
    Pool and Plan objects; ``txn``: a ctypes.c_uint32 (updated);
    ``io``: a gdn_decode_io; ``kernel_ms``: None or a ctypes float array of 3."""
    return _check("gdn_decode_transaction", lib.gdn_decode_transaction(
        ctypes.byref(d), num_layers, row_capacity, reqs, n_reqs, ctypes.byref(lim), ctypes.byref(pool.c),
        ctypes.byref(plan.c), ctypes.byref(txn), ctypes.byref(io),
        None if kernel_ms is None else ctypes.cast(kernel_ms, ctypes.c_void_p), _stream(stream)))


def gdn_decode_transaction_at(d: gdn_dims, num_layers, row_capacity, reqs, n_reqs, lim, pool, plan, txn, io, arena,
                              kernel_ms=None, stream=None):
    """gdn_decode_transaction over a state arena; ``arena``: a gdn_arena_io."""
    return _check("gdn_decode_transaction_at", lib.gdn_decode_transaction_at(
        ctypes.byref(d), num_layers, row_capacity, reqs, n_reqs, ctypes.byref(lim), ctypes.byref(pool.c),
        ctypes.byref(plan.c), ctypes.byref(txn), ctypes.byref(io), ctypes.byref(arena),
        None if kernel_ms is None else ctypes.cast(kernel_ms, ctypes.c_void_p), _stream(stream)))


def gdn_verify_at_layers(d: gdn_dims, num_layers, B, row_capacity, cu_rows, rows, state_base, state_elems_total,
                         src_off, ckpt, ckpt_layer_stride, ckpt_tag, txn, o, o_layer_stride, dev_status, stream=None):
    return _check("gdn_verify_at_layers", lib.gdn_verify_at_layers(
        ctypes.byref(d), num_layers, B, row_capacity, _ptr(cu_rows), ctypes.cast(rows, ctypes.c_void_p),
        _ptr(state_base), state_elems_total, _ptr(src_off), _ptr(ckpt), ckpt_layer_stride, _ptr(ckpt_tag), txn,
        _ptr(o), o_layer_stride, _ptr(dev_status), _stream(stream)))


def gdn_verify_replay_layers(d: gdn_dims, num_layers, B, row_capacity, cu_rows, rows, prev_capacity, prev_cu_rows,
                             prev_accept_len, prev_rows, pool, slot_stride, layer_stride, num_slots, src_slot,
                             dst_slot, o, o_layer_stride, dev_status, stream=None):
    return _check("gdn_verify_replay_layers", lib.gdn_verify_replay_layers(
        ctypes.byref(d), num_layers, B, row_capacity, _ptr(cu_rows), ctypes.cast(rows, ctypes.c_void_p),
        prev_capacity, _ptr(prev_cu_rows), _ptr(prev_accept_len), ctypes.cast(prev_rows, ctypes.c_void_p),
        _ptr(pool), slot_stride, layer_stride, num_slots, _ptr(src_slot), _ptr(dst_slot), _ptr(o), o_layer_stride,
        _ptr(dev_status), _stream(stream)))


def gdn_selftest_wait_timeout(dev_status, limit_ns: int, stream=None):
    return _check("gdn_selftest_wait_timeout",
                  lib.gdn_selftest_wait_timeout(_ptr(dev_status), int(limit_ns), _stream(stream)))


def gdn_selftest_prefill_timeout(d: gdn_dims, nseq, row_capacity, cu_seqlens, q, k, v, g, beta, pool_layer,
                                 slot_stride, num_slots, src_slot, dst_slot, o, workspace, workspace_bytes,
                                 dev_status, limit_ns: int, stream=None):
    return _check("gdn_selftest_prefill_timeout", lib.gdn_selftest_prefill_timeout(
        ctypes.byref(d), nseq, row_capacity, _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(pool_layer), slot_stride, num_slots, _ptr(src_slot), _ptr(dst_slot), _ptr(o), _ptr(workspace),
        workspace_bytes, _ptr(dev_status), int(limit_ns), _stream(stream)))


# ---------------------------------------------------------------------------
# Host planner and slot pool (host memory)
# ---------------------------------------------------------------------------

class Pool:
    """Owns the host arrays of a gdn_pool."""

    def __init__(self, num_slots: int, free_order=None):
        self.refcount = np.zeros(num_slots, dtype=np.int32)
        self.fifo = np.zeros(num_slots, dtype=np.int32)
        self._order = None if free_order is None else np.ascontiguousarray(free_order, dtype=np.int32)
        self.c = gdn_pool()
        _check("gdn_pool_init", lib.gdn_pool_init(ctypes.byref(self.c), num_slots, self.refcount.ctypes.data,
                                                  self.fifo.ctypes.data,
                                                  None if self._order is None else self._order.ctypes.data))

    def alloc(self) -> int:
        s = ctypes.c_int32(-1)
        _check("gdn_pool_alloc", lib.gdn_pool_alloc(ctypes.byref(self.c), ctypes.byref(s)))
        return s.value

    def share(self, slot: int):
        return _check("gdn_pool_share", lib.gdn_pool_share(ctypes.byref(self.c), slot))

    def release(self, slot: int) -> int:
        return int(lib.gdn_pool_release(ctypes.byref(self.c), slot))

    def free_list(self):
        n = self.c.num_slots
        return [int(self.fifo[(self.c.free_head + i) % n]) for i in range(self.c.free_count)]


class Plan:
    """Owns the host arrays of a gdn_plan for up to n requests."""

    def __init__(self, n: int):
        self.n = n
        m = max(n, 1)
        self.arrays = {k: np.zeros(m + (1 if k in ("dec_cu", "pre_cu") else 0), dtype=np.int32)
                       for k in ("k", "rows", "src", "dst", "dec_req", "dec_cu", "dec_src", "dec_dst", "pre_req",
                                 "pre_cu", "pre_src", "pre_dst")}
        self.c = gdn_plan()
        for k, a in self.arrays.items():
            setattr(self.c, k, a.ctypes.data_as(_I32P))

    def __getattr__(self, name):
        arrays = self.__dict__.get("arrays", {})
        if name in arrays:
            a = arrays[name]
            if name in ("k", "rows", "src", "dst"):
                return a[:self.n].tolist()
            if name == "dec_cu":
                return a[:self.c.n_decode + 1].tolist()
            if name == "pre_cu":
                return a[:self.c.n_prefill + 1].tolist()
            cnt = self.c.n_decode if name.startswith("dec") else self.c.n_prefill
            return a[:cnt].tolist()
        c = self.__dict__.get("c")
        if c is not None and name in dict(gdn_plan._fields_):
            return getattr(c, name)
        raise AttributeError(name)


def make_reqs(reqs) -> ctypes.Array:
    arr = (gdn_req * max(len(reqs), 1))()
    for i, r in enumerate(reqs):
        arr[i] = gdn_req(*r) if isinstance(r, (tuple, list)) else r
    return arr


def plan_transaction(reqs, n: int, lim: gdn_plan_limits, pool: Pool, plan: Plan) -> int:
    """Returns the status (not raised: planner refusals are part of the contract)."""
    return int(lib.plan_transaction(reqs, n, ctypes.byref(lim), ctypes.byref(pool.c), ctypes.byref(plan.c)))


def gdn_pool_apply(pool: Pool, plan: Plan, n: int) -> int:
    return int(lib.gdn_pool_apply(ctypes.byref(pool.c), ctypes.byref(plan.c), n))


def gdn_pool_abort(pool: Pool, plan: Plan, n: int) -> int:
    return int(lib.gdn_pool_abort(ctypes.byref(pool.c), ctypes.byref(plan.c), n))
