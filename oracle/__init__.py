"""CPU oracle for GatedDeltaNet speculative verification (FP64, plain and slow).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``.  The library never imports it,
and it imports nothing from the library.

Parts and the passages they follow:

* :func:`gdn_recurrent` / :func:`gdn_chunked` -- the gated delta rule
  (C, ``gdn_oracle.c``).  The per-head recurrence follows the state update
  named in "Native three-step MTP" (What changed: FP32 sigmoid gates, GDN
  state update shared by decode and verification); the chunked form follows
  "Run chained MTP drafting in the batch Engine" (Correctness fix).
* :func:`argmax_bf16` -- greedy target choice, lowest index on ties.
* :func:`greedy_accept` -- longest draft prefix that equals the target's
  greedy choice, then one bonus token ("Run chained MTP drafting",
  Quality follow-up: verification-row selection, per-request bonus).
* :func:`commit_plan` -- rollback: each request's slot becomes the
  checkpoint of its accepted row; a checkpoint that was not written in this
  transaction is refused (Correctness fix: a rejected request must not publish
  an uninitialised checkpoint).
* :class:`PoolModel`, :func:`plan_transaction` -- paged selection, draft
  deferral for transactions mixing prefill and draft rows, max-length clamp
  and copy-on-write of shared slots (Correctness fix; Summary; "H200 RC4
  evidence": mixed K, max-length clamping, cache reuse; "Native three-step
  MTP", Results: shared-prefix protection, duplicate-slot release, rejected
  requests, recovery after abort).

Readings where the pages are silent are listed with each function.
Parity pins for every function live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_SO = os.path.join(_HERE, "libgdnoracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (strict FP64: no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        L.oracle_gdn_recurrent.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                           P, P, P, P, P, ctypes.c_double, P, P, P]
        L.oracle_gdn_recurrent.restype = None
        L.oracle_gdn_chunked.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int,
                                         P, P, P, P, P, ctypes.c_double, P, P]
        L.oracle_gdn_chunked.restype = None
        L.oracle_gdn_chunk_wy.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          P, P, P, P, P, P, P, P]
        L.oracle_gdn_chunk_wy.restype = None
        L.oracle_argmax_bf16.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, P]
        L.oracle_argmax_bf16.restype = None
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    """Exact widening to a C-contiguous float64 array.  Accepts numpy arrays
    and torch tensors (bf16 and fp32 widen exactly to fp64)."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# ---------------------------------------------------------------------------
# Gated delta rule
# ---------------------------------------------------------------------------

@dataclass
class Unit:
    """One (request, v-head) recurrence: q,k [n,dk], v [n,dv], g,beta [n],
    S0 [dv,dk] (all float64)."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    S0: np.ndarray


def _pack(units: Sequence[Unit]):
    dk = units[0].S0.shape[1]
    dv = units[0].S0.shape[0]
    ns = [u.q.shape[0] for u in units]
    roff = np.zeros(len(units) + 1, dtype=np.int64)
    roff[1:] = np.cumsum(ns)
    R = int(roff[-1])
    cat = lambda xs, shp: (np.ascontiguousarray(np.concatenate(xs, axis=0), dtype=np.float64)
                           if R else np.zeros(shp, dtype=np.float64))
    q = cat([u.q.reshape(-1, dk) for u in units], (1, dk))
    k = cat([u.k.reshape(-1, dk) for u in units], (1, dk))
    v = cat([u.v.reshape(-1, dv) for u in units], (1, dv))
    g = cat([u.g.reshape(-1) for u in units], (1,))
    b = cat([u.beta.reshape(-1) for u in units], (1,))
    S = np.ascontiguousarray(np.stack([u.S0 for u in units]), dtype=np.float64)
    return dk, dv, roff, R, q, k, v, g, b, S


def recurrent_units(units: Sequence[Unit], q_scale: float = 1.0, want_ckpt: bool = False):
    """Run independent recurrences.  Returns (S_final [U,dv,dk], o list, ckpt list)."""
    if not units:
        return np.zeros((0,)), [], []
    dk, dv, roff, R, q, k, v, g, b, S = _pack(units)
    o = np.zeros((max(R, 1), dv), dtype=np.float64)
    ck = np.zeros((max(R, 1), dv, dk), dtype=np.float64) if want_ckpt else None
    lib().oracle_gdn_recurrent(dk, dv, len(units), _p(roff), _p(q), _p(k), _p(v), _p(g), _p(b),
                               float(q_scale), _p(S), _p(ck) if want_ckpt else None, _p(o))
    os_ = [o[roff[i]:roff[i + 1]] for i in range(len(units))]
    cks = [ck[roff[i]:roff[i + 1]] for i in range(len(units))] if want_ckpt else []
    return S, os_, cks


def chunked_units(units: Sequence[Unit], chunk: int, q_scale: float = 1.0):
    if not units:
        return np.zeros((0,)), []
    dk, dv, roff, R, q, k, v, g, b, S = _pack(units)
    o = np.zeros((max(R, 1), dv), dtype=np.float64)
    lib().oracle_gdn_chunked(dk, dv, len(units), _p(roff), int(chunk), _p(q), _p(k), _p(v), _p(g),
                             _p(b), float(q_scale), _p(S), _p(o))
    return S, [o[roff[i]:roff[i + 1]] for i in range(len(units))]


def chunk_wy(k, v, g, beta):
    """G, T, W, Ut of one chunk (for pins)."""
    k, v, g, beta = _f64(k), _f64(v), _f64(g), _f64(beta)
    n, dk = k.shape
    dv = v.shape[1]
    G = np.zeros(n)
    T = np.zeros((n, n))
    W = np.zeros((n, dk))
    Ut = np.zeros((n, dv))
    lib().oracle_gdn_chunk_wy(dk, dv, n, _p(k), _p(v), _p(g), _p(beta), _p(G), _p(T), _p(W), _p(Ut))
    return G, T, W, Ut


def head_units(q, k, v, g, beta, S0):
    """Split multi-head inputs into per-v-head units.

    q,k [n,h_qk,dk]; v [n,h_v,dv]; g,beta [n,h_v]; S0 [h_v,dv,dk].
    Reading: v-head h uses qk-head h // (h_v // h_qk) (consecutive grouping)."""
    q, k, v, g, beta, S0 = (_f64(x) for x in (q, k, v, g, beta, S0))
    h_qk, h_v = q.shape[1], v.shape[1]
    grp = h_v // h_qk
    return [Unit(q[:, h // grp], k[:, h // grp], v[:, h], g[:, h], beta[:, h], S0[h])
            for h in range(h_v)]


def gdn_recurrent(q, k, v, g, beta, S0, q_scale: float = 1.0, want_ckpt: bool = False):
    """Multi-head recurrence of one request.  Returns S [h_v,dv,dk],
    o [n,h_v,dv] (unrounded) and, if asked, ckpt [n,h_v,dv,dk]."""
    units = head_units(q, k, v, g, beta, S0)
    S, os_, cks = recurrent_units(units, q_scale, want_ckpt)
    o = np.stack(os_, axis=1)
    ck = np.stack(cks, axis=1) if want_ckpt else None
    return S, o, ck


def gdn_chunked(q, k, v, g, beta, S0, chunk: int, q_scale: float = 1.0):
    units = head_units(q, k, v, g, beta, S0)
    S, os_ = chunked_units(units, chunk, q_scale)
    return S, np.stack(os_, axis=1)


# ---------------------------------------------------------------------------
# Greedy choice and acceptance
# ---------------------------------------------------------------------------

def argmax_bf16(logits_bits: np.ndarray, vocab: Optional[int] = None) -> np.ndarray:
    """Greedy choice per row of bf16 logits given as uint16 bit patterns [rows, stride]."""
    x = np.ascontiguousarray(logits_bits, dtype=np.uint16)
    rows, stride = x.shape
    vocab = stride if vocab is None else vocab
    out = np.zeros(rows, dtype=np.int32)
    if rows:
        lib().oracle_argmax_bf16(rows, vocab, stride, _p(x), _p(out))
    return out


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a torch bf16 tensor."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


STATUS_ROWS_BAD = 2
STATUS_TOKEN_OOR = 4


@dataclass
class AcceptResult:
    accept_len: np.ndarray
    bonus: np.ndarray
    out_tokens: np.ndarray
    stats: dict
    status: int


def greedy_accept(argmax: np.ndarray, tokens: np.ndarray, cu_rows: np.ndarray, vocab: int) -> AcceptResult:
    """Acceptance per request.  Rows of request r are cu_rows[r]..cu_rows[r+1]-1;
    row 0 holds the last committed token, rows 1..K the drafts.

    j = number of leading drafts i (1..K) with tokens[t0+i] == argmax[t0+i-1];
    bonus = argmax[t0+j]; emitted tokens are argmax[t0..t0+j] (the accepted
    drafts equal them), other rows of the request get -1.
    Counters: proposed += K, evaluated += min(j+1, K), accepted += j,
    emitted += j+1; steps += 1 per call.
    Readings: a request with no rows is refused (accept_len = bonus = -1,
    status bit ROWS_BAD); a draft id outside [0, vocab) never matches and sets
    the status bit TOKEN_OOR.
    """
    B = len(cu_rows) - 1
    acc = np.full(B, -1, dtype=np.int32)
    bonus = np.full(B, -1, dtype=np.int32)
    out = np.full(int(cu_rows[-1]) if B >= 0 else 0, -1, dtype=np.int32)
    st = dict(proposed=0, evaluated=0, accepted=0, emitted=0, steps=1)
    status = 0
    for r in range(B):
        t0, t1 = int(cu_rows[r]), int(cu_rows[r + 1])
        n = t1 - t0
        if n < 1:
            status |= STATUS_ROWS_BAD
            continue
        K = n - 1
        for i in range(1, K + 1):
            if not (0 <= int(tokens[t0 + i]) < vocab):
                status |= STATUS_TOKEN_OOR
        j = 0
        while j < K and int(tokens[t0 + j + 1]) == int(argmax[t0 + j]):
            j += 1
        acc[r] = j
        bonus[r] = argmax[t0 + j]
        out[t0:t0 + j + 1] = argmax[t0:t0 + j + 1]
        st["proposed"] += K
        st["evaluated"] += min(j + 1, K)
        st["accepted"] += j
        st["emitted"] += j + 1
    return AcceptResult(acc, bonus, out, st, status)


# ---------------------------------------------------------------------------
# Commit (rollback to the accepted checkpoint)
# ---------------------------------------------------------------------------

STATUS_SLOT_OOR = 1
STATUS_CKPT_UNWRITTEN = 8
STATUS_ACCEPT_BAD = 16


def commit_plan(accept_len, cu_rows, ckpt_rows, ckpt_txn, txn, dst_slot, num_slots):
    """Which checkpoint row is copied to which slot, per (layer, request).

    ckpt_rows[l][r] / ckpt_txn[l][r]: rows written for request r by layer l's
    verify and the transaction that wrote them.  Returns (moves, status) with
    moves[l][r] = packed checkpoint row, or None when the commit is refused:
    checkpoint not written in transaction ``txn`` or accept_len outside
    [0, rows) -> CKPT_UNWRITTEN / ACCEPT_BAD; slot out of range -> SLOT_OOR.
    """
    L = len(ckpt_rows)
    B = len(accept_len)
    status = 0
    moves = [[None] * B for _ in range(L)]
    for l in range(L):
        for r in range(B):
            j = int(accept_len[r])
            if int(ckpt_txn[l][r]) != int(txn) or int(ckpt_rows[l][r]) <= 0:
                status |= STATUS_CKPT_UNWRITTEN
                continue
            if j < 0 or j >= int(ckpt_rows[l][r]):
                status |= STATUS_ACCEPT_BAD
                continue
            if not (0 <= int(dst_slot[r]) < num_slots):
                status |= STATUS_SLOT_OOR
                continue
            moves[l][r] = int(cu_rows[r]) + j
    return moves, status


# ---------------------------------------------------------------------------
# Slot pool and transaction planner (host model)
# ---------------------------------------------------------------------------

OK, ERR_ARG, ERR_DUP_SLOT, ERR_NO_SLOT = 0, -3, -4, -5
DECODE, PREFILL = 0, 1
PLAN_RECURRENT, PLAN_CHUNKED = 0, 1


class PoolModel:
    """Reference-counted state slots with a FIFO free list.

    Readings: the free list is FIFO in the given order; a slot goes back to
    the tail of the list when its count reaches zero; releasing a free slot is
    an error (duplicate release) and changes nothing."""

    def __init__(self, num_slots: int, free_order: Optional[Sequence[int]] = None):
        self.n = num_slots
        self.ref = [0] * num_slots
        self.free = list(range(num_slots) if free_order is None else free_order)

    def alloc(self):
        if not self.free:
            return ERR_NO_SLOT, -1
        s = self.free.pop(0)
        self.ref[s] = 1
        return OK, s

    def share(self, s):
        if not (0 <= s < self.n) or self.ref[s] <= 0:
            return ERR_ARG
        self.ref[s] += 1
        return OK

    def release(self, s):
        if not (0 <= s < self.n) or self.ref[s] <= 0:
            return ERR_ARG
        self.ref[s] -= 1
        if self.ref[s] == 0:
            self.free.append(s)
        return OK


@dataclass
class Req:
    kind: int
    k_draft: int = 0
    n_tokens: int = 0
    cur_len: int = 0
    max_len: int = 1 << 30
    slot: int = -1


@dataclass
class Plan:
    status: int = OK
    n_selected: int = 0
    plan: int = PLAN_RECURRENT
    deferred: int = 0
    k: List[int] = field(default_factory=list)      # per request, -1 if not selected
    rows: List[int] = field(default_factory=list)
    src: List[int] = field(default_factory=list)
    dst: List[int] = field(default_factory=list)
    dec_req: List[int] = field(default_factory=list)
    dec_cu: List[int] = field(default_factory=lambda: [0])
    dec_src: List[int] = field(default_factory=list)
    dec_dst: List[int] = field(default_factory=list)
    pre_req: List[int] = field(default_factory=list)
    pre_cu: List[int] = field(default_factory=lambda: [0])
    pre_src: List[int] = field(default_factory=list)
    pre_dst: List[int] = field(default_factory=list)


def _unreserve(pool: PoolModel, reserved: List[int]) -> None:
    """Undo fresh-slot reservations: the slots return to the head of the free
    list in their original order, so a failed plan leaves the pool as it was."""
    for s in reversed(reserved):
        pool.ref[s] = 0
        pool.free.insert(0, s)


def plan_transaction(reqs: Sequence[Req], max_rows: int, max_reqs: int, k_max: int,
                     pool: PoolModel) -> Plan:
    """Select, defer, clamp and assign slots for one transaction.

    1. Paged selection: take requests in order while rows remain in the
       budget ``max_rows`` and fewer than ``max_reqs`` are taken.  A decode
       request takes 1 + K rows with K = min(k_draft, k_max,
       max_len - cur_len - 1, budget - 1) (at least 0); a prefill takes
       min(n_tokens, max_len - cur_len, budget) rows.  Selection stops at the
       first request that gets no row.
    2. Deferral: if the selected set holds a prefill and a decode with K > 0,
       every selected decode gets K = 0 (one row); ``deferred`` counts the
       drafts cleared.  No reselection follows.
    3. Plan kind: CHUNKED when a prefill is selected, else RECURRENT.
    4. Slots: a decode or continuing prefill reads its slot and writes it in
       place when its count is 1, else a fresh slot (copy-on-write); a new
       prefill (slot -1) starts from zero and writes a fresh slot.  Fresh
       slots come from the free list; if it runs dry, every slot reserved by
       this call is returned and ERR_NO_SLOT is reported.
    Errors (fail closed, pool unchanged): a decode at or past max_len, a
    prefill with no tokens, k_draft < 0, a slot out of range or not held
    -> ERR_ARG; duplicate destination slots -> ERR_DUP_SLOT.
    """
    n = len(reqs)
    P = Plan(k=[-1] * n, rows=[0] * n, src=[-1] * n, dst=[-1] * n)
    budget = max_rows
    sel = []
    for i, r in enumerate(reqs):
        if len(sel) >= max_reqs or budget < 1:
            break
        if r.slot != -1 and not (0 <= r.slot < pool.n and pool.ref[r.slot] > 0):
            P.status = ERR_ARG
            return P
        if r.kind == DECODE:
            if r.cur_len >= r.max_len or r.k_draft < 0 or r.slot < 0:
                P.status = ERR_ARG
                return P
            K = max(0, min(r.k_draft, k_max, r.max_len - r.cur_len - 1, budget - 1))
            P.k[i] = K
            P.rows[i] = K + 1
        elif r.kind == PREFILL:
            if r.n_tokens <= 0 or r.cur_len >= r.max_len:
                P.status = ERR_ARG
                return P
            rows = min(r.n_tokens, r.max_len - r.cur_len, budget)
            P.k[i] = 0
            P.rows[i] = rows
        else:
            P.status = ERR_ARG
            return P
        budget -= P.rows[i]
        sel.append(i)
    P.n_selected = len(sel)
    has_pre = any(reqs[i].kind == PREFILL for i in sel)
    has_draft = any(reqs[i].kind == DECODE and P.k[i] > 0 for i in sel)
    if has_pre and has_draft:
        for i in sel:
            if reqs[i].kind == DECODE:
                P.deferred += P.k[i]
                P.k[i] = 0
                P.rows[i] = 1
    P.plan = PLAN_CHUNKED if has_pre else PLAN_RECURRENT
    reserved = []
    for i in sel:
        r = reqs[i]
        P.src[i] = r.slot
        if r.slot >= 0 and pool.ref[r.slot] == 1:
            P.dst[i] = r.slot
        else:
            st, s = pool.alloc()
            if st != OK:
                _unreserve(pool, reserved)
                P.status = ERR_NO_SLOT
                return P
            reserved.append(s)
            P.dst[i] = s
    dsts = [P.dst[i] for i in sel]
    if len(set(dsts)) != len(dsts):
        _unreserve(pool, reserved)
        P.status = ERR_DUP_SLOT
        return P
    for i in sel:
        if reqs[i].kind == DECODE:
            P.dec_req.append(i)
            P.dec_cu.append(P.dec_cu[-1] + P.rows[i])
            P.dec_src.append(P.src[i])
            P.dec_dst.append(P.dst[i])
        else:
            P.pre_req.append(i)
            P.pre_cu.append(P.pre_cu[-1] + P.rows[i])
            P.pre_src.append(P.src[i])
            P.pre_dst.append(P.dst[i])
    return P


def pool_apply(pool: PoolModel, reqs: Sequence[Req], P: Plan) -> int:
    """After a successful commit: every request that moved releases its old slot."""
    for i in range(len(reqs)):
        if P.k[i] >= 0 and P.src[i] >= 0 and P.dst[i] != P.src[i]:
            st = pool.release(P.src[i])
            if st != OK:
                return st
    return OK


def pool_abort(pool: PoolModel, reqs: Sequence[Req], P: Plan) -> int:
    """Abort: every fresh slot reserved by the plan goes back to the free list."""
    for i in range(len(reqs)):
        if P.k[i] >= 0 and P.dst[i] != P.src[i]:
            st = pool.release(P.dst[i])
            if st != OK:
                return st
    return OK
