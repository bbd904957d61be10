"""Per-transaction call sequence of K-draft verification, over the C ABI.

``VerifyStep`` owns the device buffers of one verification loop (state pool,
per-row checkpoints and their tags, outputs, accept workspace, telemetry,
status word) and issues, on one stream:

    gdn_verify            x num_layers   (rows -> checkpoints, o)
    mtp_greedy_accept     x 1            (argmax, accept length, bonus, tokens)
    gdn_commit            x 1            (every layer's slot <- accepted checkpoint)

Layer inputs (q, k, v, g, beta of the packed rows) and the logits are the
caller's device tensors.  All arithmetic happens in the library's kernels.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import binding as gs


@dataclass
class LayerRows:
    q: torch.Tensor      # bf16 [R, h_qk, d_k]
    k: torch.Tensor      # bf16 [R, h_qk, d_k]
    v: torch.Tensor      # bf16 [R, h_v, d_v]
    g: torch.Tensor      # fp32 [R, h_v]
    beta: torch.Tensor   # fp32 [R, h_v]


class VerifyStep:
    def __init__(self, dims: gs.gdn_dims, num_layers: int, num_slots: int, row_capacity: int, max_batch: int,
                 vocab: int, device="cuda", pool: Optional[torch.Tensor] = None, checkpoints: bool = True):
        self.d = dims
        self.L = num_layers
        self.num_slots = num_slots
        self.cap = row_capacity
        self.max_batch = max_batch
        self.vocab = vocab
        dev = torch.device(device)
        self.dev = dev
        h_v, dv, dk = dims.h_v, dims.d_v, dims.d_k
        if pool is None:
            pool = torch.zeros((num_slots, num_layers, h_v, dv, dk), dtype=torch.float32, device=dev)
        assert pool.shape == (num_slots, num_layers, h_v, dv, dk) and pool.is_contiguous()
        self.pool = pool
        self.ckpt = (torch.empty((num_layers, row_capacity, h_v, dv, dk), dtype=torch.float32, device=dev)
                     if checkpoints else None)
        self._tags = torch.zeros((num_layers * max_batch,), dtype=torch.int64, device=dev)
        self.o = torch.empty((num_layers, row_capacity, h_v, dv), dtype=torch.bfloat16, device=dev)
        self.argmax = torch.full((row_capacity,), -1, dtype=torch.int32, device=dev)
        self.accept_len = torch.full((max_batch,), -1, dtype=torch.int32, device=dev)
        self.bonus = torch.full((max_batch,), -1, dtype=torch.int32, device=dev)
        self.out_tokens = torch.full((row_capacity,), -1, dtype=torch.int32, device=dev)
        self.ws_bytes = gs.mtp_accept_workspace_bytes(row_capacity, vocab)
        self.workspace = torch.empty((max(self.ws_bytes, 8),), dtype=torch.uint8, device=dev)
        self.stats = torch.zeros((5,), dtype=torch.int64, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.slot_stride = pool.stride(0)
        self.layer_stride = pool.stride(1)
        self.ckpt_layer_stride = self.ckpt.stride(0) if checkpoints else 0
        self.txn = 0
        self._rows_cache = {}

    def rows_array(self, layer_rows: Sequence[LayerRows]):
        """The host gdn_layer_rows array of a list of per-layer inputs, built
        once per list (the list is kept alive with its array)."""
        hit = self._rows_cache.get(id(layer_rows))
        if hit is None or hit[0] is not layer_rows:
            if len(self._rows_cache) > 64:
                self._rows_cache.clear()
            hit = (layer_rows, gs.layer_rows_array(layer_rows))
            self._rows_cache[id(layer_rows)] = hit
        return hit[1]

    def verify_all(self, B: int, cu_rows: torch.Tensor, src_slot: torch.Tensor, layer_rows: Sequence[LayerRows],
                   stream=None):
        """Every layer's gdn_verify, issued by one library call."""
        assert len(layer_rows) == self.L
        gs.gdn_verify_layers(self.d, self.L, B, self.cap, cu_rows, self.rows_array(layer_rows), self.pool,
                             self.slot_stride, self.layer_stride, self.num_slots, src_slot, self.ckpt,
                             self.ckpt_layer_stride, self.tags(B), self.txn, self.o, self.o.stride(0), self.status,
                             stream)

    def tags(self, B: int) -> torch.Tensor:
        """Checkpoint tags laid out [layer][request] for a batch of B requests."""
        return self._tags[:self.L * B].view(self.L, B)

    def pool_layer(self, l: int) -> int:
        return self.pool.data_ptr() + 4 * l * self.layer_stride

    def verify_layer(self, l: int, B: int, cu_rows: torch.Tensor, src_slot: torch.Tensor, rows: LayerRows,
                     stream=None):
        gs.gdn_verify(self.d, B, self.cap, cu_rows, rows.q, rows.k, rows.v, rows.g, rows.beta, self.pool_layer(l),
                      self.slot_stride, self.num_slots, src_slot, self.ckpt[l], self.tags(B)[l], self.txn, self.o[l],
                      self.status, stream)

    def accept(self, B: int, cu_rows: torch.Tensor, logits: torch.Tensor, tokens: torch.Tensor, stream=None):
        gs.mtp_greedy_accept(B, self.cap, cu_rows, logits, self.vocab, logits.stride(0), tokens, self.argmax,
                             self.accept_len, self.bonus, self.out_tokens, self.stats, self.workspace,
                             self.ws_bytes, self.status, stream)

    def commit(self, B: int, cu_rows: torch.Tensor, dst_slot: torch.Tensor, stream=None):
        gs.gdn_commit(self.d, B, self.L, self.cap, cu_rows, self.accept_len, self.ckpt, self.ckpt_layer_stride,
                      self.tags(B), self.txn, self.pool, self.slot_stride, self.layer_stride, self.num_slots,
                      dst_slot, self.status, stream)

    def run(self, B: int, cu_rows: torch.Tensor, src_slot: torch.Tensor, dst_slot: torch.Tensor,
            layer_rows: Sequence[LayerRows], logits: torch.Tensor, tokens: torch.Tensor, stream=None):
        """One transaction: verify every layer, accept, commit.  Asynchronous."""
        self.txn = (self.txn + 1) & 0xFFFFFFFF
        self.verify_all(B, cu_rows, src_slot, layer_rows, stream)
        self.accept(B, cu_rows, logits, tokens, stream)
        self.commit(B, cu_rows, dst_slot, stream)


class TraceWriter:
    """Per-(layer, row) trace of decode transactions, for localising a parity
    failure ("Run chained MTP drafting in the batch Engine", Validation: layer
    tracing of every row).  Enabled by the environment: GDNSPEC_TRACE_DIR names
    a directory; GDNSPEC_TRACE_REQS (default 2) how many leading requests get
    their per-row checkpoints saved.  After each transaction's readback one
    ``txn_<n>.npz`` holds the row tables, the accept lengths, bonus and emitted
    tokens, every layer's outputs for every row (bf16 bits) and, for the
    traced requests, every layer's checkpoint after each of their rows."""

    def __init__(self, directory: str, n_reqs: int = 2):
        self.dir = directory
        self.n_reqs = n_reqs
        self.count = 0
        os.makedirs(directory, exist_ok=True)

    @staticmethod
    def from_env() -> "Optional[TraceWriter]":
        d = os.environ.get("GDNSPEC_TRACE_DIR")
        if not d:
            return None
        return TraceWriter(d, int(os.environ.get("GDNSPEC_TRACE_REQS", "2")))

    def write(self, vs: "VerifyStep", cu_rows: Sequence[int], src: Sequence[int], dst: Sequence[int], accept_len,
              bonus, out_tokens):
        B = len(cu_rows) - 1
        R = int(cu_rows[-1])
        rec = {"txn": np.int64(vs.txn), "cu_rows": np.asarray(cu_rows, np.int32), "src_slot": np.asarray(src, np.int32),
               "dst_slot": np.asarray(dst, np.int32), "accept_len": np.asarray(accept_len[:B], np.int32),
               "bonus": np.asarray(bonus[:B], np.int32), "out_tokens": np.asarray(out_tokens[:R], np.int32),
               "o_bf16": vs.o[:, :R].detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)}
        ck = getattr(vs, "ckpt", None)
        if ck is not None:
            for r in range(min(self.n_reqs, B)):
                a, b = int(cu_rows[r]), int(cu_rows[r + 1])
                rec["ckpt_req%d" % r] = ck[:, a:b].detach().cpu().numpy()
        np.savez_compressed(os.path.join(self.dir, "txn_%06d.npz" % self.count), **rec)
        self.count += 1


class DecodeLoop:
    """Decode-only transactions for a fixed set of requests.

    Per step: the host planner (``plan_transaction``) grants drafts, packs the
    rows and picks destination slots (copy-on-write for shared slots); the
    tables go to the device; ``VerifyStep.run`` verifies, accepts and commits;
    one device-to-host read brings back accept lengths, bonus and emitted
    tokens; the pool then releases the slots that requests moved away from.
    Host bookkeeping works on numpy views of the planner's buffers.
    """

    def __init__(self, vs: VerifyStep, slots: Sequence[int], pool: "gs.Pool", k_max: int = 3,
                 max_len: int = 1 << 30, cur_len: int = 1):
        self.vs = vs
        self.B = len(slots)
        B = self.B
        self.pool = pool
        self.plan = gs.Plan(B)
        self.lim = gs.gdn_plan_limits(vs.cap, B, k_max)
        self.reqs = (gs.gdn_req * max(B, 1))()
        self.req_np = np.ctypeslib.as_array(ctypes.cast(self.reqs, ctypes.POINTER(ctypes.c_int32)),
                                            shape=(max(B, 1), 6))
        self.req_np[:B, 0] = gs.REQ_DECODE
        self.req_np[:B, 2] = 0
        self.req_np[:B, 3] = cur_len
        self.req_np[:B, 4] = max_len
        self.req_np[:B, 5] = np.asarray(slots, dtype=np.int32)
        dev = vs.dev
        self.h_tab = torch.zeros((3, B + 1), dtype=torch.int32).pin_memory()
        self.h_tab_np = self.h_tab.numpy()
        self.d_tab = torch.zeros((3, B + 1), dtype=torch.int32, device=dev)
        self.h_out = torch.zeros((2 * B + vs.cap,), dtype=torch.int32).pin_memory()
        self._io = None
        self._arena_io = None
        self._txn = ctypes.c_uint32(vs.txn)
        self.trace = TraceWriter.from_env()

    @property
    def slot(self):
        return self.req_np[:self.B, 5].tolist()

    @property
    def cur_len(self):
        return self.req_np[:self.B, 3].tolist()

    def plan_step(self, k_draft: Sequence[int]):
        B = self.B
        self.req_np[:B, 1] = np.asarray(k_draft, dtype=np.int32)
        st = gs.plan_transaction(self.reqs, B, self.lim, self.pool, self.plan)
        if st != gs.GDN_OK:
            raise gs.GdnError("plan_transaction", st)
        p = self.plan
        if p.c.n_decode != B:
            raise RuntimeError("row budget too small for the batch: %d of %d requests selected" % (p.c.n_decode, B))
        arr = p.arrays
        self.h_tab_np[0, :B + 1] = arr["dec_cu"][:B + 1]
        self.h_tab_np[1, :B] = arr["dec_src"][:B]
        self.h_tab_np[2, :B] = arr["dec_dst"][:B]
        return p

    def upload_tables(self, stream=None):
        self.d_tab.copy_(self.h_tab, non_blocking=True)

    @property
    def cu_rows(self):
        return self.d_tab[0]

    @property
    def src_slot(self):
        return self.d_tab[1, :self.B]

    @property
    def dst_slot(self):
        return self.d_tab[2, :self.B]

    def run(self, layer_rows, logits, tokens, stream=None):
        self.vs.run(self.B, self.cu_rows, self.src_slot, self.dst_slot, layer_rows, logits, tokens, stream)

    def readback(self):
        """The step's one device-to-host read: accept_len, bonus, emitted tokens."""
        B, cap = self.B, self.vs.cap
        self.h_out[:B].copy_(self.vs.accept_len[:B], non_blocking=True)
        self.h_out[B:2 * B].copy_(self.vs.bonus[:B], non_blocking=True)
        self.h_out[2 * B:].copy_(self.vs.out_tokens, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if self.trace is not None:
            t = self.h_tab_np
            self.trace.write(self.vs, t[0, :B + 1].tolist(), t[1, :B].tolist(), t[2, :B].tolist(),
                             self.h_out[:B].numpy(), self.h_out[B:2 * B].numpy(), self.h_out[2 * B:].numpy())
        return self.h_out[:B], self.h_out[B:2 * B], self.h_out[2 * B:]

    def transaction(self, layer_rows: Sequence[LayerRows], logits: torch.Tensor, tokens: torch.Tensor,
                    kernel_ms=None, stream=None):
        """One whole decode transaction by the library's host driver
        (``gdn_decode_transaction``, or ``gdn_decode_transaction_at`` over an
        ``ArenaStep``'s state arena): plan, tables, every layer's verify,
        accept, commit, the one readback and the request bookkeeping in one
        call.  Returns the accepted draft counts of the decoded requests (a
        numpy view, valid until the next transaction).  ``kernel_ms``: None or
        a ctypes float array of 3 (verify, accept, commit device times)."""
        vs, B = self.vs, self.B
        if isinstance(vs, ReplayStep):
            raise TypeError("fixed-state replay has no one-call driver: use ReplayStep.run or ReplayGraphs")
        io = self._io
        if io is None:
            io = self._io = gs.gdn_decode_io()
            io.tables = self.d_tab.data_ptr()
            io.pool = vs.pool.data_ptr()
            io.slot_stride, io.layer_stride, io.num_slots = vs.slot_stride, vs.layer_stride, vs.num_slots
            ck = getattr(vs, "ckpt", None)
            io.ckpt, io.ckpt_layer_stride = (ck.data_ptr() if ck is not None else None), vs.ckpt_layer_stride
            io.ckpt_tag = vs._tags.data_ptr()
            io.o, io.o_layer_stride = vs.o.data_ptr(), vs.o.stride(0)
            io.vocab = vs.vocab
            io.argmax, io.accept_len = vs.argmax.data_ptr(), vs.accept_len.data_ptr()
            io.bonus, io.out_tokens = vs.bonus.data_ptr(), vs.out_tokens.data_ptr()
            io.stats = vs.stats.data_ptr()
            io.workspace, io.workspace_bytes = vs.workspace.data_ptr(), vs.ws_bytes
            io.dev_status = vs.status.data_ptr()
            io.host_tables, io.host_out = self.h_tab.data_ptr(), self.h_out.data_ptr()
        self._txn.value = vs.txn
        io.rows = ctypes.cast(vs.rows_array(layer_rows), ctypes.c_void_p).value
        io.logits, io.logit_row_stride = logits.data_ptr(), logits.stride(0)
        io.tokens = tokens.data_ptr()
        if isinstance(vs, ArenaStep):
            ar = self._arena_io
            if ar is None:
                ar = self._arena_io = gs.gdn_arena_io()
                ar.arena, ar.elems_total, ar.loc = vs.arena.data_ptr(), vs.total, vs.loc.data_ptr()
                ar.area_off[0], ar.area_off[1] = vs.area_off
            gs.gdn_decode_transaction_at(vs.d, vs.L, vs.cap, self.reqs, B, self.lim, self.pool, self.plan,
                                         self._txn, io, ar, kernel_ms, stream)
        else:
            gs.gdn_decode_transaction(vs.d, vs.L, vs.cap, self.reqs, B, self.lim, self.pool, self.plan, self._txn,
                                      io, kernel_ms, stream)
        vs.txn = self._txn.value
        n = self.plan.c.n_decode
        if self.trace is not None and not isinstance(vs, ArenaStep):
            t = self.h_tab_np      # the driver wrote the step's tables here
            self.trace.write(vs, t[0, :n + 1].tolist(), t[1, :n].tolist(), t[2, :n].tolist(), self.h_out[:n].numpy(),
                             self.h_out[B:B + n].numpy(), self.h_out[2 * B:].numpy())
        return self.h_out.numpy()[:n]

    def finish(self, accept_len):
        st = gs.gdn_pool_apply(self.pool, self.plan, self.B)
        if st != gs.GDN_OK:
            raise gs.GdnError("gdn_pool_apply", st)
        B = self.B
        self.req_np[:B, 5] = self.plan.arrays["dst"][:B]
        acc = accept_len.numpy() if hasattr(accept_len, "numpy") else np.asarray(accept_len)
        self.req_np[:B, 3] += acc[:B].astype(np.int32) + 1


class ArenaStep(VerifyStep):
    """Zero-copy commit over a state arena.

    One fp32 buffer holds the pool slots followed by two checkpoint areas;
    transaction n writes its checkpoints into area n % 2 and the commit only
    points each (request, layer) location at its accepted checkpoint, so the
    next transaction verifies from there.  ``materialize`` copies states
    back into slots when a request leaves.  The batch size is fixed (the
    location table is laid out [layer][request])."""

    def __init__(self, dims: gs.gdn_dims, num_layers: int, num_slots: int, row_capacity: int, batch: int,
                 vocab: int, device="cuda"):
        h_v, dv, dk = dims.h_v, dims.d_v, dims.d_k
        S = h_v * dv * dk
        self.S = S
        pool_elems = num_slots * num_layers * S
        ck_elems = num_layers * row_capacity * S
        self.arena = torch.empty((pool_elems + 2 * ck_elems,), dtype=torch.float32, device=device)
        pool = self.arena[:pool_elems].view(num_slots, num_layers, h_v, dv, dk)
        super().__init__(dims, num_layers, num_slots, row_capacity, batch, vocab, device, pool=pool,
                         checkpoints=False)  # the checkpoint areas live in the arena
        self.areas = [self.arena[pool_elems + i * ck_elems:pool_elems + (i + 1) * ck_elems]
                      .view(num_layers, row_capacity, h_v, dv, dk) for i in range(2)]
        self.area_off = [pool_elems, pool_elems + ck_elems]
        self.ckpt_layer_stride = row_capacity * S
        self.total = self.arena.numel()
        self.B = batch
        self.loc = torch.zeros((num_layers, batch), dtype=torch.int64, device=self.dev)

    def point_at_slots(self, slots: Sequence[int]):
        """Every request's state starts in its pool slot."""
        L = self.L
        off = [[s * self.slot_stride + l * self.layer_stride for s in slots] for l in range(L)]
        self.loc.copy_(torch.tensor(off, dtype=torch.int64))

    def run(self, B: int, cu_rows: torch.Tensor, layer_rows: Sequence[LayerRows], logits: torch.Tensor,
            tokens: torch.Tensor, stream=None):
        assert B == self.B
        self.txn = (self.txn + 1) & 0xFFFFFFFF
        self.verify_all_at(B, cu_rows, layer_rows, stream)
        self.accept(B, cu_rows, logits, tokens, stream)
        area = self.txn & 1
        gs.gdn_commit_at(self.d, B, self.L, self.cap, cu_rows, self.accept_len, self.area_off[area],
                         self.ckpt_layer_stride, self.tags(B), self.txn, self.loc, self.status, stream)

    def verify_all_at(self, B: int, cu_rows: torch.Tensor, layer_rows: Sequence[LayerRows], stream=None):
        """Every layer's gdn_verify_at for transaction self.txn (checkpoints
        into area txn % 2), issued by one library call."""
        assert B == self.B and len(layer_rows) == self.L
        gs.gdn_verify_at_layers(self.d, self.L, B, self.cap, cu_rows, self.rows_array(layer_rows), self.arena,
                                self.total, self.loc, self.areas[self.txn & 1], self.ckpt_layer_stride,
                                self.tags(B), self.txn, self.o, self.o.stride(0), self.status, stream)

    def materialize(self, dst_slot: torch.Tensor, stream=None):
        gs.gdn_materialize(self.d, self.B, self.L, self.arena, self.total, self.loc, self.pool, self.slot_stride,
                           self.layer_stride, self.num_slots, dst_slot, self.status, stream)


class ReplayStep(VerifyStep):
    """Compact fixed-state replay: no checkpoints.  Each transaction's
    ``gdn_verify_replay`` first runs the previous transaction's accepted rows
    from the slot and writes the slot (the previous commit), then runs the new
    rows for outputs only.  The caller keeps the previous transaction's layer
    rows alive until the next run (or ``flush``)."""

    def __init__(self, dims: gs.gdn_dims, num_layers: int, num_slots: int, row_capacity: int, batch: int,
                 vocab: int, device="cuda", pool: Optional[torch.Tensor] = None):
        super().__init__(dims, num_layers, num_slots, row_capacity, batch, vocab, device, pool=pool,
                         checkpoints=False)
        self.B = batch
        self.acc_bufs = [torch.full((batch,), -1, dtype=torch.int32, device=self.dev) for _ in range(2)]
        self.prev_cu = torch.zeros((batch + 1,), dtype=torch.int32, device=self.dev)
        self.no_rows = torch.zeros((batch + 1,), dtype=torch.int32, device=self.dev)
        self.prev_rows: Optional[Sequence[LayerRows]] = None
        self.prev_acc = self.acc_bufs[1]      # read by the replay: the previous accept lengths
        self.accept_len = self.acc_bufs[0]    # written by this transaction's accept
        self.pending = False

    def _advance(self):
        if self.pending:  # the accept lengths just read back become the ones to replay
            self.prev_acc, self.accept_len = self.accept_len, self.prev_acc

    def _verify_all(self, B, cu_rows, src_slot, dst_slot, layer_rows, stream=None):
        prev = self.prev_rows if self.prev_rows is not None else layer_rows
        assert len(layer_rows) == self.L and len(prev) == self.L
        gs.gdn_verify_replay_layers(self.d, self.L, B, self.cap, cu_rows, self.rows_array(layer_rows), self.cap,
                                    self.prev_cu, self.prev_acc, self.rows_array(prev), self.pool, self.slot_stride,
                                    self.layer_stride, self.num_slots, src_slot, dst_slot, self.o, self.o.stride(0),
                                    self.status, stream)

    def run(self, B: int, cu_rows: torch.Tensor, src_slot: torch.Tensor, dst_slot: torch.Tensor,
            layer_rows: Sequence[LayerRows], logits: torch.Tensor, tokens: torch.Tensor, stream=None):
        assert B == self.B
        self._advance()
        self._verify_all(B, cu_rows, src_slot, dst_slot, layer_rows, stream)
        self.accept(B, cu_rows, logits, tokens, stream)
        # this transaction's accepted rows are replayed by the next one
        self.prev_cu.copy_(cu_rows[:B + 1], non_blocking=True)
        self.prev_rows = layer_rows
        self.pending = True

    def flush(self, src_slot: torch.Tensor, dst_slot: torch.Tensor, stream=None):
        """Commit the pending accepted rows without verifying new ones."""
        if not self.pending:
            return
        self._advance()
        self._verify_all(self.B, self.no_rows, src_slot, dst_slot, self.prev_rows, stream)
        self.prev_acc.fill_(-1)
        self.pending = False


class ReplayGraphs:
    """CUDA-graph capture of replay transactions (one graph per input set).

    A replay transaction has no per-step scalar arguments: everything it
    reads lives in fixed device buffers (the loop's row/slot tables, the
    tokens, the two accept-length buffers that alternate by transaction
    parity).  With the input sets cycled in order, transaction s is fixed by
    s modulo n = lcm(number of sets, 2) -- its input set, the previous
    transaction's set and the accept-buffer parity -- and so is its whole
    launch sequence (every layer's gdn_verify_replay, the greedy accept and
    the copy of the row table for the next replay): each residue gets one
    graph, replayed with a single launch.  The caller uploads the tables and
    tokens before ``launch`` and reads back after."""

    def __init__(self, rs: ReplayStep, loop: "DecodeLoop", ring_rows: Sequence[Sequence[LayerRows]],
                 ring_logits: Sequence[torch.Tensor], tokens: torch.Tensor):
        self.rs, self.loop = rs, loop
        self.sets = len(ring_rows)
        self.n = self.sets if self.sets % 2 == 0 else 2 * self.sets
        self.graphs = []
        B = loop.B
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        saved = (rs.prev_acc, rs.accept_len, rs.prev_rows, rs.pending)
        try:
            for i in range(self.n):
                rs.prev_acc, rs.accept_len = rs.acc_bufs[(i + 1) % 2], rs.acc_bufs[i % 2]
                rs.prev_rows = ring_rows[(i - 1) % self.sets]
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    rs._verify_all(B, loop.cu_rows, loop.src_slot, loop.dst_slot, ring_rows[i % self.sets])
                    rs.accept(B, loop.cu_rows, ring_logits[i % self.sets], tokens)
                    rs.prev_cu.copy_(loop.cu_rows[:B + 1], non_blocking=True)
                self.graphs.append(g)
        finally:
            rs.prev_acc, rs.accept_len, rs.prev_rows, rs.pending = saved
        torch.cuda.current_stream().wait_stream(stream)

    def launch(self, step_no: int, ring_rows: Sequence[Sequence[LayerRows]]):
        """Transaction number ``step_no`` (its input set is step_no modulo the number of sets)."""
        i = step_no % self.n
        rs = self.rs
        rs.prev_acc, rs.accept_len = rs.acc_bufs[(i + 1) % 2], rs.acc_bufs[i % 2]
        self.graphs[i].replay()
        rs.prev_rows = ring_rows[i % self.sets]
        rs.pending = True


class StepGraphs:
    """CUDA-graph capture of checkpointing transactions: every layer's verify,
    the greedy accept and the commit, replayed with one launch per step
    ("Run chained MTP drafting in the batch Engine", H200 RC4 evidence:
    graph capture of the hybrid fixed-state step).

    A transaction's launches read fixed device buffers (the loop's row and
    slot tables, the tokens, the checkpoints, tags and locations) plus two
    arguments passed by value: the input set and the transaction id.  A graph
    fixes both, so the id cannot advance from one replay to the next; each
    graph therefore starts by clearing the checkpoint tags, which keeps the
    commit's guard meaningful (a layer whose verify did not write its tag
    leaves 0, which no id matches).  The copying commit needs one graph per
    input set; the zero-copy commit also needs the id's parity (it selects
    the checkpoint area the locations do not point into), so it takes one
    graph per residue of lcm(sets, 2) with the id alternating between two
    values.  The caller plans and uploads the tables and tokens before
    ``launch`` and reads back after."""

    def __init__(self, vs: VerifyStep, loop: "DecodeLoop", ring_rows: Sequence[Sequence[LayerRows]],
                 ring_logits: Sequence[torch.Tensor], tokens: torch.Tensor):
        arena = isinstance(vs, ArenaStep)
        if isinstance(vs, ReplayStep):
            raise TypeError("replay transactions are captured by ReplayGraphs")
        self.vs, self.loop, self.arena = vs, loop, arena
        self.sets = len(ring_rows)
        self.n = self.sets if (not arena or self.sets % 2 == 0) else 2 * self.sets
        self.graphs, self.txns = [], []
        B = loop.B
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        saved = vs.txn
        try:
            for i in range(self.n):
                # the parity an eagerly driven loop would use at step i (ids 1, 2, ...)
                txn = 2 + ((i + 1) % 2) if arena else 2
                vs.txn = txn
                rows, logits = ring_rows[i % self.sets], ring_logits[i % self.sets]
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    vs._tags.zero_()
                    if arena:
                        vs.verify_all_at(B, loop.cu_rows, rows)
                    else:
                        vs.verify_all(B, loop.cu_rows, loop.src_slot, rows)
                    vs.accept(B, loop.cu_rows, logits, tokens)
                    if arena:
                        gs.gdn_commit_at(vs.d, B, vs.L, vs.cap, loop.cu_rows, vs.accept_len, vs.area_off[txn & 1],
                                         vs.ckpt_layer_stride, vs.tags(B), txn, vs.loc, vs.status)
                    else:
                        vs.commit(B, loop.cu_rows, loop.dst_slot)
                self.graphs.append(g)
                self.txns.append(txn)
        finally:
            vs.txn = saved
        torch.cuda.current_stream().wait_stream(stream)

    def launch(self, step_no: int):
        """Transaction number ``step_no`` (input set step_no modulo the number of sets)."""
        i = step_no % self.n
        self.vs.txn = self.txns[i]
        self.graphs[i].replay()


class MixedTransaction:
    """One planned transaction that holds both prefill sequences and decode
    requests, for every layer.

    The planner has already deferred every draft of such a transaction (each
    decode request verifies one row) and given every writer a destination
    slot that no other request of the transaction reads, so the two halves
    touch disjoint state: the prefills (``gdn_chunked_prefill`` per layer,
    publishing only final states) run on a side stream while the decode half
    (verify of every layer, greedy accept, commit) runs on the caller's
    stream.  Before returning, the caller's stream waits for the side stream,
    so whatever is queued next (the readback, the next transaction's verify
    of a just-prefilled sequence) sees the published states.  With
    ``overlap=False`` both halves run in order on the caller's stream.
    """

    def __init__(self, vs: VerifyStep, max_seqs: int, max_prefill_rows: int, chunk: int = 64,
                 overlap: bool = True):
        self.vs = vs
        self.max_seqs = max_seqs
        self.max_rows = max_prefill_rows
        self.chunk = chunk
        self.overlap = overlap
        self.ws_bytes = gs.gdn_prefill_workspace_bytes(vs.d, max_seqs, max_prefill_rows)
        self.ws = torch.empty((max(self.ws_bytes, 8),), dtype=torch.uint8, device=vs.dev)
        n = max(vs.max_batch, max_seqs)
        self.h_tab = torch.zeros((6, n + 1), dtype=torch.int32).pin_memory()
        self.h_np = self.h_tab.numpy()
        self.d_tab = torch.zeros((6, n + 1), dtype=torch.int32, device=vs.dev)
        self.side = torch.cuda.Stream(device=vs.dev) if overlap else None
        self.done = torch.cuda.Event()

    def upload(self, plan: "gs.Plan", stream=None):
        """Copies the plan's decode (cu, src, dst) and prefill (cu, src, dst)
        tables to the device on the caller's stream."""
        a, c = plan.arrays, plan.c
        B, P = c.n_decode, c.n_prefill
        if B > self.vs.max_batch or P > self.max_seqs:
            raise ValueError("plan larger than the transaction buffers")
        if P and a["pre_cu"][P] > self.max_rows:
            raise ValueError("prefill rows exceed the workspace")
        self.h_np[0, :B + 1] = a["dec_cu"][:B + 1]
        self.h_np[1, :B] = a["dec_src"][:B]
        self.h_np[2, :B] = a["dec_dst"][:B]
        self.h_np[3, :P + 1] = a["pre_cu"][:P + 1]
        self.h_np[4, :P] = a["pre_src"][:P]
        self.h_np[5, :P] = a["pre_dst"][:P]
        self.d_tab.copy_(self.h_tab, non_blocking=True)

    def prefill_layers(self, plan: "gs.Plan", pre_rows: Sequence[LayerRows], pre_o, stream=None):
        vs, c = self.vs, plan.c
        P = c.n_prefill
        pre_cu = plan.arrays["pre_cu"]
        R = int(pre_cu[P])
        max_len = int(max(pre_cu[i + 1] - pre_cu[i] for i in range(P)))
        for l in range(vs.L):
            x = pre_rows[l]
            gs.gdn_chunked_prefill(vs.d, P, R, self.d_tab[3], max_len, x.q, x.k, x.v, x.g, x.beta, vs.pool_layer(l),
                                   vs.slot_stride, vs.num_slots, self.d_tab[4, :P], self.d_tab[5, :P], pre_o[l],
                                   self.chunk, self.ws, self.ws_bytes, vs.status, stream)

    def run(self, plan: "gs.Plan", dec_rows: Sequence[LayerRows], pre_rows: Sequence[LayerRows], pre_o,
            logits: torch.Tensor, tokens: torch.Tensor):
        """Queues the transaction (after ``upload``).  ``pre_o[l]`` receives
        layer l's prefill outputs; decode outputs land in ``vs.o``."""
        vs, c = self.vs, plan.c
        B, P = c.n_decode, c.n_prefill
        main = torch.cuda.current_stream(vs.dev)
        if P:
            if self.overlap:
                self.side.wait_stream(main)          # tables and inputs are queued on the caller's stream
                with torch.cuda.stream(self.side):
                    self.prefill_layers(plan, pre_rows, pre_o)
                self.done.record(self.side)
            else:
                self.prefill_layers(plan, pre_rows, pre_o)
        if B:
            vs.txn = (vs.txn + 1) & 0xFFFFFFFF
            cu, src, dst = self.d_tab[0], self.d_tab[1, :B], self.d_tab[2, :B]
            vs.verify_all(B, cu, src, dec_rows)
            vs.accept(B, cu, logits, tokens)
            vs.commit(B, cu, dst)
        if P and self.overlap:
            main.wait_event(self.done)
