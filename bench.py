#!/usr/bin/env python3
"""Benchmark: K-draft MTP verification over GatedDeltaNet layers on GB300.

One step = one decode-only transaction of the workload: host plan
(plan_transaction) -> gdn_verify for every layer -> mtp_greedy_accept ->
gdn_commit -> the one device-to-host read of accept lengths / bonus / emitted
tokens -> slot-pool release.  The metric is verified tokens per second
(sum over requests of accepted drafts + 1) and the HBM bandwidth of
verify + commit from algorithmic bytes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload paged256]
    python bench.py --impl reference ...   # the CPU oracle on the host cores

Multi-GPU (torchrun): requests are independent, so every rank runs its own
copy of the workload (weak scaling); the only collective is the barrier and
the max of the timed region.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdnsynth as sy  # noqa: E402

S_ROW_IO = lambda d: (2 * d.h_qk * d.d_k * 2 + 2 * d.h_v * d.d_v * 2 + 2 * d.h_v * 4)  # q,k,v,o bf16; g,beta fp32

WORKLOADS = {
    "paged256": sy.SPECS["paged256"],
    "cb16": sy.SPECS["cb16"],
    "batch1": sy.SPECS["batch1"],
    "tiny": sy.SPECS["tiny"],
    # a small case for ncu captures: 32 requests, 64 slots, 2 layers (inputs still larger than L2)
    "small": sy.Spec("small", sy.DIMS_FULL, 2, 32, 3, 3, 20, sy.VOCAB_FULL, 2.0, 0.85, 64, 0, 2, 40),
    # the DRAM-traffic capture case: 128 requests, 256 slots, 2 layers (~3.5 GB on the device; one verify
    # launch moves 1.35 GB, ten times L2, so lines still dirty in L2 at the end are a small share)
    "ncu128": sy.Spec("ncu128", sy.DIMS_FULL, 2, 128, 3, 3, 20, sy.VOCAB_FULL, 2.0, 0.85, 256, 0, 2, 41),
}

WORKLOAD_TEXT = {
    "paged256": "paged large batch: 256 requests in a pool of 1024 FP32 state slots (seeded permutation, 16 "
                "requests share a prefix slot, copy-on-write), 30 GDN layers, H_qk=16, H_v=32, d_k=d_v=128, K=3, "
                "acceptance Bernoulli 0.85, vocab 151936 bf16 logits",
    "cb16": "continuous batch: 16 requests x 30 GDN layers, K ~ U{0..3} per step, ragged rows, Bernoulli 0.85",
    "batch1": "batch-1 verify: 1 request, 1 GDN layer, K=3, vocab 151936",
    "tiny": "tiny: 1 request, 1 layer, 2 heads, d=16, K=3, vocab 64",
    "small": "ncu case: 32 requests, 64 slots, 2 layers, K=3",
    "ncu128": "DRAM-traffic case: 128 requests, 256 slots, 2 layers, K=3",
}

METRIC = "verified tokens/s and GDN verify+commit HBM GB/s (% of GB300 peak)"
HBM_SPEC_GBS = 7900.0   # nominal HBM3e bandwidth of one GB300, for context beside the measured peak


def src_digest(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def committed_traffic(kernel: str, src_path: str):
    """DRAM traffic of one launch of ``kernel`` from the committed ncu summary
    under profiles/ (a line ``traffic: kernel=K src_sha=H workload=W
    alg_bytes_per_launch=A dram_bytes_per_launch=D``, written from a small-case
    capture).  Returns (dram/alg ratio, note); the ratio is None, with the
    reason, when no summary holds one or the kernel source changed since."""
    import glob
    want = src_digest(src_path)
    found = None
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(f) as fh:
            for ln in fh:
                ln = ln.strip().strip("`")
                if not ln.startswith("traffic:"):
                    continue
                kv = dict(x.split("=", 1) for x in ln[len("traffic:"):].split() if "=" in x)
                if kv.get("kernel") == kernel:
                    found = (kv, os.path.basename(f))
    if found is None:
        return None, "no committed ncu DRAM capture of %s" % kernel
    kv, fname = found
    if kv.get("src_sha") != want:
        return None, "%s changed since the DRAM capture in profiles/%s" % (os.path.basename(src_path), fname)
    ratio = float(kv["dram_bytes_per_launch"]) / float(kv["alg_bytes_per_launch"])
    return ratio, "profiles/%s: %s workload, DRAM/algorithmic bytes %.4f, scaled to this launch's bytes" % (
        fname, kv.get("workload", "?"), ratio)


def prefill_flops(lengths, h_v, d=128, C=64):
    """Algorithmic flops of the chunk form: per chunk of n tokens and head,
    n^2 (6 d_k + 4 d_v) + 6 n d_k d_v + n^3 / 3."""
    tot = 0.0
    for L in lengths:
        for c0 in range(0, L, C):
            n = min(C, L - c0)
            tot += n * n * (6 * d + 4 * d) + 6 * n * d * d + n ** 3 / 3.0
    return tot * h_v


# MMA work the prefill kernel issues per (chunk, v-head), in units of one
# M128 x N64 x K16 bf16 product (2 * 128 * 64 * 16 flop): phase A 40 (S W^T
# three split terms, S Q^T two, over K = 128), [K;Q] K^T 8, phase B 28
# (U^T P^T three terms, (U^T diag(dec)) K two terms at N = 128, K = 64), W^T
# and Ut^T 16 (two terms each).  Split terms and padding rows count; the
# algorithmic flops do not.
PREFILL_MMA_UNITS_PER_CHUNK = 92
PREFILL_MMA_UNIT_FLOP = 2 * 128 * 64 * 16


def load_tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s): the measured burst figure, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


PREFILL_SETS = {
    "prefill": None,                  # 8 sequences, log-uniform lengths in [512, 32768]
    "prefill_small": [2048, 2048, 2048, 2048],
}


def bench_prefill(dev, lengths, reps=5, warmup=3):
    """Times gdn_chunked_prefill of one layer over the ragged batch (inputs
    resident in HBM; the 8 sequences' rows are ~1.6 GB, larger than L2)."""
    from speculative_decoding_hybrid_gb300 import binding as gs
    dims = sy.DIMS_FULL
    n = len(lengths)
    rows, cu, s0 = sy.prefill_inputs(lengths, dims, seed=3, device=dev)
    R = int(cu[-1])
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    pool = torch.zeros((2 * n, dims.h_v, dims.d_v, dims.d_k), dtype=torch.float32, device=dev)
    pool[:n] = s0
    src = torch.tensor([-1] * (n // 2) + list(range(n // 2, n)), dtype=torch.int32, device=dev)
    dst = torch.tensor(list(range(n, 2 * n)), dtype=torch.int32, device=dev)
    ws_bytes = gs.gdn_prefill_workspace_bytes(d, n, R)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    o = torch.empty((R, dims.h_v, dims.d_v), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_d = cu.to(dev)

    def call():
        gs.gdn_chunked_prefill(d, n, R, cu_d, max(lengths), rows.q, rows.k, rows.v, rows.g, rows.beta, pool,
                               pool.stride(0), pool.shape[0], src, dst, o, 64, ws, ws_bytes, st)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    evs = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / reps
    flops = prefill_flops(lengths, dims.h_v)
    if int(st.item()) != 0:
        raise RuntimeError("prefill status %d" % int(st.item()))
    chunks = sum((L + 63) // 64 for L in lengths)
    issued = chunks * dims.h_v * PREFILL_MMA_UNITS_PER_CHUNK * PREFILL_MMA_UNIT_FLOP
    bf16_peak = load_tensor_peak()
    return {"tokens": R, "sequences": n, "ms_per_call": ms, "tokens_per_s": R / (ms * 1e-3),
            "alg_tflops": flops / (ms * 1e-3) / 1e12,
            "tensor_frac_alg": flops / (ms * 1e-3) / 1e12 / bf16_peak,
            "issued_mma_tflops": issued / (ms * 1e-3) / 1e12,
            "tensor_frac_issued": issued / (ms * 1e-3) / 1e12 / bf16_peak,
            "bf16_peak_tflops": bf16_peak, "launches_per_call": 2,
            "workspace_bytes": ws_bytes}


def bench_mixed(dev, lengths, n_decode=256, layers=30, reps=3, warmup=1, vocab=151936):
    """One mixed transaction over every layer: the prefill set (chunked,
    publishing final states) and n_decode decode requests asking for K=3,
    which the planner defers to one row each (verify + accept + commit).
    Timed with the prefills on a side stream (overlapped) and in order on
    one stream.  Every layer reads the same prefill input set (1.6 GB, larger
    than L2) and its own decode rows."""
    from speculative_decoding_hybrid_gb300 import binding as gs
    from speculative_decoding_hybrid_gb300.step import LayerRows, MixedTransaction, VerifyStep
    dims = sy.DIMS_FULL
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    n = len(lengths)
    num_slots = n_decode + n + 8
    pool_c = gs.Pool(num_slots)
    dec_slots = [pool_c.alloc() for _ in range(n_decode)]
    cont = [pool_c.alloc() for _ in range(n - n // 2)]       # continued prefixes
    reqs = [(gs.REQ_PREFILL, 0, L, 0, 1 << 30, -1) for L in lengths[:n // 2]] + \
           [(gs.REQ_PREFILL, 0, L, 64, 1 << 30, s) for L, s in zip(lengths[n // 2:], cont)] + \
           [(gs.REQ_DECODE, 3, 0, 100, 1 << 30, s) for s in dec_slots]
    R = sum(lengths)
    plan = gs.Plan(len(reqs))
    st = gs.plan_transaction(gs.make_reqs(reqs), len(reqs), gs.gdn_plan_limits(R + 4 * n_decode, len(reqs), 3),
                             pool_c, plan)
    if st != gs.GDN_OK or plan.c.n_decode != n_decode or plan.c.n_prefill != n:
        raise RuntimeError("mixed plan: status %d" % st)
    pool = torch.empty((num_slots, layers, dims.h_v, dims.d_v, dims.d_k), dtype=torch.float32, device=dev)
    sy.state(sy.generator(5, dev), pool.shape, dev, out=pool)
    vs = VerifyStep(d, layers, num_slots, n_decode, n_decode, vocab, dev, pool=pool)
    rows, cu, _ = sy.prefill_inputs(lengths, dims, seed=3, device=dev)
    pre = [LayerRows(rows.q, rows.k, rows.v, rows.g, rows.beta)] * layers
    dec = []
    for l in range(layers):
        x = sy.rows(sy.generator(sy.mix_seed(6, l), dev), n_decode, dims, dev)
        dec.append(LayerRows(x.q, x.k, x.v, x.g, x.beta))
    lg, _ = sy.logits(sy.generator(7, dev), n_decode, vocab, 2.0, dev)
    tok = torch.zeros(n_decode, dtype=torch.int32, device=dev)
    o = torch.empty((R, dims.h_v, dims.d_v), dtype=torch.bfloat16, device=dev)
    res = {"prefill_tokens": R, "sequences": n, "decode_requests": n_decode, "layers": layers,
           "deferred_drafts": plan.deferred}
    for overlap in (True, False):
        mt = MixedTransaction(vs, n, R, overlap=overlap)
        mt.upload(plan)
        for _ in range(warmup):
            mt.run(plan, dec, pre, [o] * layers, lg, tok)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            mt.run(plan, dec, pre, [o] * layers, lg, tok)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        res["ms_overlapped" if overlap else "ms_in_order"] = ms
        del mt
    if int(vs.status.item()) != 0:
        raise RuntimeError("mixed transaction status %d" % int(vs.status.item()))
    ms = res["ms_overlapped"]
    res["tokens_per_s"] = (R + n_decode) / (ms * 1e-3)
    res["alg_tflops_prefill"] = prefill_flops(lengths, dims.h_v) * layers / (ms * 1e-3) / 1e12
    del vs, pool
    torch.cuda.empty_cache()
    return res


def rank_spec(spec: sy.Spec, rank: int) -> sy.Spec:
    """Requests are independent problems: rank r runs its own batch, drawn
    with its own seed (weak scaling, no data-path exchange)."""
    import dataclasses
    return spec if rank == 0 else dataclasses.replace(spec, seed=spec.seed + 1000 * rank)


def reduce_across_ranks(ms: float, tokens: float, device=None):
    """Whole-job figures: the slowest rank's timed region and the tokens of
    all ranks.  The barrier and these two reductions are the only collectives."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, tokens
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.idx)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload set-up (device)
# ---------------------------------------------------------------------------

class timed:
    """Records a CUDA event pair on the current stream around a block of
    ``n`` launches into ``ev[name]`` (a list of (start, end, n)); no-op when
    ``ev`` is None."""

    def __init__(self, ev, name, n):
        self.ev, self.name, self.n = ev, name, n

    def __enter__(self):
        if self.ev is not None:
            self.a = torch.cuda.Event(enable_timing=True)
            self.a.record()

    def __exit__(self, *exc):
        if self.ev is not None:
            b = torch.cuda.Event(enable_timing=True)
            b.record()
            self.ev.setdefault(self.name, []).append((self.a, b, self.n))
        return False


def per_launch_ms(ev, name):
    """Average device time per launch of a kernel class: the event-timed
    spans over the launches they enclose (back-to-back launches on one
    stream, so the few-microsecond gaps between them count against it).
    A span is an event pair, or (milliseconds, None) from the library's
    host driver, which times the same launches with events of its own."""
    spans = ev.get(name, [])
    n = sum(x[2] for x in spans)
    return sum(a if b is None else a.elapsed_time(b) for a, b, _ in spans) / max(n, 1), n


class Bench:
    def __init__(self, spec: sy.Spec, dev, rank=0, arena=False, replay=False, python_driver=False):
        from speculative_decoding_hybrid_gb300 import binding as gs
        from speculative_decoding_hybrid_gb300.step import ArenaStep, DecodeLoop, LayerRows, ReplayStep, VerifyStep
        self.arena = arena
        self.replay = replay
        self.native = not (replay or python_driver)
        self._kms = (ctypes.c_float * 3)()
        self.gs, self.spec, self.dev = gs, spec, dev
        d = spec.dims
        self.d = d
        self.cap = spec.batch * (spec.k_max + 1)
        slot_of, free, ref = sy.initial_slots(spec)
        order = []
        for s in slot_of:
            if s not in order:
                order.append(s)
        order += list(free)
        self.pool_c = gs.Pool(spec.num_slots, order)
        seen = set()
        for s in slot_of:
            if s in seen:
                self.pool_c.share(s)
            else:
                self.pool_c.alloc()
                seen.add(s)
        if arena:
            self.vs = ArenaStep(gs.dims(d.h_qk, d.h_v, d.d_k, d.d_v), spec.layers, spec.num_slots, self.cap,
                                spec.batch, spec.vocab, dev)
            sy.pool_state(spec, dev, out=self.vs.pool)
            self.vs.point_at_slots(slot_of)
        else:
            pool = torch.empty((spec.num_slots, spec.layers, d.h_v, d.d_v, d.d_k), dtype=torch.float32, device=dev)
            sy.pool_state(spec, dev, out=pool)
            cls = ReplayStep if replay else VerifyStep
            self.vs = cls(gs.dims(d.h_qk, d.h_v, d.d_k, d.d_v), spec.layers, spec.num_slots, self.cap,
                          spec.batch, spec.vocab, dev, pool=pool)
        self.loop = DecodeLoop(self.vs, slot_of, self.pool_c, k_max=spec.k_max)
        self.rows = []
        self.logits, self.targets = [], []
        for i in range(spec.ring):
            rl = []
            for l in range(spec.layers):
                r = sy.ring_rows(spec, l, i, self.cap, dev)
                rl.append(LayerRows(r.q, r.k, r.v, r.g, r.beta))
            self.rows.append(rl)
            lg, tgt = sy.ring_logits(spec, i, self.cap, dev)
            self.logits.append(lg)
            self.targets.append(tgt.tolist())
        self.ks = sy.k_table(spec, 100000 if spec.k_fixed is not None else spec.steps)
        self.tok_h = torch.zeros(self.cap, dtype=torch.int32).pin_memory()
        self.tok_d = torch.zeros(self.cap, dtype=torch.int32, device=dev)
        self.step_no = 0
        self.verified = 0
        self.last_plan = None

    def precompute_drafts(self, n_steps):
        """Draft tokens are synthetic inputs: draw them for every step before
        timing, assuming the planner grants the requested draft counts (it
        does when no request is near its length limit; checked per step)."""
        self.pre = {}
        for s in range(n_steps):
            ks = self.ks[s % self.ks.shape[0]].tolist()
            drafts = sy.step_drafts(self.spec, s, ks, self.targets[s % self.spec.ring])
            toks = [t for dr in drafts for t in dr]
            h = torch.zeros(self.cap, dtype=torch.int32)
            h[:len(toks)] = torch.tensor(toks, dtype=torch.int32)
            self.pre[s] = (ks, h.pin_memory())

    def prepare(self, s):
        """Host part of a step: plan, drafts, table upload."""
        ks = self.ks[s % self.ks.shape[0]].tolist()
        p = self.loop.plan_step(ks)
        ring = s % self.spec.ring
        pre = getattr(self, "pre", {}).get(s)
        if pre is not None and pre[0] == p.k:
            self.tok_d.copy_(pre[1], non_blocking=True)
        else:
            drafts = sy.step_drafts(self.spec, s, p.k, self.targets[ring])
            toks = [t for dr in drafts for t in dr]
            self.tok_h[:len(toks)] = torch.tensor(toks, dtype=torch.int32)
            self.tok_d.copy_(self.tok_h, non_blocking=True)
        self.loop.upload_tables()
        self.last_plan = p
        return ring, p

    def step(self, ev=None):
        """One transaction.  ``ev`` (optional) collects, per kernel class, CUDA
        event pairs around its launches and the number of launches between
        them: the verify pair spans every layer's launch of one step.  The
        copy-commit path goes through the library's host driver
        (``gdn_decode_transaction``) unless ``python_driver`` is set."""
        if self.native:
            return self.native_step(ev)
        p = self.launch(ev)
        return self.finish(p)

    def upload_drafts(self):
        """The step's draft ids (precomputed synthetic inputs for the
        requested draft counts) to the device; returns the counts."""
        s = self.step_no
        ks = self.ks[s % self.ks.shape[0]].tolist()
        pre = self.pre.get(s)
        if pre is None or pre[0] != ks:
            raise RuntimeError("draft ids of step %d were not precomputed" % s)
        self.tok_d.copy_(pre[1], non_blocking=True)
        return ks

    def native_step(self, ev=None, ks=None):
        """One transaction by ``gdn_decode_transaction``: the step's draft ids
        go to the device (unless ``ks`` says they already did), then one
        library call plans, verifies, accepts, commits and reads back."""
        s = self.step_no
        loop = self.loop
        B = loop.B
        if ks is None:
            ks = self.upload_drafts()
        loop.req_np[:B, 1] = np.asarray(ks, dtype=np.int32)
        ring = s % self.spec.ring
        acc = loop.transaction(self.rows[ring], self.logits[ring], self.tok_d,
                               kernel_ms=self._kms if ev is not None else None)
        p = loop.plan
        if p.k != ks:
            raise RuntimeError("the planner changed the draft counts of step %d" % s)
        if ev is not None:
            for name, ms, n in (("verify", self._kms[0], self.spec.layers), ("accept", self._kms[1], 1),
                                ("commit", self._kms[2], 1)):
                ev.setdefault(name, []).append((float(ms), None, n))
        self.last_plan = p
        n_ver = int(acc.sum()) + B
        self.step_no += 1
        self.verified += n_ver
        return n_ver, p

    def launch(self, ev=None):
        """Plans the step and queues its kernels (no host synchronisation)."""
        s = self.step_no
        ring, p = self.prepare(s)
        vs, loop = self.vs, self.loop
        B = loop.B
        rows = self.rows[ring]
        if self.replay:
            vs._advance()
            with timed(ev, "verify", self.spec.layers):
                vs._verify_all(B, loop.cu_rows, loop.src_slot, loop.dst_slot, rows)
            with timed(ev, "accept", 1):
                vs.accept(B, loop.cu_rows, self.logits[ring], self.tok_d)
            vs.prev_cu.copy_(loop.cu_rows[:B + 1], non_blocking=True)
            vs.prev_rows = rows
            vs.pending = True
        elif self.arena:
            vs.txn = (vs.txn + 1) & 0xFFFFFFFF
            with timed(ev, "verify", self.spec.layers):
                vs.verify_all_at(B, loop.cu_rows, rows)
            with timed(ev, "accept", 1):
                vs.accept(B, loop.cu_rows, self.logits[ring], self.tok_d)
            with timed(ev, "commit", 1):
                self.gs.gdn_commit_at(vs.d, B, vs.L, vs.cap, loop.cu_rows, vs.accept_len, vs.area_off[vs.txn & 1],
                                      vs.ckpt_layer_stride, vs.tags(B), vs.txn, vs.loc, vs.status)
        else:
            vs.txn = (vs.txn + 1) & 0xFFFFFFFF
            with timed(ev, "verify", self.spec.layers):
                vs.verify_all(B, loop.cu_rows, loop.src_slot, rows)
            with timed(ev, "accept", 1):
                vs.accept(B, loop.cu_rows, self.logits[ring], self.tok_d)
            with timed(ev, "commit", 1):
                vs.commit(B, loop.cu_rows, loop.dst_slot)
        return p

    def finish(self, p):
        """The step's one readback, then the host bookkeeping."""
        loop = self.loop
        acc, bon, out = loop.readback()
        n_ver = int(acc.sum().item()) + loop.B
        loop.finish(acc)
        self.step_no += 1
        self.verified += n_ver
        return n_ver, p

    def step_bytes(self, p):
        """Algorithmic bytes of verify (all layers) and commit for a plan."""
        d = self.d
        S = d.h_v * d.d_v * d.d_k * 4
        rows = p.decode_rows
        distinct_src = len(set(p.dec_src))
        verify = self.spec.layers * (distinct_src * S + rows * S + rows * S_ROW_IO(d))
        if self.replay:
            # read the slot, write it back (the replay), row inputs of this and the previous transaction
            verify = self.spec.layers * (p.n_decode * 2 * S + rows * S_ROW_IO(d) + rows * (S_ROW_IO(d) // 2))
        commit = 0 if (self.arena or self.replay) else self.spec.layers * p.n_decode * 2 * S
        accept = rows * self.spec.vocab * 2
        return verify, commit, accept


def run_zero_copy(spec, dev, args, replay=False, graph=False):
    """The same steps with the commit that rewrites locations instead of
    copying states (verify reads from a state arena), or with compact
    fixed-state replay (no checkpoints), optionally launched as one CUDA
    graph per transaction."""
    b = Bench(spec, dev, 0, arena=not replay, replay=replay)
    b.precompute_drafts(args.warmup + args.steps)
    for _ in range(args.warmup):
        b.step()
    torch.cuda.synchronize()
    if graph:
        from speculative_decoding_hybrid_gb300.step import ReplayGraphs
        graphs = ReplayGraphs(b.vs, b.loop, b.rows, b.logits, b.tok_d)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record()
        tok = 0
        for _ in range(args.steps):
            s = b.step_no
            b.prepare(s)
            graphs.launch(s, b.rows)
            acc, bon, out = b.loop.readback()
            tok += int(acc.sum().item()) + b.loop.B
            b.loop.finish(acc)
            b.step_no += 1
        end.record()
        torch.cuda.synchronize()
        ms = start.elapsed_time(end)
        if int(b.vs.status.item()) != 0:
            raise RuntimeError("graph replay loop status %d" % int(b.vs.status.item()))
        res = {"value": tok / (ms * 1e-3), "unit": "verified tokens/s", "ms_per_step": ms / args.steps,
               "launches_per_step": 1, "kernels_per_step": spec.layers + 2}
        del graphs, b
        torch.cuda.empty_cache()
        return res
    ev = {}
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    tok, vbytes = 0, 0
    for _ in range(args.steps):
        n, p = b.step(ev)
        tok += n
        vbytes += b.step_bytes(p)[0]
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    v_ms, n_ver = per_launch_ms(ev, "verify")
    c_ms, _ = per_launch_ms(ev, "commit")
    peak, _ = load_peaks()
    gbs = vbytes / ((v_ms * n_ver + c_ms * args.steps) * 1e-3) / 1e9
    if int(b.vs.status.item()) != 0:
        raise RuntimeError("zero-copy loop status %d" % int(b.vs.status.item()))
    res = {"value": tok / (ms * 1e-3), "unit": "verified tokens/s", "ms_per_step": ms / args.steps,
           "verify_ms": v_ms, "commit_at_ms": c_ms, "verify_commit_gbs": gbs, "verify_commit_frac": gbs / peak,
           "state_gib": (b.vs.arena.numel() if not replay else b.vs.pool.numel()) * 4 / 2 ** 30,
           "driver": "gdn_decode_transaction_at" if b.native else "Python"}
    del b
    torch.cuda.empty_cache()
    return res


def run_step_graphs(spec, dev, warmup=5, steps=None, arena=False):
    """The checkpointing transaction of a workload (every layer's verify,
    the accept and the commit; zero-copy over a state arena with ``arena``)
    replayed as one CUDA graph per step, with the host planning, uploading
    and reading back around it."""
    from speculative_decoding_hybrid_gb300.step import StepGraphs
    b = Bench(spec, dev, 0, arena=arena, python_driver=True)
    steps = steps or spec.steps
    b.precompute_drafts(warmup + 2 * steps)
    for _ in range(warmup):
        b.step()
    torch.cuda.synchronize()
    graphs = StepGraphs(b.vs, b.loop, b.rows, b.logits, b.tok_d)

    def one():
        s = b.step_no
        b.prepare(s)
        graphs.launch(s)
        acc, _, _ = b.loop.readback()
        n = int(acc.sum().item()) + b.loop.B
        b.loop.finish(acc)
        b.step_no += 1
        return n
    for _ in range(min(steps, 3)):
        one()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    tok = 0
    for _ in range(steps):
        tok += one()
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    if int(b.vs.status.item()) != 0:
        raise RuntimeError("step-graph loop status %d" % int(b.vs.status.item()))
    res = {"workload": spec.name, "value": tok / (ms * 1e-3), "unit": "verified tokens/s", "steps": steps,
           "ms_per_step": ms / steps, "launches_per_step": 1, "kernels_per_step": spec.layers + 4,
           "commit": "zero-copy (state arena)" if arena else "copy"}
    del graphs, b
    torch.cuda.empty_cache()
    return res


def run_workload_block(spec, dev, warmup=5, steps=None):
    """Another decode workload timed like the headline line (copy commit through
    gdn_decode_transaction, event-timed verify/commit), for the line's
    secondary blocks: verified tokens/s and the verify+commit HBM fraction."""
    b = Bench(spec, dev, 0)
    steps = steps or spec.steps
    b.precompute_drafts(warmup + steps)
    for _ in range(warmup):
        b.step()
    torch.cuda.synchronize()
    ev = {}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    tok = vbytes = cbytes = 0
    for _ in range(steps):
        n, p = b.step(ev)
        tok += n
        v, c, _ = b.step_bytes(p)
        vbytes += v
        cbytes += c
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    if int(b.vs.status.item()) != 0:
        raise RuntimeError("%s loop status %d" % (spec.name, int(b.vs.status.item())))
    v_ms, n_ver = per_launch_ms(ev, "verify")
    c_ms, _ = per_launch_ms(ev, "commit")
    peak, _ = load_peaks()
    gbs = (vbytes + cbytes) / ((v_ms * n_ver + c_ms * steps) * 1e-3) / 1e9
    res = {"workload": spec.name, "desc": WORKLOAD_TEXT.get(spec.name, spec.name), "value": tok / (ms * 1e-3),
           "unit": "verified tokens/s", "steps": steps, "ms_per_step": ms / steps,
           "verify_ms_per_launch": v_ms, "commit_ms": c_ms, "verify_commit_gbs": gbs,
           "verify_commit_frac": gbs / peak, "verify_commit_frac_of_spec": gbs / HBM_SPEC_GBS,
           "driver": "gdn_decode_transaction"}
    del b
    torch.cuda.empty_cache()
    return res


def bench_accept_logits(b: Bench, reps=20):
    """mtp_greedy_accept over every row of the batch on logits as the workload
    states them (N(0, 2^2), nothing planted) beside the benchmark's ring
    logits (one target per row planted at +16 so the greedy choice is known
    by construction).  Both 311 MB sets are larger than L2."""
    vs, loop = b.vs, b.loop
    B = loop.B
    R = int(loop.d_tab[0, B].item())
    g = sy.generator(sy.mix_seed(b.spec.seed, 4040), b.dev)
    plain = torch.empty((b.cap, b.spec.vocab), dtype=torch.float32, device=b.dev)
    plain.normal_(0.0, b.spec.logit_std, generator=g)
    lg_plain = plain.to(torch.bfloat16)
    del plain
    out = {"rows": R, "vocab": b.spec.vocab}
    for name, lg in (("stated_N(0,2^2)", lg_plain), ("planted_ring", b.logits[0])):
        for _ in range(3):
            vs.accept(B, loop.cu_rows, lg, b.tok_d)
        torch.cuda.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            vs.accept(B, loop.cu_rows, lg, b.tok_d)
        e.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(e) / reps
        out[name] = {"ms": ms, "gbs": R * b.spec.vocab * 2 / (ms * 1e-3) / 1e9}
    del lg_plain
    torch.cuda.empty_cache()
    return out


def _packed_layout(b: Bench):
    """Byte offsets of every layer's row inputs and the logits in one packed
    buffer (each piece 256-byte aligned)."""
    pieces, off = [], 0
    for r in b.rows[0]:
        for x in (r.q, r.k, r.v, r.g, r.beta):
            pieces.append((off, x.dtype, tuple(x.shape)))
            off += (x.numel() * x.element_size() + 255) // 256 * 256
    lg = b.logits[0]
    pieces.append((off, lg.dtype, tuple(lg.shape)))
    off += (lg.numel() * lg.element_size() + 255) // 256 * 256
    return pieces, off


def _views(buf, pieces):
    out = []
    for off, dt, shape in pieces:
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dt).element_size()
        out.append(buf[off:off + nbytes].view(dt).view(shape))
    return out


def stage_e2e(b: Bench):
    """Every ring set's inputs packed into one pinned host buffer, and two
    device staging buffers of the same layout (one copy per step)."""
    from speculative_decoding_hybrid_gb300.step import LayerRows
    pieces, total = _packed_layout(b)
    host = []
    for i in range(b.spec.ring):
        hb = torch.empty((total,), dtype=torch.uint8).pin_memory()
        src = [x for r in b.rows[i] for x in (r.q, r.k, r.v, r.g, r.beta)] + [b.logits[i]]
        for v, x in zip(_views(hb, pieces), src):
            v.copy_(x.detach().to("cpu"))
        host.append(hb)
    stages = []
    for _ in range(2):
        db = torch.empty((total,), dtype=torch.uint8, device=b.dev)
        vs = _views(db, pieces)
        rows = [LayerRows(*vs[5 * l:5 * l + 5]) for l in range(len(b.rows[0]))]
        stages.append((db, rows, vs[-1]))
    return host, stages


def run_e2e(b: Bench, host, stages, steps, warmup):
    """Same step through the public API, with every step's inputs copied from
    pinned host memory and the results read back inside the timed region.
    A step's kernels are queued first; then the next step's inputs (one
    packed copy) go to the other device staging buffer on a copy stream while
    this step computes; a step waits for its own inputs' copy event."""
    spec = b.spec
    saved_rows, saved_logits = b.rows, b.logits
    copy_stream = torch.cuda.Stream()
    compute = torch.cuda.current_stream()
    done = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    free = [torch.cuda.Event(), torch.cuda.Event()]
    moved_bytes = [0]
    copies = []   # (start, done) events of the input copies issued in the timed region

    def issue_copy(step_no, slot, timed_copy=False):
        hb = host[step_no % spec.ring]
        db = stages[slot][0]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(free[slot])  # the staging set's previous reader is done
            if timed_copy:
                st = torch.cuda.Event(enable_timing=True)
                st.record(copy_stream)
            db.copy_(hb, non_blocking=True)
            done[slot].record(copy_stream)
            if timed_copy:
                en = torch.cuda.Event(enable_timing=True)
                en.record(copy_stream)
                copies.append((st, en))
        moved_bytes[0] += hb.numel()

    marks = []   # (start, end) events of the timed steps on the compute stream

    def one(slot, mark=False):
        compute.wait_event(done[slot])
        _, rows, logits = stages[slot]
        b.rows = [rows] * spec.ring
        b.logits = [logits] * spec.ring
        if mark:
            marks.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
            marks[-1][0].record(compute)
        if b.native:
            # the library's host driver blocks until the step is done: the
            # step's draft ids go first, then the next step's inputs are
            # queued on the copy stream (their staging set was released by
            # the step before), then the step runs
            ks = b.upload_drafts()
            issue_copy(b.step_no + 1, slot ^ 1, timed_copy=mark)
            r = b.native_step(ks=ks)
            free[slot].record(compute)
            if mark:
                marks[-1][1].record(compute)
            return r
        p = b.launch()
        free[slot].record(compute)
        if mark:
            marks[-1][1].record(compute)
        issue_copy(b.step_no + 1, slot ^ 1, timed_copy=mark)       # next step's inputs, overlapped
        return b.finish(p)                        # the step's one readback

    try:
        for e in free:
            e.record(compute)
        slot = 0
        issue_copy(b.step_no, slot)
        for _ in range(warmup):
            one(slot)
            slot ^= 1
        torch.cuda.synchronize()
        moved_bytes[0] = 0
        t0 = time.perf_counter()
        tok = 0
        for _ in range(steps):
            n, p = one(slot, mark=True)
            slot ^= 1
            tok += n
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        b.rows, b.logits = saved_rows, saved_logits
    # the packed input copy alone, for context (how much of a step it would cost unhidden)
    ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(copy_stream):
        ca.record(copy_stream)
        stages[0][0].copy_(host[0], non_blocking=True)
        cb.record(copy_stream)
    torch.cuda.synchronize()
    copy_ms = ca.elapsed_time(cb)
    # device idle time between a step's last kernel and the next step's first
    # (the host's readback, planning and launch of the next step)
    gaps = [marks[i][1].elapsed_time(marks[i + 1][0]) for i in range(len(marks) - 1)]
    gap_ms = sum(gaps) / len(gaps) if gaps else 0.0
    # the steps' own device time with the input copies beside them
    spans = [a.elapsed_time(c) for a, c in marks]
    step_ms = sum(spans) / len(spans) if spans else 0.0
    # the input copies as they ran beside the steps (HBM shared with the kernels)
    in_step = [a.elapsed_time(c) for a, c in copies]
    copy_in_step_ms = sum(in_step) / len(in_step) if in_step else 0.0
    h2d = moved_bytes[0] / steps + (b.loop.B + 1) * 3 * 4 + b.cap * 4   # inputs + tables + tokens
    d2h = (2 * spec.batch + b.cap) * 4
    return tok / dt, h2d, d2h, copy_ms, gap_ms, copy_in_step_ms, step_ms


# ---------------------------------------------------------------------------
# CPU oracle arm (baseline)
# ---------------------------------------------------------------------------

def oracle_sample_step(spec: sy.Spec, step: int, n_req: int, seed: int = 0):
    """One step of the workload for n_req requests, run by the FP64 oracle:
    planner model, recurrence over every layer and head with checkpoints,
    greedy choice over the vocabulary, acceptance and commit.  Returns the
    verified tokens."""
    import oracle
    d = spec.dims
    K = spec.k_fixed if spec.k_fixed is not None else spec.k_max
    pool = oracle.PoolModel(n_req)
    reqs = []
    for i in range(n_req):
        _, s = pool.alloc()
        reqs.append(oracle.Req(oracle.DECODE, K, cur_len=1, slot=s))
    P = oracle.plan_transaction(reqs, n_req * (K + 1), n_req, spec.k_max, pool)
    cu = P.dec_cu
    R = cu[-1]
    gen = sy.generator(sy.mix_seed(seed, 4242, step))
    lg, tgt = sy.logits(gen, R, spec.vocab, spec.logit_std)
    drafts = sy.step_drafts(spec, step, P.k, tgt.tolist())
    toks = np.array([t for dr in drafts for t in dr], np.int32)
    am = oracle.argmax_bf16(oracle.bf16_bits(lg))
    res = oracle.greedy_accept(am, toks, np.array(cu), spec.vocab)
    for l in range(spec.layers):
        rows = sy.rows(gen, R, d)
        S0 = sy.state(gen, (n_req, d.h_v, d.d_v, d.d_k))
        units = []
        for r in range(n_req):
            a, b = cu[r], cu[r + 1]
            units += oracle.head_units(rows.q[a:b], rows.k[a:b], rows.v[a:b], rows.g[a:b], rows.beta[a:b], S0[r])
        S, o, ck = oracle.recurrent_units(units, want_ckpt=True)
        for r in range(n_req):
            j = int(res.accept_len[r])
            _ = [ck[r * d.h_v + h][j] for h in range(d.h_v)]     # commit: the accepted checkpoint
    return int(res.accept_len.sum()) + n_req


def cpu_baseline(spec: sy.Spec, budget_s: float = 12.0, n_req: int = 16):
    import oracle
    t0 = time.perf_counter()
    tok, steps = 0, 0
    while steps == 0 or time.perf_counter() - t0 < budget_s:
        tok += oracle_sample_step(spec, steps, n_req)
        steps += 1
    dt = time.perf_counter() - t0
    return {"value": tok / dt, "unit": "verified tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d steps x %d requests x %d layers of the %s workload (FP64 C oracle, OpenMP over "
                      "(request, head); inputs drawn on the host with the same recipe)" %
                      (steps, n_req, spec.layers, spec.name)}


def run_reference(args, spec):
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    n_req = min(4, spec.batch)
    for w in range(args.warmup):
        oracle_sample_step(spec, w, n_req)
    t0 = time.perf_counter()
    tok = 0
    for s in range(args.steps):
        tok += oracle_sample_step(spec, args.warmup + s, n_req)
    dt = time.perf_counter() - t0
    val = tok / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "verified tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "desc": WORKLOAD_TEXT[args.workload],
                       "per_step_sample": "%d of %d requests" % (n_req, spec.batch)},
            "cpu_baseline": {"value": val, "unit": "verified tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": "each step: %d requests x %d layers of the %s workload"
                                                         % (n_req, spec.layers, spec.name)},
            "e2e": {"value": val, "unit": "verified tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="paged256", choices=sorted(WORKLOADS) + sorted(PREFILL_SETS))
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cb16", action="store_true",
                    help="skip the continuous-batch (cb16) block that runs after the paged256 line's loop")
    ap.add_argument("--no-batch1", action="store_true",
                    help="skip the batch-1 block (host driver and CUDA-graph steps)")
    ap.add_argument("--step-graph", dest="step_graph", action="store_true", default=True,
                    help="also time the paged256 checkpointing step as one CUDA graph per step")
    ap.add_argument("--no-step-graph", dest="step_graph", action="store_false")
    ap.add_argument("--zero-copy", dest="zero_copy", action="store_true", default=True,
                    help="also time the zero-copy commit (state arena) on the same workload")
    ap.add_argument("--no-zero-copy", dest="zero_copy", action="store_false")
    ap.add_argument("--replay", dest="replay", action="store_true", default=True,
                    help="also time compact fixed-state replay (no checkpoints) on the same workload")
    ap.add_argument("--no-replay", dest="replay", action="store_false")
    ap.add_argument("--python-driver", action="store_true",
                    help="drive the copy-commit steps from Python (one library call per stage) instead of "
                         "gdn_decode_transaction")
    args = ap.parse_args()
    if args.workload in PREFILL_SETS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "prefill-only workloads have no CPU timing arm"}))
            return
        from speculative_decoding_hybrid_gb300 import build
        build.build()
        dev = torch.device("cuda", 0)
        lengths = PREFILL_SETS[args.workload] or sy.prefill_lengths()
        r = bench_prefill(dev, lengths, reps=args.steps or 5, warmup=args.warmup)
        print(json.dumps({"metric": "chunked prefill tokens/s", "value": r["tokens_per_s"], "unit": "tokens/s",
                          "workload": args.workload, "prefill": r}), flush=True)
        return
    spec = WORKLOADS[args.workload]
    if args.steps is None:
        args.steps = min(spec.steps, 100)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        run_reference(args, spec)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from speculative_decoding_hybrid_gb300 import build
    build.build()
    b = Bench(rank_spec(spec, rank), dev, rank, python_driver=args.python_driver)
    native_driver = b.native
    b.precompute_drafts(args.warmup + args.steps + (0 if args.no_e2e else 3 + args.e2e_steps))
    for _ in range(args.warmup):
        b.step()
    torch.cuda.synchronize()

    ev = {}
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if world == 1 else local)
    sampler.start()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    tok = 0
    vbytes = cbytes = abytes = 0
    for _ in range(args.steps):
        n, p = b.step(ev)
        tok += n
        v, c, a = b.step_bytes(p)
        vbytes += v
        cbytes += c
        abytes += a
    end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = start.elapsed_time(end)
    ms, tok_all = reduce_across_ranks(ms, tok, dev)

    v_ms, n_ver_launch = per_launch_ms(ev, "verify")
    a_ms, _ = per_launch_ms(ev, "accept")
    c_ms, _ = per_launch_ms(ev, "commit")
    peak, peak_kind = load_peaks()
    v_per_launch = vbytes / max(n_ver_launch, 1)
    achieved = v_per_launch / (v_ms * 1e-3) / 1e9
    vc_gbs = (vbytes + cbytes) / ((v_ms * n_ver_launch + c_ms * args.steps) * 1e-3) / 1e9
    src = os.path.join(ROOT, "speculative_decoding_hybrid_gb300", "csrc", "gdn_recurrent.cu")
    ratio, traffic_note = committed_traffic("gdn_verify", src)
    traffic = ratio * v_per_launch if ratio is not None else None

    l2desc = "inputs larger than L2: state pool %.1f GiB, checkpoints %.1f GiB, ring of %d input sets" % (
        b.vs.pool.numel() * 4 / 2 ** 30, b.vs.ckpt.numel() * 4 / 2 ** 30, spec.ring)
    e2e = None
    if not args.no_e2e:
        host, stages = stage_e2e(b)
        val, h2d, d2h, copy_ms, gap_ms, copy_in_step_ms, step_ms = run_e2e(b, host, stages, args.e2e_steps, 3)
        del host, stages
        if world > 1:
            t = torch.tensor([val], device=dev, dtype=torch.float64)
            dist.all_reduce(t)
            val = float(t.item())
        e2e = {"value": val, "unit": "verified tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps,
               "input_copy_ms_alone": copy_ms, "input_copy_gbs": h2d / (copy_ms * 1e-3) / 1e9,
               "device_idle_ms_between_steps": gap_ms, "input_copy_ms_beside_steps": copy_in_step_ms,
               "device_ms_per_step_beside_copies": step_ms}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    def guarded(fn, *a, **k):
        """A secondary measurement that fails records its error instead of
        losing the main line."""
        try:
            return fn(*a, **k)
        except Exception as e:  # noqa: BLE001
            torch.cuda.synchronize()
            return {"error": "%s: %s" % (type(e).__name__, e)}

    prefill = mixed = None
    if not args.no_prefill and args.workload == "paged256":
        prefill = guarded(bench_prefill, dev, sy.prefill_lengths())
        mixed = guarded(bench_mixed, dev, sy.prefill_lengths())
    accept_plain = None
    if world == 1:
        accept_plain = guarded(bench_accept_logits, b)
    zero_copy = replay = replay_graph = cb16 = batch1 = step_graph = None
    if (args.zero_copy or args.replay) and world == 1:
        del b
        torch.cuda.empty_cache()
        if args.workload == "paged256" and not args.no_cb16:
            cb16 = guarded(run_workload_block, WORKLOADS["cb16"], dev, warmup=args.warmup)
            torch.cuda.empty_cache()
        if args.workload == "paged256" and not args.no_batch1:
            b1 = WORKLOADS["batch1"]
            batch1 = {"desc": WORKLOAD_TEXT["batch1"] + "; its 16 MB of state and inputs stay in L2 (the case is "
                              "bound by launches and the host, not HBM)",
                      "driver": guarded(run_workload_block, b1, dev, warmup=args.warmup, steps=400),
                      "step_graph_copy": guarded(run_step_graphs, b1, dev, warmup=args.warmup, steps=400),
                      "step_graph_zero_copy": guarded(run_step_graphs, b1, dev, warmup=args.warmup, steps=400,
                                                      arena=True)}
            torch.cuda.empty_cache()
        if args.workload == "paged256" and args.step_graph:
            step_graph = guarded(run_step_graphs, spec, dev, warmup=args.warmup, steps=args.steps)
            torch.cuda.empty_cache()
        if args.replay:
            replay = guarded(run_zero_copy, spec, dev, args, replay=True)
            torch.cuda.empty_cache()
            replay_graph = guarded(run_zero_copy, spec, dev, args, replay=True, graph=True)
            torch.cuda.empty_cache()
        if args.zero_copy:
            zero_copy = guarded(run_zero_copy, spec, dev, args)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = guarded(cpu_baseline, spec)
    line = {
        "metric": METRIC,
        "value": tok_all / (ms * 1e-3),
        "unit": "verified tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "desc": WORKLOAD_TEXT[args.workload],
                   "l2": l2desc,
                   "driver": "gdn_decode_transaction (one library call per step)" if native_driver
                   else "Python (one library call per stage)",
                   "parallelism": "replicas (requests sharded, no collective)" if world > 1 else "single GPU"},
        "verify_commit_gbs": vc_gbs,
        "verify_commit_frac": vc_gbs / peak,
        "verify_commit_frac_of_spec": vc_gbs / HBM_SPEC_GBS,
        "roofline": {"bound": "hbm", "kernel": "gdn_verify", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_note,
                     "peak_source": peak_kind, "peak_spec": HBM_SPEC_GBS, "frac_of_spec": achieved / HBM_SPEC_GBS,
                     "alg_bytes_per_launch": v_per_launch, "avg_launch_ms": v_ms},
        "kernels_ms": {"gdn_verify": v_ms, "mtp_greedy_accept": a_ms, "gdn_commit": c_ms,
                       "commit_gbs": cbytes / args.steps / (c_ms * 1e-3) / 1e9,
                       "accept_gbs": abytes / args.steps / (a_ms * 1e-3) / 1e9},
        # per step: every layer's verify, the two accept kernels, the commit,
        # and with the host driver its commit gate and two table-moving kernels
        "gpu_launches": args.steps * (spec.layers + 3 + (3 if native_driver else 0)),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "acceptance": {"verified_tokens": tok, "requests": spec.batch},
        "accept_stated_logits": accept_plain,
        "cb16": cb16,
        "batch1": batch1,
        "step_graph": step_graph,
        "prefill": prefill,
        "mixed_transaction": mixed,
        "zero_copy_commit": zero_copy,
        "fixed_state_replay": replay,
        "fixed_state_replay_cuda_graph": replay_graph,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
