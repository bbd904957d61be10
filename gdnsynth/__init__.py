"""Seeded synthetic inputs for GatedDeltaNet speculative verification.

This module only draws tensors: it holds none of the method's arithmetic
(no recurrence, no argmax, no acceptance rule, no planning).  Both the CPU
oracle tests and the CUDA path are fed from here, so that the two sides see
the same input bits.

Recipe (one line per tensor; all draws from a seeded ``torch.Generator``):

* q, k : N(0, 1) per element, L2-normalised per (row, qk-head) in fp32, then
  rounded to bf16 (round-to-nearest-even).
* v    : N(0, 1), rounded to bf16.
* g    : log(sigmoid(x)) with x ~ N(2, 1), computed and stored in fp32
  (the log-decay; alpha = exp(g) lies in (0, 1)).
* beta : sigmoid(x) with x ~ N(0, 1), computed and stored in fp32.
* S_0  : N(0, 0.1^2) fp32 recurrent state, laid out [h_v][d_v][d_k].
* logits: N(0, std^2) rounded to bf16; in every row one target id, drawn
  uniformly, is set to +16.0 so that the row's greedy choice is known by
  construction (an N(0, 4) draw reaches 16 with probability ~1e-15).
* drafts: draft i of a request repeats the target of the row before it
  with probability ``p_accept``, independently, until the first miss; a miss
  is ``(target + 1 + r) mod V`` with r uniform in [0, V-2]; drafts after the
  first miss are uniform in [0, V).

Sizes and seeds of the workloads live in ``SPECS`` and :func:`prefill_lengths`.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

TARGET_LOGIT = 16.0


def mix_seed(*parts: int) -> int:
    """Stable 63-bit seed from integer parts (splitmix64 finaliser chain)."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x = z ^ (z >> 31)
    return x & 0x7FFFFFFFFFFFFFFF


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


@dataclasses.dataclass
class Dims:
    h_qk: int
    h_v: int
    d_k: int
    d_v: int

    @property
    def state_elems(self) -> int:
        return self.h_v * self.d_v * self.d_k


@dataclasses.dataclass
class Rows:
    """Per-token layer inputs, packed by row: q,k [R,h_qk,d_k] bf16,
    v [R,h_v,d_v] bf16, g,beta [R,h_v] fp32."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor

    @property
    def n(self) -> int:
        return self.q.shape[0]

    def slice(self, a: int, b: int) -> "Rows":
        return Rows(self.q[a:b], self.k[a:b], self.v[a:b], self.g[a:b], self.beta[a:b])

    def to(self, device) -> "Rows":
        return Rows(*(t.to(device) for t in (self.q, self.k, self.v, self.g, self.beta)))


# Every draw happens on the generator's own device (so a seed gives the same
# numbers wherever the result is asked for) and is then moved to ``device``.

def _unit_bf16(gen, shape):
    x = torch.randn(shape, generator=gen, device=gen.device, dtype=torch.float32)
    if x.numel():
        x = x / x.norm(dim=-1, keepdim=True)
    return x.to(torch.bfloat16)


def rows(gen, n: int, dims: Dims, device="cpu") -> Rows:
    gd = gen.device
    q = _unit_bf16(gen, (n, dims.h_qk, dims.d_k))
    k = _unit_bf16(gen, (n, dims.h_qk, dims.d_k))
    v = torch.randn((n, dims.h_v, dims.d_v), generator=gen, device=gd, dtype=torch.float32).to(torch.bfloat16)
    xg = torch.randn((n, dims.h_v), generator=gen, device=gd, dtype=torch.float32) + 2.0
    g = torch.nn.functional.logsigmoid(xg)
    xb = torch.randn((n, dims.h_v), generator=gen, device=gd, dtype=torch.float32)
    beta = torch.sigmoid(xb)
    return Rows(*(t.to(device).contiguous() for t in (q, k, v, g, beta)))


def state(gen, shape, device="cpu", std: float = 0.1, out: Optional[torch.Tensor] = None):
    """fp32 N(0, std^2) state; ``shape`` ends in (h_v, d_v, d_k).  With ``out``
    the draw is written into it (it must live on the generator's device)."""
    if out is None:
        x = torch.empty(shape, dtype=torch.float32, device=gen.device)
        x.normal_(0.0, std, generator=gen)
        return x.to(device)
    out.normal_(0.0, std, generator=gen)
    return out


def logits(gen, n: int, vocab: int, std: float, device="cpu"):
    """bf16 logits [n, vocab] and the planted target id per row (int64)."""
    gd = gen.device
    lg = torch.empty((n, vocab), dtype=torch.float32, device=gd)
    if n:
        lg.normal_(0.0, std, generator=gen)
    lg = lg.to(torch.bfloat16)
    tgt = torch.randint(0, vocab, (n,), generator=gen, device=gd, dtype=torch.int64)
    if n:
        lg[torch.arange(n, device=gd), tgt] = TARGET_LOGIT
    return lg.to(device), tgt.to(device)


def drafts(gen_cpu, targets: List[int], ks: List[int], vocab: int, p_accept: float,
           last_tokens: Optional[List[int]] = None, pattern=None) -> List[List[int]]:
    """Token ids per request: [last committed token, draft 1..K_r].

    ``targets`` are the planted target ids of the packed rows (request r's rows
    follow those of request r-1; request r has K_r+1 rows).  ``pattern``, when
    given, is a per-request list of booleans that fixes hit/miss per draft
    instead of the Bernoulli draw.
    """
    out = []
    row = 0
    for r, K in enumerate(ks):
        u = torch.rand(K + 2, generator=gen_cpu).tolist()
        rr = torch.randint(0, max(vocab - 1, 1), (K + 2,), generator=gen_cpu).tolist()
        uni = torch.randint(0, vocab, (K + 2,), generator=gen_cpu).tolist()
        first = last_tokens[r] if last_tokens is not None else uni[K + 1]
        toks = [int(first)]
        alive = True
        for i in range(1, K + 1):
            tprev = int(targets[row + i - 1])
            hit = (pattern[r][i - 1] if pattern is not None else u[i] < p_accept)
            if alive and hit:
                toks.append(tprev)
            elif alive:
                toks.append((tprev + 1 + rr[i]) % vocab)
                alive = False
            else:
                toks.append(uni[i])
        out.append(toks)
        row += K + 1
    return out


# ---------------------------------------------------------------------------
# Workloads: the five verification/prefill workloads, sized as stated.
# ---------------------------------------------------------------------------

DIMS_TINY = Dims(h_qk=2, h_v=2, d_k=16, d_v=16)
DIMS_FULL = Dims(h_qk=16, h_v=32, d_k=128, d_v=128)
VOCAB_FULL = 151936


@dataclasses.dataclass
class Spec:
    name: str
    dims: Dims
    layers: int
    batch: int
    k_fixed: Optional[int]       # None: K_r ~ U{0..k_max} per step and request
    k_max: int
    steps: int
    vocab: int
    logit_std: float
    p_accept: float
    num_slots: int
    shared_prefix: int           # requests sharing slot of request 0 (copy-on-write)
    ring: int                    # distinct input sets cycled over steps
    seed: int


SPECS = {
    "tiny": Spec("tiny", DIMS_TINY, 1, 1, 3, 3, 1, 64, 1.0, 1.0, 1, 0, 1, 0),
    "batch1": Spec("batch1", DIMS_FULL, 1, 1, 3, 3, 1, VOCAB_FULL, 2.0, 0.85, 1, 0, 1, 1),
    "cb16": Spec("cb16", DIMS_FULL, 30, 16, None, 3, 200, VOCAB_FULL, 2.0, 0.85, 16, 0, 4, 2),
    "paged256": Spec("paged256", DIMS_FULL, 30, 256, 3, 3, 100, VOCAB_FULL, 2.0, 0.85, 1024, 16, 4, 4),
}


def k_table(spec: Spec, steps: Optional[int] = None) -> torch.Tensor:
    """Requested draft count per (step, request), int32 [steps, batch]."""
    steps = spec.steps if steps is None else steps
    if spec.k_fixed is not None:
        return torch.full((steps, spec.batch), spec.k_fixed, dtype=torch.int32)
    gen = generator(mix_seed(spec.seed, 101))
    return torch.randint(0, spec.k_max + 1, (steps, spec.batch), generator=gen, dtype=torch.int32)


def initial_slots(spec: Spec):
    """Slot table (a seeded permutation of the pool) for the workload.

    Returns (slot_of_request [batch] list, free slots in FIFO order, refcounts).
    The first ``shared_prefix`` requests all start on one slot."""
    gen = generator(mix_seed(spec.seed, 202))
    perm = torch.randperm(spec.num_slots, generator=gen).tolist() if spec.num_slots > 1 else [0]
    share = max(spec.shared_prefix, 1)
    slot_of = []
    for r in range(spec.batch):
        slot_of.append(perm[0] if r < share else perm[r - share + 1])
    used = spec.batch - share + 1
    free = perm[used:]
    ref = [0] * spec.num_slots
    for s in slot_of:
        ref[s] += 1
    return slot_of, free, ref


def ring_rows(spec: Spec, layer: int, ring_idx: int, n: int, device="cpu") -> Rows:
    gen = generator(mix_seed(spec.seed, 303, layer, ring_idx), device)
    return rows(gen, n, spec.dims, device)


def ring_logits(spec: Spec, ring_idx: int, n: int, device="cpu"):
    gen = generator(mix_seed(spec.seed, 404, ring_idx), device)
    return logits(gen, n, spec.vocab, spec.logit_std, device)


def step_drafts(spec: Spec, step: int, ks: List[int], targets: List[int]) -> List[List[int]]:
    gen = generator(mix_seed(spec.seed, 505, step))
    pattern = None
    if spec.name == "tiny":
        pattern = [[True, True, False]]
    return drafts(gen, targets, ks, spec.vocab, spec.p_accept, pattern=pattern)


def pool_state(spec: Spec, device="cpu", out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Initial pool [num_slots, layers, h_v, d_v, d_k] fp32, N(0, 0.1^2)."""
    d = spec.dims
    gen = generator(mix_seed(spec.seed, 606), device)
    return state(gen, (spec.num_slots, spec.layers, d.h_v, d.d_v, d.d_k), device, 0.1, out)


# ---------------------------------------------------------------------------
# Chunked-prefill workload: 8 sequences, log-uniform lengths in [512, 32768].
# ---------------------------------------------------------------------------

def prefill_lengths(n: int = 8, lo: int = 512, hi: int = 32768, seed: int = 3) -> List[int]:
    gen = generator(mix_seed(seed, 707))
    u = torch.rand(n, generator=gen, dtype=torch.float64).tolist()
    return [int(round(math.exp(math.log(lo) + x * (math.log(hi) - math.log(lo))))) for x in u]


def prefill_inputs(lengths: List[int], dims: Dims, seed: int = 3, device="cpu"):
    """Packed rows for ragged sequences, cu_seqlens (int32, len n+1) and
    initial states [n, h_v, d_v, d_k]: the first half start from zero, the
    second half from N(0, 0.1^2) (a continued prefix)."""
    total = sum(lengths)
    gen = generator(mix_seed(seed, 808), device)
    r = rows(gen, total, dims, device)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    s0 = torch.zeros((len(lengths), dims.h_v, dims.d_v, dims.d_k), dtype=torch.float32, device=device)
    half = len(lengths) // 2
    if len(lengths) - half:
        s0[half:] = state(generator(mix_seed(seed, 809), device), s0[half:].shape, device, 0.1)
    return r, torch.tensor(cu, dtype=torch.int32), s0
