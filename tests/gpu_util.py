"""Helpers shared by the GPU parity tests: tolerances and oracle glue."""
import numpy as np
import torch

import oracle

# Tolerances (written from the arithmetic; see the parity section of the design notes):
#   FP32 state: |x - y| <= 1e-4 * max(|y|, 1e-2 * max|y over the head|)
#   bf16 output vs the unrounded FP64 value: |o - y| <= max(2e-3, (2^-8 + 1e-4) |y|)
#   (bf16 rounding of an FP32 value is within half an ulp, at most 2^-8 of
#   it; the FP32 value itself may sit 1e-4 relative from y, the FP32 budget)
STATE_RTOL = 1e-4
STATE_FLOOR = 1e-2
OUT_ATOL = 2e-3
OUT_RREL = 2.0 ** -8 + 1e-4


# Worst ratio of error to bound seen per check in this session (printed in
# the terminal summary by conftest.py, so that drift toward a bound shows
# even in a passing run).
WORST = {}


def noted(name, ratio):
    """Records ratio (error / allowed, <= 1 passes) under name; returns it."""
    r = float(ratio)
    if r > WORST.get(name, -1.0):
        WORST[name] = r
    return r


def state_err(gpu, ref):
    """Worst ratio err/allowed over a [..., h_v, d_v, d_k] state (<= 1 passes)."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    head_max = np.max(np.abs(r), axis=(-1, -2), keepdims=True)
    scale = np.maximum(np.abs(r), STATE_FLOOR * head_max)
    scale = np.where(scale == 0, 1e-30, scale)
    return float(np.max(np.abs(g - r) / (STATE_RTOL * scale))) if g.size else 0.0


def out_err(gpu_bf16, ref):
    g = gpu_bf16.detach().to("cpu").to(torch.float64).numpy() if hasattr(gpu_bf16, "detach") else gpu_bf16
    r = np.asarray(ref, dtype=np.float64)
    allowed = np.maximum(OUT_ATOL, OUT_RREL * np.abs(r))
    return float(np.max(np.abs(g - r) / allowed)) if g.size else 0.0


def build_lib():
    from speculative_decoding_hybrid_gb300 import build
    build.build()


def rows_to_host(rows):
    return [t.detach().to("cpu") for t in (rows.q, rows.k, rows.v, rows.g, rows.beta)]


def oracle_request(rows_host, a, b, S0, q_scale=1.0):
    q, k, v, g, beta = rows_host
    return oracle.gdn_recurrent(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], S0, q_scale, want_ckpt=True)


class OracleFollow:
    """FP64 oracle states of a few requests of a multi-layer loop, advanced
    transaction by transaction beside the GPU: every layer's rows of a
    followed request run through the oracle recurrence from its state, the
    outputs are held to the bf16 bound, the accept length is the oracle's own
    greedy acceptance (checked equal to the GPU's), and the state moves to the
    accepted checkpoint.  ``states[r]`` is [layers][h_v, d_v, d_k]."""

    def __init__(self, init_states):
        self.S = {r: [np.asarray(x, dtype=np.float64) for x in st] for r, st in init_states.items()}
        self.worst_out = 0.0
        self.worst_state = 0.0

    def step(self, cu, rows_host, logits, tokens, vocab, gpu_accept, o_gpu):
        """cu: packed row offsets (list); rows_host: per layer (q, k, v, g, beta)
        CPU tensors of the packed rows; logits, tokens: the transaction's;
        gpu_accept: the GPU's accept lengths; o_gpu: [layers, rows, h_v, d_v]."""
        am = oracle.argmax_bf16(oracle.bf16_bits(logits[:cu[-1]]), vocab)
        res = oracle.greedy_accept(am, np.asarray(tokens[:cu[-1]].cpu(), dtype=np.int32), np.asarray(cu), vocab)
        assert [int(x) for x in res.accept_len] == [int(x) for x in gpu_accept[:len(cu) - 1]]
        o_cpu = o_gpu.detach().to("cpu")
        for r in self.S:
            a, b = cu[r], cu[r + 1]
            j = int(res.accept_len[r])
            for l, rh in enumerate(rows_host):
                q, k, v, g, beta = (t[a:b] for t in rh)
                _, o_ref, ck = oracle.gdn_recurrent(q, k, v, g, beta, self.S[r][l], 1.0, want_ckpt=True)
                self.worst_out = max(self.worst_out, out_err(o_cpu[l, a:b], o_ref))
                self.S[r][l] = ck[j]

    def check_state(self, r, gpu_layers):
        """gpu_layers: [layers][h_v, d_v, d_k] of request r on the GPU."""
        for l, x in enumerate(gpu_layers):
            self.worst_state = max(self.worst_state, state_err(np.asarray(x), self.S[r][l]))
        return self.worst_state
