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
