"""The per-(layer, row) trace (GDNSPEC_TRACE_DIR) of a multi-step decode
loop, compared row by row with the FP64 oracle after the fact: every traced
row's output of every layer within the bf16 bound and every traced
checkpoint within the state bound ("Run chained MTP drafting in the batch
Engine", Validation: layer tracing of every row)."""
import glob
import os

import numpy as np
import pytest
import torch

import gdnsynth as sy
import oracle
from gpu_util import build_lib, noted, out_err, state_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def test_trace_rows_match_oracle(gs, cuda_dev, tmp_path, monkeypatch):
    monkeypatch.setenv("GDNSPEC_TRACE_DIR", str(tmp_path))
    monkeypatch.setenv("GDNSPEC_TRACE_REQS", "2")
    from speculative_decoding_hybrid_gb300.step import DecodeLoop, LayerRows, VerifyStep
    dims = sy.Dims(4, 8, 128, 128)
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    L, B, num_slots, vocab, steps = 2, 4, 8, 1024, 3
    cap = B * 4
    init = sy.state(sy.generator(61), (num_slots, L, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    vs = VerifyStep(d, L, num_slots, cap, B, vocab, cuda_dev, pool=init.clone())
    pool = gs.Pool(num_slots)
    for _ in range(B):
        pool.alloc()
    loop = DecodeLoop(vs, list(range(B)), pool)
    inputs = []
    for s in range(steps):
        p = loop.plan_step([3, 1, 2, 0])
        cu = p.dec_cu
        rows = [sy.rows(sy.generator(800 + 10 * s + l), cu[-1], dims, cuda_dev) for l in range(L)]
        lg, tgt = sy.logits(sy.generator(900 + s), cu[-1], vocab, 2.0, cuda_dev)
        toks = torch.tensor(sum(sy.drafts(sy.generator(950 + s), tgt.tolist(), p.k, vocab, 0.85), []),
                            dtype=torch.int32, device=cuda_dev)
        loop.upload_tables()
        loop.run([LayerRows(r.q, r.k, r.v, r.g, r.beta) for r in rows], lg, toks)
        acc, _, _ = loop.readback()
        loop.finish(acc.clone())
        inputs.append([[t.cpu() for t in (r.q, r.k, r.v, r.g, r.beta)] for r in rows])
    files = sorted(glob.glob(os.path.join(str(tmp_path), "txn_*.npz")))
    assert len(files) == steps
    S = {r: [init[r, l].cpu().numpy().astype(np.float64) for l in range(L)] for r in range(2)}
    checked_rows = 0
    worst_o = worst_s = 0.0
    for s, f in enumerate(files):
        z = np.load(f)
        cu = z["cu_rows"].tolist()
        o = torch.from_numpy(z["o_bf16"].view(np.int16)).view(torch.bfloat16)
        for r in range(2):
            a, b = cu[r], cu[r + 1]
            ck = z["ckpt_req%d" % r]
            for l in range(L):
                q, k, v, g, beta = (t[a:b] for t in inputs[s][l])
                _, o_ref, ck_ref = oracle.gdn_recurrent(q, k, v, g, beta, S[r][l], 1.0, want_ckpt=True)
                for row in range(b - a):               # row by row, as the trace is meant to be read
                    worst_o = max(worst_o, out_err(o[l, a + row], o_ref[row]))
                    worst_s = max(worst_s, state_err(ck[l, row], ck_ref[row]))
                    checked_rows += 1
                S[r][l] = ck_ref[int(z["accept_len"][r])]
    print("trace: %d (layer, row) pairs, worst output %.3f, worst checkpoint %.3f of their bounds" %
          (checked_rows, worst_o, worst_s))
    assert checked_rows == steps * L * (4 + 2)
    assert noted("trace: outputs", worst_o) <= 1.0 and noted("trace: checkpoints", worst_s) <= 1.0
