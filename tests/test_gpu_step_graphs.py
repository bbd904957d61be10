"""CUDA graphs of the checkpointing transaction (every layer's gdn_verify,
mtp_greedy_accept, gdn_commit -- or gdn_verify_at / gdn_commit_at over a
state arena), replayed one launch per step: the same accept lengths, emitted
tokens, outputs and committed states as the eagerly launched transactions,
and both held to the FP64 oracle for the followed requests ("Run chained MTP
drafting in the batch Engine", H200 RC4 evidence: graph capture of the
hybrid fixed-state step)."""
import numpy as np
import pytest
import torch

import gdnsynth as sy
from gpu_util import OracleFollow, build_lib, noted

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def _state_of(vs, loop, r, arena):
    """[layers][h_v, d_v, d_k] of request r as the loop holds it."""
    if arena:
        return [vs.arena[int(vs.loc[l, r]):int(vs.loc[l, r]) + vs.S].view(vs.d.h_v, vs.d.d_v, vs.d.d_k).cpu().numpy()
                for l in range(vs.L)]
    return [vs.pool[loop.slot[r], l].cpu().numpy() for l in range(vs.L)]


@pytest.mark.parametrize("arena", [False, True])
def test_step_graphs_match_eager_and_oracle(gs, cuda_dev, arena):
    from speculative_decoding_hybrid_gb300.step import ArenaStep, DecodeLoop, LayerRows, StepGraphs, VerifyStep
    dims = sy.Dims(4, 8, 128, 128)
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    L, B, num_slots, vocab, steps, ring = 2, 5, 12, 2048, 8, 3
    cap = B * 4
    init = sy.state(sy.generator(21), (num_slots, L, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    slots = [0, 0, 1, 2, 3]                                # requests 0 and 1 share a slot
    runs = []
    for _ in range(2):
        if arena:
            vs = ArenaStep(d, L, num_slots, cap, B, vocab, cuda_dev)
            vs.pool.copy_(init)
            vs.point_at_slots(slots)
        else:
            vs = VerifyStep(d, L, num_slots, cap, B, vocab, cuda_dev, pool=init.clone())
        pool = gs.Pool(num_slots)
        for _ in range(4):
            pool.alloc()
        pool.share(0)
        runs.append((vs, DecodeLoop(vs, slots, pool)))
    (ve, le), (vg, lg) = runs
    rows = [[LayerRows(*(t for t in (x.q, x.k, x.v, x.g, x.beta)))
             for x in (sy.rows(sy.generator(500 + 10 * i + l), cap, dims, cuda_dev) for l in range(L))]
            for i in range(ring)]
    rows_host = [[[t.cpu() for t in (x.q, x.k, x.v, x.g, x.beta)] for x in rr] for rr in rows]
    logits = [sy.logits(sy.generator(600 + i), cap, vocab, 2.0, cuda_dev) for i in range(ring)]
    tok_e = torch.zeros(cap, dtype=torch.int32, device=cuda_dev)
    tok_g = torch.zeros(cap, dtype=torch.int32, device=cuda_dev)
    lg.plan_step([3] * B)                                  # tables exist before the capture
    lg.upload_tables()
    graphs = StepGraphs(vg, lg, rows, [x[0] for x in logits], tok_g)
    assert len(graphs.graphs) == (2 * ring if arena else ring)
    # the capture executed nothing: restart the graph loop's planner state
    pool = gs.Pool(num_slots)
    for _ in range(4):
        pool.alloc()
    pool.share(0)
    lg.pool = pool
    lg.req_np[:B, 3] = 1
    follow = OracleFollow({r: [init[slots[r], l].cpu().numpy() for l in range(L)] for r in (1, 3)})
    kg = sy.generator(7)
    for s in range(steps):
        i = s % ring
        ks = torch.randint(0, 4, (B,), generator=kg).tolist()
        pe, pg = le.plan_step(ks), lg.plan_step(ks)
        assert pe.dec_cu == pg.dec_cu and pe.dec_dst == pg.dec_dst
        cu = pe.dec_cu
        tk = sum(sy.drafts(sy.generator(700 + s), logits[i][1].tolist(), pe.k, vocab, 0.85), [])
        tk = torch.tensor(tk + [0] * (cap - len(tk)), dtype=torch.int32)
        tok_e.copy_(tk)
        tok_g.copy_(tk)
        le.upload_tables()
        if arena:
            ve.run(B, le.cu_rows, rows[i], logits[i][0], tok_e)
        else:
            ve.run(B, le.cu_rows, le.src_slot, le.dst_slot, rows[i], logits[i][0], tok_e)
        ae = le.readback()[0].clone()
        lg.upload_tables()
        graphs.launch(s)
        ag = lg.readback()[0].clone()
        R = cu[-1]
        assert int(ve.status.item()) == 0 and int(vg.status.item()) == 0
        assert torch.equal(ae, ag), s
        assert torch.equal(ve.out_tokens[:R], vg.out_tokens[:R]) and torch.equal(ve.o[:, :R], vg.o[:, :R]), s
        follow.step(cu, rows_host[i], logits[i][0].cpu(), tk, vocab, ag.tolist(), vg.o[:, :R])
        le.finish(ae)
        lg.finish(ag)
        for r in follow.S:
            assert all(np.array_equal(x, y) for x, y in zip(_state_of(ve, le, r, arena), _state_of(vg, lg, r, arena)))
            follow.check_state(r, _state_of(vg, lg, r, arena))
    assert le.slot == lg.slot
    print("step graphs (%s): worst state %.3f, worst output %.3f of their bounds" %
          ("arena" if arena else "copy", follow.worst_state, follow.worst_out))
    mode = "arena" if arena else "copy"
    assert noted("step graphs (%s): state" % mode, follow.worst_state) <= 1.0
    assert noted("step graphs (%s): outputs" % mode, follow.worst_out) <= 1.0
