"""Compact fixed-state replay (gdn_verify_replay) against the checkpoint path:
same planner decisions, same accepted lengths, emitted tokens and outputs,
and bit-for-bit the same committed states, including a copy-on-write slot."""
import pytest
import torch

import gdnsynth as sy
from gpu_util import build_lib, noted

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def _pool(gs, num_slots):
    p = gs.Pool(num_slots, [5, 0, 3, 7, 1, 2, 4, 6, 8, 9, 10, 11])
    for _ in range(5):
        p.alloc()
    p.share(5)
    return p


def _replay_matches_checkpoints(gs, cuda_dev, dims, k_hi, p_accept, steps, label):
    """Both decode loops over the same steps: draft counts drawn from
    0..k_hi (request 2 always asks for k_hi), draft hits Bernoulli with
    p_accept(step); every step's accepted lengths, tokens and outputs equal,
    the final slots bit-identical, three requests (one of them request 2)
    followed by the oracle."""
    from speculative_decoding_hybrid_gb300.step import DecodeLoop, LayerRows, ReplayStep, VerifyStep
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    L, B, num_slots, vocab = 3, 6, 12, 4096
    cap = B * (k_hi + 1)
    init = sy.state(sy.generator(3), (num_slots, L, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    slots = [5, 5, 0, 3, 7, 1]              # requests 0 and 1 share slot 5
    vs = VerifyStep(d, L, num_slots, cap, B, vocab, cuda_dev, pool=init.clone())
    rs = ReplayStep(d, L, num_slots, cap, B, vocab, cuda_dev, pool=init.clone())
    lc = DecodeLoop(vs, slots, _pool(gs, num_slots), k_max=k_hi)
    lr = DecodeLoop(rs, slots, _pool(gs, num_slots), k_max=k_hi)
    from gpu_util import OracleFollow
    follow = OracleFollow({r: [init[slots[r], l].cpu().numpy() for l in range(L)] for r in (1, 2, 4)})
    kg = sy.generator(4)
    keep = []
    max_replayed = 0
    for s in range(steps):
        ks = torch.randint(0, k_hi + 1, (B,), generator=kg).tolist()
        ks[2] = k_hi
        pc = lc.plan_step(ks)
        pr = lr.plan_step(ks)
        assert pc.dec_cu == pr.dec_cu and pc.dec_src == pr.dec_src and pc.dec_dst == pr.dec_dst
        cu = pc.dec_cu
        R = cu[-1]
        rows = [sy.rows(sy.generator(50 * s + l), R, dims, cuda_dev) for l in range(L)]
        lrows = [LayerRows(r.q, r.k, r.v, r.g, r.beta) for r in rows]
        keep.append(lrows)
        lg, tgt = sy.logits(sy.generator(70 + s), R, vocab, 2.0, cuda_dev)
        toks = torch.tensor(sum(sy.drafts(sy.generator(90 + s), tgt.tolist(), pc.k, vocab, p_accept(s)), []),
                            dtype=torch.int32, device=cuda_dev)
        lc.upload_tables()
        lc.run(lrows, lg, toks)
        ac, bc, oc = (x.clone() for x in lc.readback())
        lr.upload_tables()
        lr.run(lrows, lg, toks)
        ar, br, orr = (x.clone() for x in lr.readback())
        max_replayed = max(max_replayed, int(ar.max()) + 1)  # replayed by the next launch or the flush
        assert int(vs.status.item()) == 0 and int(rs.status.item()) == 0
        assert torch.equal(ac, ar) and torch.equal(bc, br) and torch.equal(oc[:R], orr[:R])
        assert torch.equal(vs.o[:, :R], rs.o[:, :R]), "outputs are computed from bit-identical states"
        # the replay loop's outputs and accept lengths against the FP64 oracle
        follow.step(cu, [[t.cpu() for t in (x.q, x.k, x.v, x.g, x.beta)] for x in rows], lg.cpu(), toks.cpu(),
                    vocab, ar.tolist(), rs.o[:, :R])
        lc.finish(ac)
        lr.finish(ar)
    assert lc.slot == lr.slot
    cur = torch.tensor(lr.slot, dtype=torch.int32, device=cuda_dev)
    rs.flush(cur, cur)
    torch.cuda.synchronize()
    assert int(rs.status.item()) == 0
    for r in range(B):
        assert torch.equal(rs.pool[lr.slot[r]], vs.pool[lc.slot[r]]), r
    # the replayed (committed) states of the followed requests against the oracle
    for r in follow.S:
        follow.check_state(r, [rs.pool[lr.slot[r], l].cpu().numpy() for l in range(L)])
    print("replay vs oracle: worst state %.3f, worst output %.3f of their bounds" %
          (follow.worst_state, follow.worst_out))
    assert noted("fixed-state replay%s: state" % label, follow.worst_state) <= 1.0
    assert noted("fixed-state replay%s: outputs" % label, follow.worst_out) <= 1.0
    # the shared slot was never written by either path
    assert torch.equal(rs.pool[5], init[5]) and torch.equal(vs.pool[5], init[5])
    return max_replayed


def test_replay_loop_matches_checkpoint_loop(gs, cuda_dev):
    _replay_matches_checkpoints(gs, cuda_dev, sy.Dims(4, 8, 128, 128), 3, lambda s: 0.85, 7, "")


@pytest.mark.parametrize("dims", [sy.Dims(4, 8, 128, 128), sy.Dims(2, 4, 64, 64), sy.Dims(2, 4, 32, 32),
                                  sy.Dims(2, 2, 16, 16)], ids=["d128", "d64", "d32", "d16"])
def test_replay_at_the_maximum_draft_count(gs, cuda_dev, dims):
    """K = 15: a request that accepted all 15 drafts replays 16 rows (the most
    one launch takes) before its 16 new rows; every other step draws its hits
    at 0.85, so short and long replays mix."""
    top = _replay_matches_checkpoints(gs, cuda_dev, dims, 15, lambda s: 1.0 if s % 2 == 0 else 0.85, 5,
                                      " K=15 d%d" % dims.d_k)
    assert top == 16, "no step replayed the maximum of 16 rows"


def test_replay_refuses_more_accepted_rows_than_existed(gs, cuda_dev):
    from speculative_decoding_hybrid_gb300.step import LayerRows
    dims = sy.Dims(2, 4, 64, 64)
    d = gs.dims(2, 4, 64, 64)
    pool = sy.state(sy.generator(1), (3, 4, 64, 64)).to(cuda_dev)
    before = pool.clone()
    r = sy.rows(sy.generator(2), 4, dims, cuda_dev)
    cu = torch.tensor([0, 2, 4], dtype=torch.int32, device=cuda_dev)
    prev_cu = torch.tensor([0, 2, 4], dtype=torch.int32, device=cuda_dev)
    prev_acc = torch.tensor([5, 1], dtype=torch.int32, device=cuda_dev)   # request 0 claims 6 of its 2 rows
    slots = torch.tensor([0, 1], dtype=torch.int32, device=cuda_dev)
    o = torch.zeros((4, 4, 64), dtype=torch.bfloat16, device=cuda_dev)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    gs.gdn_verify_replay(d, 2, 4, cu, r.q, r.k, r.v, r.g, r.beta, 4, prev_cu, prev_acc, r.k, r.v, r.g, r.beta,
                         pool, pool.stride(0), 3, slots, slots, o, st)
    torch.cuda.synchronize()
    assert int(st.item()) & gs.DEV_ROWS_BAD
    assert torch.equal(pool[0], before[0])            # refused: slot untouched
    assert not torch.equal(pool[1], before[1])        # request 1 replayed its 2 rows


@pytest.mark.parametrize("ring", [4, 3])
def test_replay_graphs_match_eager_transactions(gs, cuda_dev, ring):
    """One CUDA graph per transaction residue (input set and accept-buffer
    parity) replays a whole transaction (30 verify launches in the paged
    workload, 2 here) with identical results; an odd number of input sets
    takes twice as many graphs."""
    from speculative_decoding_hybrid_gb300.step import DecodeLoop, LayerRows, ReplayGraphs, ReplayStep
    dims = sy.Dims(4, 8, 128, 128)
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    L, B, num_slots, vocab, steps = 2, 5, 8, 2048, 9
    cap = B * 4
    init = sy.state(sy.generator(8), (num_slots, L, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    slots = [0, 1, 2, 3, 4]
    mk = lambda: gs.Pool(num_slots)
    pools = []
    for _ in range(2):
        p = mk()
        for _ in range(5):
            p.alloc()
        pools.append(p)
    eager = ReplayStep(d, L, num_slots, cap, B, vocab, cuda_dev, pool=init.clone())
    graph = ReplayStep(d, L, num_slots, cap, B, vocab, cuda_dev, pool=init.clone())
    le, lg_ = DecodeLoop(eager, slots, pools[0]), DecodeLoop(graph, slots, pools[1])
    rows = [[LayerRows(*(t for t in (r.q, r.k, r.v, r.g, r.beta)))
             for r in (sy.rows(sy.generator(100 * i + l), cap, dims, cuda_dev) for l in range(L))] for i in range(ring)]
    logits = [sy.logits(sy.generator(200 + i), cap, vocab, 2.0, cuda_dev) for i in range(ring)]
    tok_e = torch.zeros(cap, dtype=torch.int32, device=cuda_dev)
    tok_g = torch.zeros(cap, dtype=torch.int32, device=cuda_dev)
    lg_.plan_step([3] * B)          # the tables the graphs read exist before capture
    lg_.upload_tables()
    graphs = ReplayGraphs(graph, lg_, rows, [x[0] for x in logits], tok_g)
    assert len(graphs.graphs) == (ring if ring % 2 == 0 else 2 * ring)
    # restart the graph loop's planner state (the capture executed nothing)
    lg_.pool = pools[1] = mk()
    for _ in range(5):
        lg_.pool.alloc()
    lg_.req_np[:B, 3] = 1
    from gpu_util import OracleFollow
    follow = OracleFollow({r: [init[slots[r], l].cpu().numpy() for l in range(L)] for r in (0, 3)})
    rows_host = [[[t.cpu() for t in (x.q, x.k, x.v, x.g, x.beta)] for x in rr] for rr in rows]
    for s in range(steps):
        i = s % ring
        ks = [3, 2, 3, 1, 3]
        pe, pg = le.plan_step(ks), lg_.plan_step(ks)
        assert pe.dec_cu == pg.dec_cu
        tk = sum(sy.drafts(sy.generator(300 + s), logits[i][1].tolist(), ks, vocab, 0.85), [])
        tk = torch.tensor(tk + [0] * (cap - len(tk)), dtype=torch.int32)
        tok_e.copy_(tk)
        tok_g.copy_(tk)
        le.upload_tables()
        eager.run(B, le.cu_rows, le.src_slot, le.dst_slot, rows[i], logits[i][0], tok_e)
        ae = le.readback()[0].clone()
        lg_.upload_tables()
        graphs.launch(s, rows)
        ag = lg_.readback()[0].clone()
        assert torch.equal(ae, ag), s
        R = pe.dec_cu[-1]
        assert torch.equal(eager.o[:, :R], graph.o[:, :R]), s
        follow.step(pe.dec_cu, rows_host[i], logits[i][0].cpu(), tk, vocab, ag.tolist(), graph.o[:, :R])
        le.finish(ae)
        lg_.finish(ag)
    cur = torch.tensor(le.slot, dtype=torch.int32, device=cuda_dev)
    eager.flush(cur, cur)
    graph.flush(cur, cur)
    torch.cuda.synchronize()
    assert int(eager.status.item()) == 0 and int(graph.status.item()) == 0
    assert torch.equal(eager.pool, graph.pool)
    for r in follow.S:
        follow.check_state(r, [graph.pool[lg_.slot[r], l].cpu().numpy() for l in range(L)])
    assert noted("replay graphs: state", follow.worst_state) <= 1.0, follow.worst_state
    assert noted("replay graphs: outputs", follow.worst_out) <= 1.0, follow.worst_out
