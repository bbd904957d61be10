"""The mixed-transaction driver: prefill sequences and decode requests of one
planned transaction, for every layer, with the prefills on a side stream.

Checks that the overlapped run writes bit-for-bit what the in-order run
writes (the two halves touch disjoint slots), that every published prefill
state matches the FP64 token-by-token oracle and every decode request
advanced by exactly one token (drafts deferred), and that the next
transaction, queued right after on the caller's stream, reads the published
states."""
import numpy as np
import pytest
import torch

import gdnsynth as sy
import oracle
from gpu_util import build_lib, noted, out_err, state_err

pytestmark = pytest.mark.gpu

CHUNK_STATE_RTOL = 5e-3
DIMS = sy.Dims(4, 8, 128, 128)
L, NUM_SLOTS, VOCAB = 2, 16, 1024
PLENS = [200, 64, 17]


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def _plan(gs):
    pool = gs.Pool(NUM_SLOTS)
    slots = [pool.alloc() for _ in range(4)]           # 0, 1, 2, 3
    pool.share(slots[2])                               # decode requests 2 and 3 share slot 2
    dec = [(gs.REQ_DECODE, 3, 0, 10, 1 << 30, s) for s in (slots[0], slots[1], slots[2], slots[2])]
    pre = [(gs.REQ_PREFILL, 0, PLENS[0], 0, 1 << 30, -1), (gs.REQ_PREFILL, 0, PLENS[1], 0, 1 << 30, -1),
           (gs.REQ_PREFILL, 0, PLENS[2], 40, 1 << 30, slots[3])]   # the last one continues slot 3
    reqs = pre[:2] + dec[:2] + pre[2:] + dec[2:]
    plan = gs.Plan(len(reqs))
    st = gs.plan_transaction(gs.make_reqs(reqs), len(reqs), gs.gdn_plan_limits(4096, 8, 3), pool, plan)
    assert st == gs.GDN_OK
    return pool, plan


def _inputs(dev):
    from speculative_decoding_hybrid_gb300.step import LayerRows
    pre, dec = [], []
    for l in range(L):
        r, cu, _ = sy.prefill_inputs(PLENS, DIMS, seed=60 + l)
        pre.append(LayerRows(*(t.to(dev) for t in (r.q, r.k, r.v, r.g, r.beta))))
        x = sy.rows(sy.generator(80 + l), 4, DIMS, dev)
        dec.append(LayerRows(x.q, x.k, x.v, x.g, x.beta))
    lg, _ = sy.logits(sy.generator(90), 4, VOCAB, 2.0, dev)
    return pre, dec, lg


def _run(gs, dev, plan, init, overlap, pre, dec, lg):
    from speculative_decoding_hybrid_gb300.step import MixedTransaction, VerifyStep
    d = gs.dims(DIMS.h_qk, DIMS.h_v, DIMS.d_k, DIMS.d_v)
    vs = VerifyStep(d, L, NUM_SLOTS, 16, 4, VOCAB, dev, pool=init.clone())
    mt = MixedTransaction(vs, 4, 512, overlap=overlap)
    R = sum(PLENS)
    pre_o = torch.full((L, R, DIMS.h_v, DIMS.d_v), float("nan"), dtype=torch.bfloat16, device=dev)
    mt.upload(plan)
    mt.run(plan, dec, pre, pre_o, lg, torch.zeros(4, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    return vs, pre_o


def test_mixed_transaction_overlapped_equals_in_order(gs, cuda_dev):
    pool, plan = _plan(gs)
    assert plan.deferred == 12 and plan.k == [0] * 7 and plan.plan == gs.PLAN_CHUNKED
    assert plan.c.n_decode == 4 and plan.c.n_prefill == 3
    assert len(set(plan.pre_dst) | set(plan.dec_dst)) == 7           # every writer has its own slot
    init = sy.state(sy.generator(55), (NUM_SLOTS, L, DIMS.h_v, DIMS.d_v, DIMS.d_k)).to(cuda_dev)
    pre, dec, lg = _inputs(cuda_dev)
    a, oa = _run(gs, cuda_dev, plan, init, True, pre, dec, lg)
    b, ob = _run(gs, cuda_dev, plan, init, False, pre, dec, lg)
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert torch.equal(a.pool, b.pool)
    assert torch.equal(oa, ob)
    assert torch.equal(a.o[:, :4], b.o[:, :4])
    assert a.accept_len[:4].tolist() == [0, 0, 0, 0]

    # FP64 oracle: published prefill states and outputs, decode states
    cu = plan.pre_cu
    for l in range(L):
        ph = [t.cpu() for t in (pre[l].q, pre[l].k, pre[l].v, pre[l].g, pre[l].beta)]
        for i in range(3):
            s, e = cu[i], cu[i + 1]
            S0 = np.zeros((DIMS.h_v, 128, 128)) if plan.pre_src[i] < 0 else \
                init[plan.pre_src[i], l].cpu().numpy().astype(np.float64)
            S, o_ref, _ = oracle.gdn_recurrent(*(t[s:e] for t in ph), S0)
            got = a.pool[plan.pre_dst[i], l].cpu().numpy()
            rel = max(np.linalg.norm(got[h] - S[h]) / np.linalg.norm(S[h]) for h in range(DIMS.h_v))
            assert rel <= CHUNK_STATE_RTOL, (l, i, rel)
            assert noted("mixed: prefill outputs", out_err(oa[l, s:e], o_ref)) <= 1.0
        dh = [t.cpu() for t in (dec[l].q, dec[l].k, dec[l].v, dec[l].g, dec[l].beta)]
        for r in range(4):
            S0 = init[plan.dec_src[r], l].cpu().numpy().astype(np.float64)
            S, o_ref, _ = oracle.gdn_recurrent(*(t[r:r + 1] for t in dh), S0)
            assert noted("mixed: decode state", state_err(a.pool[plan.dec_dst[r], l].cpu().numpy(), S)) <= 1.0
            assert noted("mixed: decode outputs", out_err(a.o[l, r:r + 1], o_ref)) <= 1.0
    # slots nobody wrote are untouched
    written = set(plan.pre_dst) | set(plan.dec_dst)
    for s in range(NUM_SLOTS):
        if s not in written:
            assert torch.equal(a.pool[s], init[s])
    assert gs.gdn_pool_apply(pool, plan, 7) == gs.GDN_OK


def test_next_transaction_reads_published_prefill_state(gs, cuda_dev):
    """Queue the mixed transaction and, right after it on the same stream
    with no host synchronisation, verify the prefilled sequences: the verify
    must see the published final states."""
    from speculative_decoding_hybrid_gb300.step import LayerRows, MixedTransaction, VerifyStep
    pool, plan = _plan(gs)
    init = sy.state(sy.generator(56), (NUM_SLOTS, L, DIMS.h_v, DIMS.d_v, DIMS.d_k)).to(cuda_dev)
    pre, dec, lg = _inputs(cuda_dev)
    d = gs.dims(DIMS.h_qk, DIMS.h_v, DIMS.d_k, DIMS.d_v)
    vs = VerifyStep(d, L, NUM_SLOTS, 16, 4, VOCAB, cuda_dev, pool=init.clone())
    mt = MixedTransaction(vs, 4, 512, overlap=True)
    pre_o = torch.empty((L, sum(PLENS), DIMS.h_v, DIMS.d_v), dtype=torch.bfloat16, device=cuda_dev)
    mt.upload(plan)
    nxt = sy.rows(sy.generator(95), 12, DIMS, cuda_dev)                 # 3 sequences x K=3 drafts
    nrows = [LayerRows(nxt.q, nxt.k, nxt.v, nxt.g, nxt.beta)] * L
    cu2 = torch.tensor([0, 4, 8, 12], dtype=torch.int32, device=cuda_dev)
    src2 = torch.tensor(plan.pre_dst, dtype=torch.int32, device=cuda_dev)
    mt.run(plan, dec, pre, pre_o, lg, torch.zeros(4, dtype=torch.int32, device=cuda_dev))
    vs2 = VerifyStep(d, L, NUM_SLOTS, 16, 3, VOCAB, cuda_dev, pool=vs.pool)
    vs2.txn = 9
    vs2.verify_all(3, cu2, src2, nrows)
    torch.cuda.synchronize()
    assert int(vs.status.item()) == 0 and int(vs2.status.item()) == 0
    nh = [t.cpu() for t in (nxt.q, nxt.k, nxt.v, nxt.g, nxt.beta)]
    for l in range(L):
        for i in range(3):
            published = vs.pool[plan.pre_dst[i], l].cpu().numpy().astype(np.float64)
            _, _, ck = oracle.gdn_recurrent(*(t[4 * i:4 * i + 4] for t in nh), published, want_ckpt=True)
            assert noted("mixed: verify after publish", state_err(vs2.ckpt[l, 4 * i:4 * i + 4].cpu().numpy(), ck)) <= 1.0
