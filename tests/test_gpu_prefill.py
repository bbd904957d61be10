"""GPU parity of gdn_chunked_prefill against the FP64 token-by-token oracle,
and the mixed prefill + draft transaction (deferral, publication order)."""
import numpy as np
import pytest
import torch

import gdnsynth as sy
import oracle
from gpu_util import build_lib, noted, out_err, state_err

pytestmark = pytest.mark.gpu

CHUNK_STATE_RTOL = 5e-3   # ||S_chunk - S_rec||_F / ||S_rec||_F per (sequence, head)


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def run_prefill(gs, dev, dims, lengths, src, dst, pool, seed=3, cap=None, shape_rows=None):
    rows, cu, s0 = sy.prefill_inputs(lengths, dims, seed=seed)
    if shape_rows is not None:
        rows = shape_rows(rows)
    R = int(cu[-1])
    cap = R if cap is None else cap
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    ws_bytes = gs.gdn_prefill_workspace_bytes(d, len(lengths), cap)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    # rows R .. cap-1 (capacity no sequence uses) hold NaN
    pad = lambda x: torch.cat([x, torch.full((cap - R,) + tuple(x.shape[1:]), float("nan"), dtype=x.dtype)])
    r = sy.Rows(pad(rows.q), pad(rows.k), pad(rows.v), pad(rows.g), pad(rows.beta)).to(dev)
    o = torch.full((max(cap, 1), dims.h_v, dims.d_v), float("nan"), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_d = cu.to(dev)
    gs.gdn_chunked_prefill(d, len(lengths), cap, cu_d, max(lengths) if lengths else 0, r.q, r.k, r.v, r.g, r.beta,
                           pool, pool.stride(0), pool.shape[0], torch.tensor(src, dtype=torch.int32, device=dev),
                           torch.tensor(dst, dtype=torch.int32, device=dev), o, 64, ws, ws_bytes, st)
    torch.cuda.synchronize()
    return rows, cu, o, int(st.item())


def check_sequences(rows, cu, o, S0s, finals, lengths):
    worst_s, worst_o = 0.0, 0.0
    units = []
    for i, L in enumerate(lengths):
        a, b = int(cu[i]), int(cu[i + 1])
        units += oracle.head_units(rows.q[a:b], rows.k[a:b], rows.v[a:b], rows.g[a:b], rows.beta[a:b], S0s[i])
    H = rows.v.shape[1]
    S, o_list, _ = oracle.recurrent_units(units)
    o_cpu = o.cpu()
    for i, L in enumerate(lengths):
        a, b = int(cu[i]), int(cu[i + 1])
        ref = S[i * H:(i + 1) * H]
        got = finals[i].astype(np.float64)
        for h in range(H):
            rel = np.linalg.norm(got[h] - ref[h]) / max(np.linalg.norm(ref[h]), 1e-30)
            worst_s = max(worst_s, rel)
        if L:
            o_ref = np.stack(o_list[i * H:(i + 1) * H], axis=1)
            worst_o = max(worst_o, out_err(o_cpu[a:b], o_ref))
    return worst_s, worst_o


@pytest.mark.parametrize("lengths", [[1, 63, 64, 200], [129], [0, 5, 64, 65]])
def test_prefill_small_ragged(gs, cuda_dev, lengths):
    dims = sy.Dims(2, 4, 128, 128)
    n = len(lengths)
    pool = sy.state(sy.generator(1), (2 * n + 1, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    init = pool.clone()
    src = [(-1 if i % 2 == 0 else i) for i in range(n)]
    dst = [n + i for i in range(n)]
    dst[-1] = src[-1] if src[-1] >= 0 else dst[-1]            # one in-place publish
    rows, cu, o, st = run_prefill(gs, cuda_dev, dims, lengths, src, dst, pool)
    assert st == 0
    S0s = [np.zeros((dims.h_v, 128, 128)) if s < 0 else init[s].cpu().numpy() for s in src]
    finals = [pool[d].cpu().numpy() for d in dst]
    ws, wo = check_sequences(rows, cu, o, S0s, finals, lengths)
    assert noted("prefill small_ragged: state (rel. Frobenius / 5e-3)", ws / CHUNK_STATE_RTOL) <= 1.0, ws
    assert noted("prefill small_ragged: outputs", wo) <= 1.0, wo
    for s in range(2 * n + 1):
        if s not in dst:
            assert torch.equal(pool[s], init[s]), "only destination slots are written"


@pytest.mark.parametrize("h_qk,h_v", [(4, 4), (1, 4), (2, 8)], ids=["grp1", "grp4", "grp4b"])
def test_prefill_head_grouping(gs, cuda_dev, h_qk, h_v):
    """Every v-head reads the q/k head h_v // h_qk of its group (no grouping,
    four v-heads per q/k head), with the start states of half the sequences
    taken from slots."""
    dims = sy.Dims(h_qk, h_v, 128, 128)
    lengths = [97, 64, 3]
    n = len(lengths)
    pool = sy.state(sy.generator(13), (2 * n, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    init = pool.clone()
    src = [-1, 1, 2]
    dst = [n + i for i in range(n)]
    rows, cu, o, st = run_prefill(gs, cuda_dev, dims, lengths, src, dst, pool, seed=17)
    assert st == 0
    S0s = [np.zeros((dims.h_v, 128, 128)) if x < 0 else init[x].cpu().numpy() for x in src]
    ws, wo = check_sequences(rows, cu, o, S0s, [pool[d].cpu().numpy() for d in dst], lengths)
    assert noted("prefill head_grouping: state (rel. Frobenius / 5e-3)", ws / CHUNK_STATE_RTOL) <= 1.0, ws
    assert noted("prefill head_grouping: outputs", wo) <= 1.0, wo


def _strong_decay(r):
    return sy.Rows(r.q, r.k, r.v, torch.full_like(r.g, -20.0), r.beta)


def _repeated_keys_no_decay(r):
    # runs of 8 tokens share one (already unit-norm, bf16) key; g = 0, beta = 1:
    # the in-chunk matrix A has its largest entries and T = (I + A)^{-1} its
    # largest cancellations
    k = r.k.clone()
    for t in range(0, k.shape[0], 8):
        k[t:t + 8] = k[t]
    return sy.Rows(r.q, k, r.v, torch.zeros_like(r.g), torch.ones_like(r.beta))


def _tiny_beta(r):
    return sy.Rows(r.q, r.k, r.v, r.g, torch.full_like(r.beta, 1e-6))


@pytest.mark.parametrize("d", [128, 32])
@pytest.mark.parametrize("shape", [_strong_decay, _repeated_keys_no_decay, _tiny_beta],
                         ids=["strong_decay", "repeated_keys_no_decay", "tiny_beta"])
def test_prefill_extreme_gates(gs, cuda_dev, shape, d):
    """Gates and keys at the edges of their ranges, against the FP64
    recurrence: g = -20 on every token (the in-chunk exponentials underflow
    to zero), g = 0 and beta = 1 with keys repeated in runs of 8, and
    beta = 1e-6; start states from zero and from slots; on the tensor-core
    kernel (d = 128) and the fp32 one (d = 32)."""
    dims = sy.Dims(2, 4, d, d)
    lengths = [130, 64, 7]
    n = len(lengths)
    pool = sy.state(sy.generator(23), (2 * n, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    init = pool.clone()
    src = [-1, 1, 2]
    dst = [n + i for i in range(n)]
    rows, cu, o, st = run_prefill(gs, cuda_dev, dims, lengths, src, dst, pool, seed=29, shape_rows=shape)
    assert st == 0
    S0s = [np.zeros((dims.h_v, d, d)) if x < 0 else init[x].cpu().numpy() for x in src]
    finals = [pool[j].cpu().numpy() for j in dst]
    assert all(np.isfinite(f).all() for f in finals)
    ws, wo = check_sequences(rows, cu, o, S0s, finals, lengths)
    name = "%s d=%d" % (shape.__name__.strip("_"), d)
    assert noted("prefill extreme %s: state (rel. Frobenius / 5e-3)" % name, ws / CHUNK_STATE_RTOL) <= 1.0, ws
    assert noted("prefill extreme %s: outputs" % name, wo) <= 1.0, wo


def test_prefill_unused_rows_do_not_leak(gs, cuda_dev):
    """Capacity past the last sequence holds NaN in q, k, v, g and beta; the
    last chunk's 64-row window reaches into it, and nothing of it may reach
    the outputs or the published states."""
    dims = sy.Dims(2, 4, 128, 128)
    lengths = [70, 5]
    n = len(lengths)
    pool = torch.zeros((2 * n, dims.h_v, dims.d_v, dims.d_k), dtype=torch.float32, device=cuda_dev)
    rows, cu, o, st = run_prefill(gs, cuda_dev, dims, lengths, [-1] * n, [n + i for i in range(n)], pool,
                                  cap=sum(lengths) + 100)
    assert st == 0
    finals = [pool[n + i].cpu().numpy() for i in range(n)]
    assert all(np.isfinite(f).all() for f in finals)
    ws, wo = check_sequences(rows, cu, o, [np.zeros((dims.h_v, 128, 128))] * n, finals, lengths)
    assert noted("prefill unused_rows_do_not_leak: state (rel. Frobenius / 5e-3)", ws / CHUNK_STATE_RTOL) <= 1.0, ws
    assert noted("prefill unused_rows_do_not_leak: outputs", wo) <= 1.0, wo


def test_prefill_workload_full_size(gs, cuda_dev):
    """Eight sequences, log-uniform lengths in [512, 32768], 32 v-heads, d=128,
    chunk 64; the first four start from zero, the last four from a state."""
    dims = sy.DIMS_FULL
    lengths = sy.prefill_lengths()
    n = len(lengths)
    rows, cu, s0 = sy.prefill_inputs(lengths, dims, seed=3)
    pool = torch.zeros((2 * n, dims.h_v, dims.d_v, dims.d_k), dtype=torch.float32, device=cuda_dev)
    pool[:n] = s0.to(cuda_dev)
    src = [-1] * (n // 2) + list(range(n // 2, n))
    dst = list(range(n, 2 * n))
    rows2, cu2, o, st = run_prefill(gs, cuda_dev, dims, lengths, src, dst, pool)
    assert st == 0
    finals = [pool[d].cpu().numpy() for d in dst]
    ws, wo = check_sequences(rows, cu, o, [s0[i].numpy() for i in range(n)], finals, lengths)
    print("prefill full size: worst state rel %.3e, worst output ratio %.3f" % (ws, wo))
    assert noted("prefill workload_full_size: state (rel. Frobenius / 5e-3)", ws / CHUNK_STATE_RTOL) <= 1.0, ws
    assert noted("prefill workload_full_size: outputs", wo) <= 1.0, wo


def test_mixed_transaction_defers_then_resumes(gs, cuda_dev):
    """Four prefills and four decode requests asking for K=3 share a
    transaction: the planner defers every draft (12 rows), decode requests
    advance by one token, prefills publish their final state; the next,
    decode-only transaction resumes K=3 and reads the published state."""
    from speculative_decoding_hybrid_gb300.step import LayerRows, VerifyStep
    dims = sy.DIMS_FULL
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    num_slots = 12
    pool_c = gs.Pool(num_slots)
    dec_slots = [pool_c.alloc() for _ in range(4)]
    init = sy.state(sy.generator(77), (num_slots, 1, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    vs = VerifyStep(d, 1, num_slots, 64, 8, 1024, cuda_dev, pool=init.clone())
    plens = [300, 64, 129, 17]
    reqs = [(gs.REQ_PREFILL, 0, L, 0, 1 << 30, -1) for L in plens] + \
           [(gs.REQ_DECODE, 3, 0, 10, 1 << 30, s) for s in dec_slots]
    plan = gs.Plan(8)
    st = gs.plan_transaction(gs.make_reqs(reqs), 8, gs.gdn_plan_limits(4096, 8, 3), pool_c, plan)
    assert st == gs.GDN_OK and plan.deferred == 12 and plan.plan == gs.PLAN_CHUNKED
    assert plan.k == [0] * 8 and plan.dec_cu == [0, 1, 2, 3, 4] and plan.pre_cu == [0, 300, 364, 493, 510]
    # oracle planner agrees
    mp = oracle.PoolModel(num_slots)
    for _ in range(4):
        mp.alloc()
    pm = oracle.plan_transaction([oracle.Req(oracle.PREFILL, n_tokens=L) for L in plens] +
                                 [oracle.Req(oracle.DECODE, 3, cur_len=10, slot=s) for s in dec_slots],
                                 4096, 8, 3, mp)
    assert pm.deferred == 12 and pm.dst == plan.dst and pm.dec_cu == plan.dec_cu
    # prefills: chunked, publishing only the final state into their fresh slots
    pr, pcu, ps0 = sy.prefill_inputs(plens, dims, seed=12)
    R = int(pcu[-1])
    pool_l = vs.pool[:, 0]
    ws_bytes = gs.gdn_prefill_workspace_bytes(d, 4, R)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda_dev)
    o = torch.empty((R, dims.h_v, dims.d_v), dtype=torch.bfloat16, device=cuda_dev)
    prd = pr.to(cuda_dev)
    stat = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    gs.gdn_chunked_prefill(d, 4, R, pcu.to(cuda_dev), max(plens), prd.q, prd.k, prd.v, prd.g, prd.beta, pool_l,
                           vs.slot_stride, num_slots, torch.tensor(plan.pre_src, dtype=torch.int32, device=cuda_dev),
                           torch.tensor(plan.pre_dst, dtype=torch.int32, device=cuda_dev), o, 64, ws, ws_bytes, stat)
    # decode requests: one token each (K = 0), verify + accept + commit
    dr = sy.rows(sy.generator(13), 4, dims, cuda_dev)
    cu = torch.tensor(plan.dec_cu, dtype=torch.int32, device=cuda_dev)
    srcs = torch.tensor(plan.dec_src, dtype=torch.int32, device=cuda_dev)
    dsts = torch.tensor(plan.dec_dst, dtype=torch.int32, device=cuda_dev)
    lg, tgt = sy.logits(sy.generator(14), 4, 1024, 2.0, cuda_dev)
    vs.run(4, cu, srcs, dsts, [LayerRows(dr.q, dr.k, dr.v, dr.g, dr.beta)], lg,
           torch.zeros(4, dtype=torch.int32, device=cuda_dev))
    torch.cuda.synchronize()
    assert int(stat.item()) == 0 and int(vs.status.item()) == 0
    assert vs.accept_len[:4].tolist() == [0, 0, 0, 0]                 # one token each, no drafts
    # oracle: prefill final states and decode steps
    for i in range(4):
        a, b = int(pcu[i]), int(pcu[i + 1])
        S, _, _ = oracle.gdn_recurrent(pr.q[a:b], pr.k[a:b], pr.v[a:b], pr.g[a:b], pr.beta[a:b],
                                       np.zeros((dims.h_v, 128, 128)))
        got = vs.pool[plan.pre_dst[i], 0].cpu().numpy()
        rel = max(np.linalg.norm(got[h] - S[h]) / np.linalg.norm(S[h]) for h in range(dims.h_v))
        assert rel <= CHUNK_STATE_RTOL
    drh = dr.to("cpu")
    for i, s in enumerate(dec_slots):
        S, _, _ = oracle.gdn_recurrent(drh.q[i:i + 1], drh.k[i:i + 1], drh.v[i:i + 1], drh.g[i:i + 1],
                                       drh.beta[i:i + 1], init[s, 0].cpu().numpy())
        assert noted("mixed transaction: decode state", state_err(vs.pool[plan.dec_dst[i], 0].cpu().numpy(), S)) <= 1.0
    assert gs.gdn_pool_apply(pool_c, plan, 8) == gs.GDN_OK
    # next transaction: decode-only (the four prefilled sequences now decode too) -> K = 3 again
    slots2 = plan.dst
    reqs2 = [(gs.REQ_DECODE, 3, 0, 400, 1 << 30, s) for s in slots2]
    plan2 = gs.Plan(8)
    assert gs.plan_transaction(gs.make_reqs(reqs2), 8, gs.gdn_plan_limits(4096, 8, 3), pool_c, plan2) == gs.GDN_OK
    assert plan2.k == [3] * 8 and plan2.deferred == 0 and plan2.plan == gs.PLAN_RECURRENT
    published = vs.pool[plan.pre_dst[0], 0].clone()
    r2 = sy.rows(sy.generator(15), 32, dims, cuda_dev)
    cu2 = torch.tensor(plan2.dec_cu, dtype=torch.int32, device=cuda_dev)
    src2 = torch.tensor(plan2.dec_src, dtype=torch.int32, device=cuda_dev)
    vs2 = VerifyStep(d, 1, num_slots, 32, 8, 1024, cuda_dev, pool=vs.pool)
    vs2.txn = 5
    vs2.verify_layer(0, 8, cu2, src2, LayerRows(r2.q, r2.k, r2.v, r2.g, r2.beta))
    torch.cuda.synchronize()
    r2h = r2.to("cpu")
    S, o_ref, ck = oracle.gdn_recurrent(r2h.q[0:4], r2h.k[0:4], r2h.v[0:4], r2h.g[0:4], r2h.beta[0:4],
                                        published.cpu().numpy(), want_ckpt=True)
    assert noted("mixed transaction: verify after publish", state_err(vs2.ckpt[0, 0:4].cpu().numpy(), ck)) <= 1.0       # verify read the published state


def test_prefill_fail_closed(gs, cuda_dev):
    dims = sy.Dims(2, 4, 128, 128)
    pool = torch.zeros((4, 4, 128, 128), device=cuda_dev)
    d = gs.dims(2, 4, 128, 128)
    z = torch.zeros(64, dtype=torch.int32, device=cuda_dev)
    with pytest.raises(gs.GdnError) as e:          # chunk length other than 64
        gs.gdn_chunked_prefill(d, 1, 8, z, 8, pool, pool, pool, pool, pool, pool, pool.stride(0), 4, z, z, pool,
                               32, pool, 1 << 20, z)
    assert e.value.status == gs.GDN_ERR_ARG
    with pytest.raises(gs.GdnError) as e:          # workspace too small (it holds nseq int32)
        gs.gdn_chunked_prefill(d, 1, 8, z, 8, pool, pool, pool, pool, pool, pool, pool.stride(0), 4, z, z, pool,
                               64, pool, 2, z)
    assert e.value.status == gs.GDN_ERR_WORKSPACE
    # a destination slot outside the pool is refused on the device, nothing written
    rows, cu, o, st = run_prefill(gs, cuda_dev, dims, [70], [-1], [9], pool)
    assert st & gs.DEV_SLOT_OOR
    assert torch.count_nonzero(pool) == 0


def test_prefill_timed_out_wait_publishes_nothing(gs, cuda_dev):
    """A bounded wait that runs out makes the prefill refuse to publish
    ([ENGINE] Correctness fix: never publish a state that was not computed in
    full).  The self-test entry point withholds the tensor copy of every
    sequence's last chunk, so the wait for it gives up after 2 ms: the status
    word carries GDN_DEV_TIMEOUT and every destination slot keeps its bytes.
    A normal call made afterwards with that bit still set publishes nothing
    either; once the bit is cleared the same call publishes."""
    dims = sy.Dims(2, 4, 128, 128)
    lengths = [40, 130, 64]
    n = len(lengths)
    rows, cu, s0 = sy.prefill_inputs(lengths, dims, seed=5)
    R = int(cu[-1])
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    pool = sy.state(sy.generator(9), (2 * n, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    init = pool.clone()
    r = rows.to(cuda_dev)
    ws_bytes = gs.gdn_prefill_workspace_bytes(d, n, R)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=cuda_dev)
    o = torch.zeros((R, dims.h_v, dims.d_v), dtype=torch.bfloat16, device=cuda_dev)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    cu_d = cu.to(cuda_dev)
    src = torch.tensor([-1, 1, 2], dtype=torch.int32, device=cuda_dev)
    dst = torch.tensor([3, 4, 5], dtype=torch.int32, device=cuda_dev)
    gs.gdn_selftest_prefill_timeout(d, n, R, cu_d, r.q, r.k, r.v, r.g, r.beta, pool, pool.stride(0), pool.shape[0],
                                    src, dst, o, ws, ws_bytes, st, 2_000_000)
    torch.cuda.synchronize()
    assert int(st.item()) & gs.DEV_TIMEOUT
    assert torch.equal(pool, init)
    gs.gdn_chunked_prefill(d, n, R, cu_d, max(lengths), r.q, r.k, r.v, r.g, r.beta, pool, pool.stride(0),
                           pool.shape[0], src, dst, o, 64, ws, ws_bytes, st)
    torch.cuda.synchronize()
    assert torch.equal(pool, init), "a call made while the timeout bit is set publishes nothing"
    st.zero_()
    gs.gdn_chunked_prefill(d, n, R, cu_d, max(lengths), r.q, r.k, r.v, r.g, r.beta, pool, pool.stride(0),
                           pool.shape[0], src, dst, o, 64, ws, ws_bytes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    S0s = [np.zeros((dims.h_v, 128, 128)), init[1].cpu().numpy(), init[2].cpu().numpy()]
    ws_, wo_ = check_sequences(rows, cu, o, S0s, [pool[int(x)].cpu().numpy() for x in dst.tolist()], lengths)
    assert noted("prefill timed_out_wait_publishes_nothing: state (rel. Frobenius / 5e-3)", ws_ / CHUNK_STATE_RTOL) <= 1.0, ws_
    assert noted("prefill timed_out_wait_publishes_nothing: outputs", wo_) <= 1.0, wo_


@pytest.mark.parametrize("d,heads,lengths", [
    (16, (2, 2), [1, 40, 64, 130]),        # the tiny workload's head shape, ragged lengths, partial chunks
    (32, (2, 4), [0, 63, 65, 200]),
    (64, (4, 8), [7, 128, 300]),
])
def test_prefill_small_head_sizes(gs, cuda_dev, d, heads, lengths):
    """d_k = d_v in {16, 32, 64} (the fp32 chunk-form kernel): final states
    within 5e-3 (Frobenius, per sequence and head) of the FP64 recurrence and
    outputs within the bf16 bound, from zero and from a given state; slots
    that are not destinations keep their bytes."""
    dims = sy.Dims(heads[0], heads[1], d, d)
    n = len(lengths)
    pool = sy.state(sy.generator(31 + d), (2 * n + 1, dims.h_v, d, d)).to(cuda_dev)
    init = pool.clone()
    src = [(-1 if i % 2 == 0 else i) for i in range(n)]
    dst = [n + i for i in range(n)]
    rows, cu, o, st = run_prefill(gs, cuda_dev, dims, lengths, src, dst, pool, seed=40 + d, cap=sum(lengths) + 70)
    assert st == 0
    S0s = [np.zeros((dims.h_v, d, d)) if s < 0 else init[s].cpu().numpy() for s in src]
    finals = [pool[x].cpu().numpy() for x in dst]
    ws, wo = check_sequences(rows, cu, o, S0s, finals, lengths)
    print("prefill d=%d: worst state rel %.3e, worst output ratio %.3f" % (d, ws, wo))
    assert noted("prefill small_head_sizes: state (rel. Frobenius / 5e-3)", ws / CHUNK_STATE_RTOL) <= 1.0, ws
    assert noted("prefill small_head_sizes: outputs", wo) <= 1.0, wo
    for s_ in range(2 * n + 1):
        if s_ not in dst:
            assert torch.equal(pool[s_], init[s_])
