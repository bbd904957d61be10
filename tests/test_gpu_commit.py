"""GPU checks of gdn_commit: bit-exact copies of the accepted checkpoint,
refusal of checkpoints not written in this transaction, and commit j equal
to j+1 decode steps."""
import numpy as np
import pytest
import torch

import gdnsynth as sy
import oracle
from gpu_util import build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def _stack(gs, dev, dims, rows_per_req, L, num_slots, seed):
    from speculative_decoding_hybrid_gb300.step import LayerRows, VerifyStep
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    B = len(rows_per_req)
    cu = [0]
    for n in rows_per_req:
        cu.append(cu[-1] + n)
    R = cu[-1]
    pool = sy.state(sy.generator(seed), (num_slots, L, dims.h_v, dims.d_v, dims.d_k), dev)
    vs = VerifyStep(d, L, num_slots, R, B, 64, dev, pool=pool)
    rows = [sy.rows(sy.generator(seed + 1 + l), R, dims, dev) for l in range(L)]
    lrows = [LayerRows(r.q, r.k, r.v, r.g, r.beta) for r in rows]
    return d, B, cu, R, vs, lrows


def test_commit_copies_accepted_checkpoint_and_refuses_the_rest(gs, cuda_dev):
    dims = sy.Dims(4, 8, 64, 64)
    d, B, cu, R, vs, lrows = _stack(gs, cuda_dev, dims, [4, 2, 4, 1], 3, 9, 2)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=cuda_dev)
    src = torch.tensor([0, 3, 5, 7], dtype=torch.int32, device=cuda_dev)
    dst = torch.tensor([0, 8, 5, 1], dtype=torch.int32, device=cuda_dev)
    vs.txn = 41
    for l in range(3):
        vs.verify_layer(l, B, cu_d, src, lrows[l])
    vs.accept_len[:B] = torch.tensor([2, 0, 3, 0], dtype=torch.int32, device=cuda_dev)
    before = vs.pool.clone()
    vs.commit(B, cu_d, dst)
    torch.cuda.synchronize()
    assert int(vs.status.item()) == 0
    acc = [2, 0, 3, 0]
    moved = {}
    for r in range(B):
        for l in range(3):
            assert torch.equal(vs.pool[int(dst[r]), l], vs.ckpt[l, cu[r] + acc[r]])
        moved[int(dst[r])] = True
    for s in range(9):
        if s not in moved:
            assert torch.equal(vs.pool[s], before[s])

    # the oracle's commit rule gives the same moves
    tags = vs.tags(B).cpu().numpy().astype(np.uint64)
    moves, st = oracle.commit_plan(acc, cu, tags & 0xffffffff, tags >> 32, 41, dst.tolist(), 9)
    assert st == 0 and moves == [[cu[r] + acc[r] for r in range(B)] for _ in range(3)]

    # stale transaction id: nothing is written
    snap = vs.pool.clone()
    vs.txn = 42
    vs.commit(B, cu_d, dst)
    torch.cuda.synchronize()
    assert int(vs.status.item()) & gs.DEV_CKPT_UNWRITTEN
    assert torch.equal(vs.pool, snap)

    # accept length beyond the rows written, a slot outside the pool
    vs.txn = 41
    vs.status.zero_()
    vs.accept_len[:B] = torch.tensor([2, 2, 3, 0], dtype=torch.int32, device=cuda_dev)
    bad_dst = torch.tensor([0, 8, 5, 99], dtype=torch.int32, device=cuda_dev)
    vs.commit(B, cu_d, bad_dst)
    torch.cuda.synchronize()
    st = int(vs.status.item())
    assert st & gs.DEV_ACCEPT_BAD and st & gs.DEV_SLOT_OOR
    assert torch.equal(vs.pool[8], snap[8]) and torch.equal(vs.pool[1], snap[1])

    # a timed-out asynchronous copy earlier in the transaction blocks the whole commit
    vs.status.fill_(gs.DEV_TIMEOUT)
    vs.accept_len[:B] = torch.tensor([1, 1, 1, 0], dtype=torch.int32, device=cuda_dev)
    snap = vs.pool.clone()
    vs.commit(B, cu_d, dst)
    torch.cuda.synchronize()
    assert torch.equal(vs.pool, snap)


def test_commit_j_equals_j_plus_1_decode_steps(gs, cuda_dev):
    dims = sy.DIMS_FULL
    d, B, cu, R, vs, lrows = _stack(gs, cuda_dev, dims, [4, 4, 3], 2, 4, 5)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=cuda_dev)
    slots = torch.tensor([0, 1, 2], dtype=torch.int32, device=cuda_dev)
    ref = vs.pool.clone()
    vs.txn = 1
    for l in range(2):
        vs.verify_layer(l, B, cu_d, slots, lrows[l])
    acc = [3, 1, 0]
    vs.accept_len[:B] = torch.tensor(acc, dtype=torch.int32, device=cuda_dev)
    vs.commit(B, cu_d, slots)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    for r in range(B):
        for l in range(2):
            lay = ref[:, l].contiguous()
            for i in range(acc[r] + 1):
                t = cu[r] + i
                o = torch.empty((1, d.h_v, d.d_v), dtype=torch.bfloat16, device=cuda_dev)
                s = slots[r:r + 1]
                x = lrows[l]
                gs.gdn_decode_step(d, 1, x.q[t:t + 1], x.k[t:t + 1], x.v[t:t + 1], x.g[t:t + 1], x.beta[t:t + 1],
                                   lay, lay.stride(0), 4, s, s, o, st)
            torch.cuda.synchronize()
            assert torch.equal(vs.pool[r, l], lay[r]), (r, l)
    assert int(vs.status.item()) == 0 and int(st.item()) == 0


def test_bounded_wait_gives_up_and_reports(gs, cuda_dev):
    """The bounded wait behind every asynchronous copy: a barrier that is never
    completed makes the kernel give up after the limit and report
    GDN_DEV_TIMEOUT; the context stays usable and a later commit refuses."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    t0 = time.perf_counter()
    gs.gdn_selftest_wait_timeout(st, 20_000_000)     # 20 ms
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(st.item()) == gs.DEV_TIMEOUT
    x = torch.arange(4, device=cuda_dev).sum()       # the context still works
    assert int(x.item()) == 6
    with pytest.raises(gs.GdnError):
        gs.gdn_selftest_wait_timeout(st, 0)
