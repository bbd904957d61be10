"""gdn_decode_transaction (the library's host driver of one decode
transaction) against the same transaction driven from Python one library
call at a time: over several steps with ragged draft counts and a shared
prefix slot (copy-on-write), every committed state, accept length, emitted
token, telemetry counter, slot-pool entry and request record is identical."""
import numpy as np
import pytest
import torch

import gdnsynth as sy
from gpu_util import build_lib

pytestmark = pytest.mark.gpu

# 12 requests, 2 layers, K ~ U{0..3}, 4 of them on request 0's slot, 24 slots, 2 input sets
SPEC = sy.Spec("driver", sy.DIMS_FULL, 2, 12, None, 3, 6, 4096, 2.0, 0.85, 24, 4, 2, 7)


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


@pytest.mark.parametrize("arena", [False, True])
def test_native_transaction_matches_python_driver(gs, cuda_dev, arena):
    """Copy commit (gdn_decode_transaction) and zero-copy commit over a state
    arena (gdn_decode_transaction_at)."""
    import bench
    steps = SPEC.steps
    runs = []
    for python_driver in (True, False):
        b = bench.Bench(SPEC, cuda_dev, arena=arena, python_driver=python_driver)
        assert b.native == (not python_driver)
        b.precompute_drafts(steps)
        per_step = []
        for _ in range(steps):
            n, p = b.step()
            torch.cuda.synchronize()
            B = b.loop.B
            per_step.append((n, p.k, p.dst, b.loop.h_out[:B].clone(), b.loop.h_out[B:2 * B].clone(),
                             b.vs.out_tokens[:p.decode_rows].clone()))
        runs.append((b, per_step))
    (a, sa), (n, sn) = runs
    for x, y in zip(sa, sn):
        assert x[0] == y[0] and x[1] == y[1] and x[2] == y[2]
        assert torch.equal(x[3], y[3]) and torch.equal(x[4], y[4]) and torch.equal(x[5], y[5])
    assert int(a.vs.status.item()) == 0 and int(n.vs.status.item()) == 0
    assert torch.equal(a.vs.pool, n.vs.pool)
    if arena:
        assert torch.equal(a.vs.loc, n.vs.loc) and torch.equal(a.vs.arena, n.vs.arena)
    assert torch.equal(a.vs.stats, n.vs.stats)
    assert a.vs.txn == n.vs.txn == steps
    assert np.array_equal(a.loop.req_np, n.loop.req_np)
    assert np.array_equal(a.pool_c.refcount, n.pool_c.refcount)
    assert a.pool_c.free_list() == n.pool_c.free_list()
    assert sum(k for x in sa for k in x[1]) > 0 and a.verified == n.verified


def test_native_transaction_refuses_a_prefill(gs, cuda_dev):
    """A request list holding a prefill is not a decode transaction: it is
    refused before anything is planned or launched; the slot pool, the
    requests and the transaction counter are unchanged."""
    import bench
    b = bench.Bench(SPEC, cuda_dev)
    loop = b.loop
    before = (b.pool_c.refcount.copy(), b.pool_c.free_list(), loop.req_np.copy())
    loop.req_np[0, 0] = gs.REQ_PREFILL
    loop.req_np[0, 2] = 5
    loop.req_np[0, 5] = -1
    with pytest.raises(gs.GdnError) as e:
        loop.transaction(b.rows[0], b.logits[0], b.tok_d)
    assert e.value.status == gs.GDN_ERR_ARG
    assert np.array_equal(b.pool_c.refcount, before[0]) and b.pool_c.free_list() == before[1]
    loop.req_np[0] = before[2][0]
    assert np.array_equal(loop.req_np, before[2])
    assert b.vs.txn == 0


def _snapshot(b, arena):
    return (b.pool_c.refcount.copy(), b.pool_c.free_list(), b.loop.req_np.copy(), b.vs.txn,
            b.vs.pool.clone(), b.vs.loc.clone() if arena else None)


def _assert_unchanged(b, arena, before):
    ref, free, req, txn, pool, loc = before
    assert np.array_equal(b.pool_c.refcount, ref) and b.pool_c.free_list() == free
    keep = [0, 2, 3, 4, 5]                      # all but k_draft, which the step itself sets before the call
    assert np.array_equal(b.loop.req_np[:, keep], req[:, keep])
    assert b.vs.txn == txn and b.loop._txn.value == txn
    assert torch.equal(b.vs.pool, pool)
    if arena:
        assert torch.equal(b.vs.loc, loc)


@pytest.mark.parametrize("arena", [False, True])
def test_native_transaction_refused_on_device_commits_nothing(gs, cuda_dev, arena):
    """A problem only the device sees makes the host driver refuse the whole
    transaction ([NATIVE] Results, recovery after abort): no state, slot or
    location is written, the slot pool, the requests and the transaction
    counter are left as they were, every accept length reads -1, and the
    status word names the cause.  Two injected causes, both made on the
    host: a bounded wait reported as run out (GDN_DEV_TIMEOUT already in the
    status word), and a start state the device finds out of range.  After
    the status word is cleared the same loop goes on and commits."""
    import bench
    b = bench.Bench(SPEC, cuda_dev, arena=arena)
    b.precompute_drafts(4)
    b.step()                                   # one committed transaction first (COW moves included)
    torch.cuda.synchronize()
    loop = b.loop
    B = loop.B

    before = _snapshot(b, arena)
    b.vs.status.fill_(gs.DEV_TIMEOUT)
    with pytest.raises(gs.GdnError) as e:
        b.native_step()
    torch.cuda.synchronize()
    assert e.value.status == gs.GDN_ERR_REFUSED
    assert int(b.vs.status.item()) & gs.DEV_TIMEOUT
    assert (b.vs.accept_len[:B] == -1).all()
    _assert_unchanged(b, arena, before)

    b.vs.status.zero_()
    if arena:
        saved = b.vs.loc[1, 3].clone()
        b.vs.loc[1, 3] = -4                     # layer 1 of request 3 points outside the arena
    else:
        saved = loop._io.num_slots
        loop._io.num_slots = int(max(loop.slot)) # the request on the highest slot is out of range
    before = _snapshot(b, arena)
    with pytest.raises(gs.GdnError) as e:
        b.native_step()
    torch.cuda.synchronize()
    assert e.value.status == gs.GDN_ERR_REFUSED
    st = int(b.vs.status.item())
    assert st & gs.DEV_SLOT_OOR and st & gs.DEV_CKPT_UNWRITTEN
    assert (b.vs.accept_len[:B] == -1).all()
    _assert_unchanged(b, arena, before)
    if arena:
        b.vs.loc[1, 3] = saved
    else:
        loop._io.num_slots = saved

    b.vs.status.zero_()
    n, p = b.step()                            # the loop goes on from where it was
    torch.cuda.synchronize()
    assert int(b.vs.status.item()) == 0 and n > 0
    assert b.vs.txn == before[3] + 1
