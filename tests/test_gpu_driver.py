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
