"""The multi-layer calls (gdn_verify_layers, gdn_verify_at_layers,
gdn_verify_replay_layers) issue the per-layer calls in layer order: every
output, checkpoint, tag and slot they write is bit-for-bit what the
layer-by-layer calls write on the same inputs."""
import pytest
import torch

import gdnsynth as sy
from gpu_util import build_lib

pytestmark = pytest.mark.gpu

DIMS = sy.Dims(4, 8, 128, 128)
L, B, NUM_SLOTS = 3, 5, 9


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def _inputs(cuda_dev, seed):
    from speculative_decoding_hybrid_gb300.step import LayerRows
    ks = [3, 0, 2, 1, 3]
    cu = [0]
    for k in ks:
        cu.append(cu[-1] + k + 1)
    cap = B * 4
    rows = []
    for l in range(L):
        r = sy.rows(sy.generator(seed + l), cap, DIMS, cuda_dev)
        rows.append(LayerRows(r.q, r.k, r.v, r.g, r.beta))
    pool = sy.state(sy.generator(seed + 50), (NUM_SLOTS, L, DIMS.h_v, DIMS.d_v, DIMS.d_k)).to(cuda_dev)
    src = torch.tensor([4, 4, 0, 7, 2], dtype=torch.int32, device=cuda_dev)   # requests 0 and 1 share slot 4
    dst = torch.tensor([8, 1, 0, 7, 2], dtype=torch.int32, device=cuda_dev)   # the shared slot is only read
    cu_t = torch.tensor(cu, dtype=torch.int32, device=cuda_dev)
    return cap, cu_t, rows, pool, src, dst


def test_verify_layers_matches_per_layer_calls(gs, cuda_dev):
    from speculative_decoding_hybrid_gb300.step import VerifyStep
    d = gs.dims(DIMS.h_qk, DIMS.h_v, DIMS.d_k, DIMS.d_v)
    cap, cu, rows, pool, src, _ = _inputs(cuda_dev, 11)
    a = VerifyStep(d, L, NUM_SLOTS, cap, B, 64, cuda_dev, pool=pool.clone())
    b = VerifyStep(d, L, NUM_SLOTS, cap, B, 64, cuda_dev, pool=pool.clone())
    for vs in (a, b):
        vs.ckpt.zero_()
        vs.o.zero_()
        vs.txn = 7
    for l in range(L):
        a.verify_layer(l, B, cu, src, rows[l])
    b.verify_all(B, cu, src, rows)
    torch.cuda.synchronize()
    R = int(cu[-1])
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert torch.equal(a.o[:, :R], b.o[:, :R])
    assert torch.equal(a.ckpt[:, :R], b.ckpt[:, :R])
    assert torch.equal(a.tags(B), b.tags(B))
    assert torch.equal(a.pool, b.pool) and torch.equal(b.pool, pool)     # verify leaves the slots alone


def test_verify_at_layers_matches_per_layer_calls(gs, cuda_dev):
    from speculative_decoding_hybrid_gb300.step import ArenaStep
    d = gs.dims(DIMS.h_qk, DIMS.h_v, DIMS.d_k, DIMS.d_v)
    cap, cu, rows, pool, src, _ = _inputs(cuda_dev, 21)
    slots = src.tolist()
    steps = []
    for _ in range(2):
        st = ArenaStep(d, L, NUM_SLOTS, cap, B, 64, cuda_dev)
        st.pool.copy_(pool)
        st.point_at_slots(slots)
        st.arena[st.area_off[0]:].zero_()
        st.o.zero_()
        st.txn = 4
        steps.append(st)
    a, b = steps
    for l in range(L):
        x = rows[l]
        gs.gdn_verify_at(a.d, B, a.cap, cu, x.q, x.k, x.v, x.g, x.beta, a.arena, a.total, a.loc[l],
                         a.areas[a.txn & 1][l], a.tags(B)[l], a.txn, a.o[l], a.status)
    b.verify_all_at(B, cu, rows)
    torch.cuda.synchronize()
    R = int(cu[-1])
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert torch.equal(a.o[:, :R], b.o[:, :R])
    assert torch.equal(a.areas[0][:, :R], b.areas[0][:, :R])
    assert torch.equal(a.tags(B), b.tags(B))


def test_verify_replay_layers_matches_per_layer_calls(gs, cuda_dev):
    from speculative_decoding_hybrid_gb300.step import ReplayStep
    d = gs.dims(DIMS.h_qk, DIMS.h_v, DIMS.d_k, DIMS.d_v)
    cap, cu, rows, pool, src, dst = _inputs(cuda_dev, 31)
    _, _, prev_rows, _, _, _ = _inputs(cuda_dev, 41)
    prev_acc = torch.tensor([2, 0, 1, 0, 3], dtype=torch.int32, device=cuda_dev)
    a = ReplayStep(d, L, NUM_SLOTS, cap, B, 64, cuda_dev, pool=pool.clone())
    b = ReplayStep(d, L, NUM_SLOTS, cap, B, 64, cuda_dev, pool=pool.clone())
    for rs in (a, b):
        rs.prev_cu.copy_(cu)
        rs.prev_acc.copy_(prev_acc)
        rs.prev_rows = prev_rows
        rs.o.zero_()
    for l in range(L):
        x, p = rows[l], prev_rows[l]
        gs.gdn_verify_replay(a.d, B, a.cap, cu, x.q, x.k, x.v, x.g, x.beta, a.cap, a.prev_cu, a.prev_acc, p.k, p.v,
                             p.g, p.beta, a.pool_layer(l), a.slot_stride, a.num_slots, src, dst, a.o[l], a.status)
    b._verify_all(B, cu, src, dst, rows)
    torch.cuda.synchronize()
    R = int(cu[-1])
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert torch.equal(a.o[:, :R], b.o[:, :R])
    assert torch.equal(a.pool, b.pool)
    assert not torch.equal(b.pool, pool)                                    # the replay wrote the slots


def test_commit_then_verify_layers_back_to_back(gs, cuda_dev):
    """A commit followed at once (same stream, nothing in between) by a
    multi-layer verify on a batch small enough for one wave: every layer,
    the later ones included, must start from the committed state.  Checked
    against the FP64 oracle run from the committed checkpoints and bit for
    bit against the same calls with a device synchronisation in between."""
    import oracle
    from gpu_util import noted, out_err, state_err
    dims = sy.DIMS_FULL
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    Lb, rows_n, j = 3, 4, 2
    cu = torch.tensor([0, rows_n], dtype=torch.int32, device=cuda_dev)
    slot = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    from speculative_decoding_hybrid_gb300.step import LayerRows, VerifyStep
    steps = [[LayerRows(*(t for t in (r.q, r.k, r.v, r.g, r.beta)))
              for r in (sy.rows(sy.generator(900 + 10 * s + l), rows_n, dims, cuda_dev) for l in range(Lb))]
             for s in range(2)]
    pool0 = sy.state(sy.generator(950), (1, Lb, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    results = []
    for sync in (False, True):
        vs = VerifyStep(d, Lb, 1, rows_n, 1, 64, cuda_dev, pool=pool0.clone())
        vs.accept_len.fill_(j)
        vs.txn = 1
        vs.verify_all(1, cu, slot, steps[0])
        vs.commit(1, cu, slot)
        if sync:
            torch.cuda.synchronize()
        vs.txn = 2
        vs.verify_all(1, cu, slot, steps[1])
        torch.cuda.synchronize()
        assert int(vs.status.item()) == 0
        results.append((vs.ckpt[:, :rows_n].clone(), vs.o[:, :rows_n].clone(), vs.pool.clone()))
    assert torch.equal(results[0][0], results[1][0]) and torch.equal(results[0][1], results[1][1])
    ck, o, pool = results[0]
    for l in range(Lb):
        h0 = [t.cpu() for t in (steps[0][l].q, steps[0][l].k, steps[0][l].v, steps[0][l].g, steps[0][l].beta)]
        _, _, ck0 = oracle.gdn_recurrent(*h0, pool0[0, l].cpu(), 1.0, want_ckpt=True)
        committed = ck0[j]
        assert noted("commit then verify back to back: committed state", state_err(pool[0, l].cpu().numpy(), committed)) <= 1.0
        h1 = [t.cpu() for t in (steps[1][l].q, steps[1][l].k, steps[1][l].v, steps[1][l].g, steps[1][l].beta)]
        _, o_ref, ck1 = oracle.gdn_recurrent(*h1, torch.from_numpy(committed), 1.0, want_ckpt=True)
        assert noted("commit then verify back to back: checkpoints", state_err(ck[l].cpu().numpy(), ck1)) <= 1.0, l
        assert noted("commit then verify back to back: outputs", out_err(o[l], o_ref)) <= 1.0, l
