"""Zero-copy commit (gdn_verify_at / gdn_commit_at / gdn_materialize): the
arena loop gives bit-for-bit the states and tokens of the copying loop, and
refuses stale checkpoints and out-of-range locations."""
import numpy as np
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


def _arena_matches_copy(gs, cuda_dev, dims, k_hi, p_accept, steps, label):
    """The copying loop and the zero-copy loop over the same steps: draft
    counts from 0..k_hi (request 2 always asks for k_hi), hits Bernoulli with
    p_accept(step); three requests followed by the FP64 oracle."""
    from speculative_decoding_hybrid_gb300.step import ArenaStep, LayerRows, VerifyStep
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    L, B, num_slots, vocab = 3, 6, 8, 4096
    cap = B * (k_hi + 1)
    init = sy.state(sy.generator(1), (num_slots, L, dims.h_v, dims.d_v, dims.d_k)).to(cuda_dev)
    slots = [5, 0, 3, 7, 1, 6]
    vs = VerifyStep(d, L, num_slots, cap, B, vocab, cuda_dev, pool=init.clone())
    ar = ArenaStep(d, L, num_slots, cap, B, vocab, cuda_dev)
    ar.pool.copy_(init)
    ar.point_at_slots(slots)
    slot_d = torch.tensor(slots, dtype=torch.int32, device=cuda_dev)
    from gpu_util import OracleFollow
    follow = OracleFollow({r: [init[slots[r], l].cpu().numpy() for l in range(L)] for r in (0, 2, 4)})
    kg = sy.generator(2)
    max_acc = []
    for s in range(steps):
        ks = torch.randint(0, k_hi + 1, (B,), generator=kg).tolist()
        ks[2] = k_hi
        cu = [0]
        for k in ks:
            cu.append(cu[-1] + k + 1)
        R = cu[-1]
        rows = [sy.rows(sy.generator(100 * s + l), R, dims, cuda_dev) for l in range(L)]
        lrows = [LayerRows(r.q, r.k, r.v, r.g, r.beta) for r in rows]
        lg, tgt = sy.logits(sy.generator(7 + s), R, vocab, 2.0, cuda_dev)
        toks = torch.tensor(sum(sy.drafts(sy.generator(9 + s), tgt.tolist(), ks, vocab, p_accept(s)), []),
                            dtype=torch.int32, device=cuda_dev)
        cu_d = torch.tensor(cu, dtype=torch.int32, device=cuda_dev)
        vs.run(B, cu_d, slot_d, slot_d, lrows, lg, toks)
        ar.run(B, cu_d, lrows, lg, toks)
        torch.cuda.synchronize()
        assert int(vs.status.item()) == 0 and int(ar.status.item()) == 0
        assert torch.equal(vs.accept_len[:B], ar.accept_len[:B])
        assert torch.equal(vs.out_tokens[:R], ar.out_tokens[:R])
        assert torch.equal(vs.o[:, :R], ar.o[:, :R])
        # the FP64 oracle, followed for two requests: outputs, accept lengths and
        # the state each location now points at
        follow.step(cu, [[t.cpu() for t in (x.q, x.k, x.v, x.g, x.beta)] for x in rows], lg.cpu(), toks.cpu(), vocab,
                    ar.accept_len[:B].tolist(), ar.o[:, :R])
        for r in follow.S:
            follow.check_state(r, [ar.arena[int(ar.loc[l, r]):int(ar.loc[l, r]) + ar.S].view(dims.h_v, dims.d_v, dims.d_k).cpu()
                                   .numpy() for l in range(L)])
        # every location points at the accepted checkpoint of this transaction's area
        area = ar.txn & 1
        acc = ar.accept_len[:B].tolist()
        max_acc.append(max(acc))
        for l in range(L):
            for r in range(B):
                assert int(ar.loc[l, r]) == ar.area_off[area] + l * ar.ckpt_layer_stride + (cu[r] + acc[r]) * ar.S
    # states agree bit for bit once copied home
    ar.materialize(slot_d)
    torch.cuda.synchronize()
    assert int(ar.status.item()) == 0
    for sl in slots:
        assert torch.equal(ar.pool[sl], vs.pool[sl])
    print("zero-copy commit vs oracle: worst state %.3f, worst output %.3f of their bounds" %
          (follow.worst_state, follow.worst_out))
    assert noted("zero-copy commit%s: state" % label, follow.worst_state) <= 1.0
    assert noted("zero-copy commit%s: outputs" % label, follow.worst_out) <= 1.0
    return max(max_acc)


def test_arena_loop_matches_copy_loop(gs, cuda_dev):
    _arena_matches_copy(gs, cuda_dev, sy.Dims(4, 8, 128, 128), 3, lambda s: 0.85, 7, "")


@pytest.mark.parametrize("dims", [sy.Dims(4, 8, 128, 128), sy.Dims(2, 4, 64, 64), sy.Dims(2, 4, 32, 32),
                                  sy.Dims(2, 2, 16, 16)], ids=["d128", "d64", "d32", "d16"])
def test_arena_loop_at_the_maximum_draft_count(gs, cuda_dev, dims):
    """K = 15 (16 rows per request, the most one verify launch takes): on the
    all-hit steps the location points at checkpoint 15 of the request."""
    top = _arena_matches_copy(gs, cuda_dev, dims, 15, lambda s: 1.0 if s % 2 == 0 else 0.85, 5,
                              " K=15 d%d" % dims.d_k)
    assert top == 15, "no step accepted all 15 drafts"


def test_commit_at_refuses_stale_tags_and_bad_locations(gs, cuda_dev):
    from speculative_decoding_hybrid_gb300.step import ArenaStep, LayerRows
    dims = sy.Dims(2, 4, 64, 64)
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v)
    L, B = 2, 3
    ar = ArenaStep(d, L, 4, 12, B, 256, cuda_dev)
    ar.pool.normal_()
    ar.point_at_slots([0, 1, 2])
    cu = [0, 4, 6, 9]
    cu_d = torch.tensor(cu, dtype=torch.int32, device=cuda_dev)
    rows = [sy.rows(sy.generator(l), 9, dims, cuda_dev) for l in range(L)]
    lrows = [LayerRows(r.q, r.k, r.v, r.g, r.beta) for r in rows]
    lg, tgt = sy.logits(sy.generator(5), 9, 256, 2.0, cuda_dev)
    toks = torch.zeros(9, dtype=torch.int32, device=cuda_dev)
    # request 1's location is outside the arena: refused, the others run
    ar.loc[0, 1] = ar.total
    ar.run(B, cu_d, lrows, lg, toks)
    torch.cuda.synchronize()
    assert int(ar.status.item()) & gs.DEV_SLOT_OOR
    # its layer-0 checkpoint was not written, so its layer-0 location is unchanged
    assert int(ar.loc[0, 1]) == ar.total
    assert int(ar.status.item()) & gs.DEV_CKPT_UNWRITTEN
    # a stale transaction id leaves every location as it was
    before = ar.loc.clone()
    ar.status.zero_()
    gs.gdn_commit_at(d, B, L, ar.cap, cu_d, ar.accept_len, ar.area_off[0], ar.ckpt_layer_stride, ar.tags(B),
                     ar.txn + 5, ar.loc, ar.status)
    torch.cuda.synchronize()
    assert torch.equal(ar.loc, before) and int(ar.status.item()) & gs.DEV_CKPT_UNWRITTEN
