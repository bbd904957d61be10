"""GPU parity of gdn_verify / gdn_decode_step against the FP64 oracle, plus
the decode/verify rounding identity (bit-exact) and fail-closed paths."""
import numpy as np
import pytest
import torch

import gdnsynth as sy
import oracle
from gpu_util import build_lib, noted, oracle_request, out_err, rows_to_host, state_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def _setup(gs, dims, rows_per_req, num_slots, seed, dev, q_scale=1.0):
    d = gs.dims(dims.h_qk, dims.h_v, dims.d_k, dims.d_v, q_scale)
    B = len(rows_per_req)
    cu = [0]
    for n in rows_per_req:
        cu.append(cu[-1] + n)
    R = cu[-1]
    gen = sy.generator(seed)
    rows = sy.rows(gen, R, dims)
    pool = sy.state(sy.generator(seed + 1), (num_slots, dims.h_v, dims.d_v, dims.d_k))
    perm = torch.randperm(num_slots, generator=sy.generator(seed + 2))[:B].to(torch.int32)
    return d, B, cu, R, rows, pool, perm


def _dev(x, dev):
    return x.to(dev).contiguous()


def _verify(gs, d, B, cu, R, rows, pool_d, src_d, dev, txn=7, cap=None):
    cap = R if cap is None else cap
    ck = torch.full((max(cap, 1), d.h_v, d.d_v, d.d_k), float("nan"), device=dev)
    tags = torch.zeros(max(B, 1), dtype=torch.int64, device=dev)
    o = torch.zeros((max(cap, 1), d.h_v, d.d_v), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
    r = rows.to(dev)
    gs.gdn_verify(d, B, cap, cu_d, r.q, r.k, r.v, r.g, r.beta, pool_d, pool_d.stride(0), pool_d.shape[0], src_d, ck,
                  tags, txn, o, st)
    torch.cuda.synchronize()
    return ck, tags, o, st


CASES = [
    ("tiny", sy.DIMS_TINY, [4], 2),
    ("batch1", sy.DIMS_FULL, [4], 3),
    ("ragged", sy.DIMS_FULL, [1, 4, 2, 16, 3], 8),
    ("dk32", sy.Dims(2, 4, 32, 32), [3, 1, 5], 4),
    ("dk64", sy.Dims(4, 8, 64, 64), [2, 4], 3),
    ("gqa4", sy.Dims(2, 8, 128, 128), [4, 2], 2),
]


@pytest.mark.parametrize("name,dims,rows_per_req,num_slots", CASES, ids=[c[0] for c in CASES])
def test_verify_matches_oracle(gs, cuda_dev, name, dims, rows_per_req, num_slots):
    q_scale = 0.75 if name == "dk64" else 1.0
    d, B, cu, R, rows, pool, perm = _setup(gs, dims, rows_per_req, num_slots, 11, cuda_dev, q_scale)
    pool_d = _dev(pool, cuda_dev)
    before = pool_d.clone()
    src = _dev(perm, cuda_dev)
    ck, tags, o, st = _verify(gs, d, B, cu, R, rows, pool_d, src, cuda_dev)
    assert int(st.item()) == 0
    assert torch.equal(pool_d, before), "verify must not write the slot"
    tg = tags.cpu().numpy().astype(np.uint64)
    host = rows_to_host(rows)
    for r in range(B):
        assert int(tg[r]) == (7 << 32) | rows_per_req[r]
        S, o_ref, ck_ref = oracle_request(host, cu[r], cu[r + 1], pool[int(perm[r])], q_scale)
        assert noted("verify %s: checkpoints" % name, state_err(ck[cu[r]:cu[r + 1]].cpu().numpy(), ck_ref)) <= 1.0
        assert noted("verify %s: outputs" % name, out_err(o[cu[r]:cu[r + 1]], o_ref)) <= 1.0


@pytest.mark.parametrize("name,dims,rows_per_req,num_slots", CASES[:4], ids=[c[0] for c in CASES[:4]])
def test_checkpoint_j_is_bit_identical_to_j_plus_1_decode_steps(gs, cuda_dev, name, dims, rows_per_req, num_slots):
    d, B, cu, R, rows, pool, perm = _setup(gs, dims, rows_per_req, num_slots, 5, cuda_dev)
    pool_d = _dev(pool, cuda_dev)
    src = _dev(perm, cuda_dev)
    ck, tags, o, st = _verify(gs, d, B, cu, R, rows, pool_d.clone(), src, cuda_dev)
    # decode: request r's row i runs as one decode step, state in place
    dec_pool = pool_d.clone()
    st2 = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    r_dev = rows.to(cuda_dev)
    for i in range(max(rows_per_req)):
        live = [r for r in range(B) if i < rows_per_req[r]]
        idx = torch.tensor([cu[r] + i for r in live], dtype=torch.long, device=cuda_dev)
        sl = torch.tensor([int(perm[r]) for r in live], dtype=torch.int32, device=cuda_dev)
        od = torch.zeros((len(live), d.h_v, d.d_v), dtype=torch.bfloat16, device=cuda_dev)
        gs.gdn_decode_step(d, len(live), r_dev.q[idx].contiguous(), r_dev.k[idx].contiguous(),
                           r_dev.v[idx].contiguous(), r_dev.g[idx].contiguous(), r_dev.beta[idx].contiguous(),
                           dec_pool, dec_pool.stride(0), dec_pool.shape[0], sl, sl, od, st2)
        torch.cuda.synchronize()
        for n, r in enumerate(live):
            assert torch.equal(dec_pool[int(perm[r])], ck[cu[r] + i]), (r, i)
            assert torch.equal(od[n], o[cu[r] + i]), (r, i)
    assert int(st2.item()) == 0


def test_decode_step_matches_oracle_and_copy_on_write(gs, cuda_dev):
    dims = sy.DIMS_FULL
    d, B, cu, R, rows, pool, perm = _setup(gs, dims, [1, 1, 1], 6, 21, cuda_dev)
    pool_d = _dev(pool, cuda_dev)
    src = torch.tensor([0, 0, 3], dtype=torch.int32, device=cuda_dev)     # two readers of slot 0
    dst = torch.tensor([4, 5, 3], dtype=torch.int32, device=cuda_dev)     # copy-on-write + in place
    o = torch.zeros((B, d.h_v, d.d_v), dtype=torch.bfloat16, device=cuda_dev)
    st = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    r = rows.to(cuda_dev)
    gs.gdn_decode_step(d, B, r.q, r.k, r.v, r.g, r.beta, pool_d, pool_d.stride(0), 6, src, dst, o, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(pool_d[0].cpu(), pool[0]), "shared slot must stay untouched"
    host = rows_to_host(rows)
    for i, (s, t) in enumerate([(0, 4), (0, 5), (3, 3)]):
        S, o_ref, _ = oracle_request(host, i, i + 1, pool[s])
        assert noted("decode step: state", state_err(pool_d[t].cpu().numpy()[None], S[None])) <= 1.0
        assert noted("decode step: outputs", out_err(o[i:i + 1], o_ref)) <= 1.0


def test_batch_invariance(gs, cuda_dev):
    """A request's checkpoints and outputs do not depend on its neighbours."""
    dims = sy.DIMS_FULL
    d, B, cu, R, rows, pool, perm = _setup(gs, dims, [4, 1, 3, 4, 2, 4, 4, 1, 2, 3, 4, 4, 4, 1, 2, 4], 16, 3,
                                           cuda_dev)
    pool_d = _dev(pool, cuda_dev)
    src = _dev(perm, cuda_dev)
    ck, tags, o, st = _verify(gs, d, B, cu, R, rows, pool_d, src, cuda_dev)
    for r in (0, 5, 15):
        sub = rows.slice(cu[r], cu[r + 1])
        ck1, _, o1, _ = _verify(gs, d, 1, [0, cu[r + 1] - cu[r]], cu[r + 1] - cu[r], sub, pool_d, src[r:r + 1],
                                cuda_dev)
        assert torch.equal(ck1, ck[cu[r]:cu[r + 1]])
        assert torch.equal(o1, o[cu[r]:cu[r + 1]])


def test_fail_closed_paths(gs, cuda_dev):
    dims = sy.DIMS_TINY
    d, B, cu, R, rows, pool, perm = _setup(gs, dims, [2, 3, 2], 4, 8, cuda_dev)
    pool_d = _dev(pool, cuda_dev)
    # request 1 names a slot outside the pool; request 0 and 2 still run
    src = torch.tensor([1, 9, 2], dtype=torch.int32, device=cuda_dev)
    ck, tags, o, st = _verify(gs, d, B, cu, R, rows, pool_d, src, cuda_dev)
    assert int(st.item()) & gs.DEV_SLOT_OOR
    tg = tags.cpu().numpy().astype(np.uint64)
    assert int(tg[1]) == (7 << 32)
    assert torch.isnan(ck[cu[1]:cu[2]]).all(), "a refused request writes no checkpoint"
    assert not torch.isnan(ck[cu[0]:cu[1]]).any() and not torch.isnan(ck[cu[2]:cu[3]]).any()
    # rows beyond the capacity and more rows than the draft limit allows
    src = torch.tensor([1, 2, 3], dtype=torch.int32, device=cuda_dev)
    ck, tags, o, st = _verify(gs, d, B, cu, R, rows, pool_d, src, cuda_dev, cap=5)
    assert int(st.item()) & gs.DEV_ROWS_BAD
    assert int(tags.cpu().numpy().astype(np.uint64)[2]) == (7 << 32)
    big = [20]
    d2, B2, cu2, R2, rows2, pool2, perm2 = _setup(gs, dims, big, 4, 8, cuda_dev)
    ck, tags, o, st = _verify(gs, d2, 1, cu2, R2, rows2, pool_d, torch.tensor([0], dtype=torch.int32,
                                                                              device=cuda_dev), cuda_dev)
    assert int(st.item()) & gs.DEV_ROWS_BAD
    # host-visible errors launch nothing
    with pytest.raises(gs.GdnError):
        gs.gdn_verify(gs.dims(2, 3, 16, 16), 1, 4, 0, 0, 0, 0, 0, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0)
    # an empty batch is a no-op
    gs.gdn_verify(d, 0, 0, torch.zeros(1, dtype=torch.int32, device=cuda_dev), *([pool_d] * 5), pool_d,
                  pool_d.stride(0), 4, src, pool_d, tags, 1, pool_d, st)
