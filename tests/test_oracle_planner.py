"""Pins for the oracle's transaction planner and slot-pool model (CPU only).

Golden cases in ``tests/golden/planner_cases.json`` encode the pages' wording
(each case carries its citation); the remaining tests check invariants that
the deferral, clamp and copy-on-write rules imply, over random request sets.
"""
import json
import os
import random

import pytest

import oracle
from oracle import DECODE, PREFILL, Req

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = json.load(open(os.path.join(HERE, "golden", "planner_cases.json")))["cases"]


def pool_from(spec):
    p = oracle.PoolModel(spec["num_slots"], spec["free_order"])
    for _ in range(spec["take"]):
        st, _s = p.alloc()
        assert st == oracle.OK
    for s in spec["share"]:
        assert p.share(s) == oracle.OK
    return p


def reqs_from(lst):
    out = []
    for r in lst:
        out.append(Req(kind=DECODE if r["kind"] == "decode" else PREFILL,
                       k_draft=r.get("k_draft", 0), n_tokens=r.get("n_tokens", 0),
                       cur_len=r.get("cur_len", 0), max_len=r.get("max_len", 1 << 30),
                       slot=r.get("slot", -1)))
    return out


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_golden_case(case):
    pool = pool_from(case["pool"])
    lim = case["limits"]
    P = oracle.plan_transaction(reqs_from(case["reqs"]), lim["max_rows"], lim["max_reqs"], lim["k_max"], pool)
    e = case["expect"]
    assert P.status == e["status"]
    assert P.n_selected == e["n_selected"]
    assert P.plan == (oracle.PLAN_CHUNKED if e["plan"] == "chunked" else oracle.PLAN_RECURRENT)
    assert P.deferred == e["deferred"]
    assert P.k == e["k"] and P.rows == e["rows"]
    assert P.src == e["src"] and P.dst == e["dst"]
    assert P.dec_cu == e["dec_cu"] and P.pre_cu == e["pre_cu"]


def test_cow_then_apply_releases_shared_slot_once():
    pool = oracle.PoolModel(8, [5, 0, 1, 2, 3, 4, 6, 7])
    pool.alloc()
    pool.share(5)
    reqs = [Req(DECODE, 3, cur_len=10, slot=5), Req(DECODE, 3, cur_len=10, slot=5)]
    P = oracle.plan_transaction(reqs, 64, 64, 3, pool)
    assert P.dst == [0, 1] and pool.ref[5] == 2
    assert oracle.pool_apply(pool, reqs, P) == oracle.OK
    assert pool.ref[5] == 0 and pool.free[-1] == 5
    # a second release of the same slot is a duplicate release: refused, no change
    free_before = list(pool.free)
    assert pool.release(5) == oracle.ERR_ARG
    assert pool.free == free_before


def test_abort_restores_the_pool():
    pool = oracle.PoolModel(6)
    for _ in range(2):
        pool.alloc()
    pool.share(0)
    before = (list(pool.ref), list(pool.free))
    reqs = [Req(DECODE, 3, cur_len=1, slot=0), Req(PREFILL, n_tokens=9), Req(DECODE, 2, cur_len=1, slot=1)]
    P = oracle.plan_transaction(reqs, 64, 64, 3, pool)
    assert P.status == oracle.OK and P.deferred == 5
    assert oracle.pool_abort(pool, reqs, P) == oracle.OK
    assert sorted(pool.free) == sorted(before[1]) and pool.ref == before[0]


def test_out_of_slots_rolls_back_reservations():
    pool = oracle.PoolModel(3)
    pool.alloc()
    before = (list(pool.ref), list(pool.free))
    reqs = [Req(PREFILL, n_tokens=4), Req(PREFILL, n_tokens=4), Req(PREFILL, n_tokens=4)]
    P = oracle.plan_transaction(reqs, 64, 64, 3, pool)
    assert P.status == oracle.ERR_NO_SLOT
    assert (pool.ref, pool.free) == before


def test_inconsistent_slot_claims_fail_closed():
    pool = oracle.PoolModel(4)
    pool.alloc()
    before = (list(pool.ref), list(pool.free))
    # two requests claim slot 0 whose count is 1: both would write it in place
    reqs = [Req(DECODE, 1, cur_len=3, slot=0), Req(DECODE, 1, cur_len=3, slot=0)]
    P = oracle.plan_transaction(reqs, 64, 64, 3, pool)
    assert P.status == oracle.ERR_DUP_SLOT and (pool.ref, pool.free) == before
    # a slot that is not held, a finished sequence, an empty prefill
    for bad in ([Req(DECODE, 1, cur_len=3, slot=2)], [Req(DECODE, 1, cur_len=9, max_len=9, slot=0)],
                [Req(PREFILL, n_tokens=0)], [Req(DECODE, 1, cur_len=3, slot=7)]):
        P = oracle.plan_transaction(bad, 64, 64, 3, pool)
        assert P.status == oracle.ERR_ARG and (pool.ref, pool.free) == before


def _random_case(rng):
    n_slots = rng.randint(4, 24)
    pool = oracle.PoolModel(n_slots, rng.sample(range(n_slots), n_slots))
    held = []
    for _ in range(rng.randint(0, n_slots // 2)):
        held.append(pool.alloc()[1])
    for s in held:
        if rng.random() < 0.3:
            pool.share(s)
    reqs = []
    for _ in range(rng.randint(0, 10)):
        if held and rng.random() < 0.7:
            s = rng.choice(held)
            ml = rng.randint(5, 40)
            reqs.append(Req(DECODE, rng.randint(0, 5), cur_len=rng.randint(0, ml - 1), max_len=ml, slot=s))
        else:
            reqs.append(Req(PREFILL, n_tokens=rng.randint(1, 50), cur_len=0,
                            slot=rng.choice(held + [-1, -1]) if held else -1))
    return pool, reqs, rng.randint(1, 80), rng.randint(1, 8), rng.randint(0, 15)


def test_plan_invariants_over_random_sets():
    rng = random.Random(7)
    for _ in range(3000):
        pool, reqs, max_rows, max_reqs, k_max = _random_case(rng)
        ref_before = list(pool.ref)
        P = oracle.plan_transaction(reqs, max_rows, max_reqs, k_max, pool)
        if P.status != oracle.OK:
            assert pool.ref == ref_before
            continue
        sel = [i for i in range(len(reqs)) if P.k[i] >= 0]
        assert sel == list(range(P.n_selected))
        assert sum(P.rows) <= max_rows and P.n_selected <= max_reqs
        has_pre = any(reqs[i].kind == PREFILL for i in sel)
        if has_pre:
            assert all(P.k[i] == 0 for i in sel)
        for i in sel:
            r = reqs[i]
            if r.kind == DECODE:
                assert P.rows[i] == P.k[i] + 1
                assert r.cur_len + P.k[i] + 1 <= r.max_len and P.k[i] <= k_max
                if not has_pre:
                    budget = max_rows - sum(P.rows[:i])
                    assert P.k[i] == max(0, min(r.k_draft, k_max, r.max_len - r.cur_len - 1, budget - 1))
            # in place iff the slot was held once; shared slots are never written
            if r.slot >= 0 and ref_before[r.slot] == 1:
                assert P.dst[i] == r.slot
            else:
                assert P.dst[i] != r.slot and ref_before[P.dst[i]] == 0
        dsts = [P.dst[i] for i in sel]
        assert len(set(dsts)) == len(dsts)
        assert P.dec_cu[-1] + P.pre_cu[-1] == sum(P.rows)
