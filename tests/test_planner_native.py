"""The library's host planner and slot pool against the oracle's model:
identical plans (bit for bit) on the golden cases and on random request sets,
and identical pool state afterwards."""
import json
import os
import random

import pytest

import oracle
from oracle import DECODE, PREFILL, Req
from speculative_decoding_hybrid_gb300 import binding as gs

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = json.load(open(os.path.join(HERE, "golden", "planner_cases.json")))["cases"]


def to_c(reqs):
    return gs.make_reqs([(r.kind, r.k_draft, r.n_tokens, r.cur_len, r.max_len, r.slot) for r in reqs])


def run_both(reqs, free_order, take, share, max_rows, max_reqs, k_max):
    n_slots = len(free_order)
    mp = oracle.PoolModel(n_slots, list(free_order))
    cp = gs.Pool(n_slots, free_order)
    for _ in range(take):
        mp.alloc()
        cp.alloc()
    for s in share:
        mp.share(s)
        cp.share(s)
    P = oracle.plan_transaction(reqs, max_rows, max_reqs, k_max, mp)
    plan = gs.Plan(len(reqs))
    st = gs.plan_transaction(to_c(reqs), len(reqs), gs.gdn_plan_limits(max_rows, max_reqs, k_max), cp, plan)
    return P, plan, st, mp, cp


def assert_same(P, plan, st, mp, cp):
    assert st == P.status
    assert list(cp.refcount) == mp.ref
    assert cp.free_list() == mp.free
    if st != 0:
        return
    assert plan.n_selected == P.n_selected and plan.plan == P.plan and plan.deferred == P.deferred
    assert plan.k == P.k and plan.rows == P.rows and plan.src == P.src and plan.dst == P.dst
    assert plan.dec_req == P.dec_req and plan.dec_cu == P.dec_cu
    assert plan.dec_src == P.dec_src and plan.dec_dst == P.dec_dst
    assert plan.pre_req == P.pre_req and plan.pre_cu == P.pre_cu
    assert plan.pre_src == P.pre_src and plan.pre_dst == P.pre_dst
    assert plan.decode_rows == P.dec_cu[-1] and plan.prefill_rows == P.pre_cu[-1]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_golden_cases_native(case):
    from test_oracle_planner import reqs_from
    p = case["pool"]
    lim = case["limits"]
    out = run_both(reqs_from(case["reqs"]), p["free_order"], p["take"], p["share"], lim["max_rows"],
                   lim["max_reqs"], lim["k_max"])
    assert_same(*out)


def test_random_sets_match_the_model():
    rng = random.Random(11)
    for it in range(3000):
        n_slots = rng.randint(2, 20)
        order = rng.sample(range(n_slots), n_slots)
        take = rng.randint(0, n_slots)
        held = order[:take]
        share = [s for s in held if rng.random() < 0.3]
        reqs = []
        for _ in range(rng.randint(0, 9)):
            if held and rng.random() < 0.65:
                ml = rng.randint(3, 30)
                reqs.append(Req(DECODE, rng.randint(-1 if rng.random() < 0.02 else 0, 6),
                                cur_len=rng.randint(0, ml), max_len=ml, slot=rng.choice(held)))
            else:
                reqs.append(Req(PREFILL, n_tokens=rng.randint(0 if rng.random() < 0.02 else 1, 40),
                                cur_len=0, slot=rng.choice(held + [-1, -1, -1]) if held else -1))
        out = run_both(reqs, order, take, share, rng.randint(0, 70), rng.randint(0, 8), rng.randint(0, 15))
        assert_same(*out)


def test_apply_abort_and_duplicate_release_native():
    cp = gs.Pool(6, [2, 0, 1, 3, 4, 5])
    s = cp.alloc()
    cp.share(s)
    reqs = [Req(DECODE, 3, cur_len=4, slot=s), Req(DECODE, 3, cur_len=4, slot=s)]
    plan = gs.Plan(2)
    assert gs.plan_transaction(to_c(reqs), 2, gs.gdn_plan_limits(64, 64, 3), cp, plan) == gs.GDN_OK
    assert plan.dst == [0, 1]
    before = (list(cp.refcount), cp.free_list())
    assert gs.gdn_pool_abort(cp, plan, 2) == gs.GDN_OK
    assert list(cp.refcount) == [0, 0, 2, 0, 0, 0]
    assert gs.plan_transaction(to_c(reqs), 2, gs.gdn_plan_limits(64, 64, 3), cp, plan) == gs.GDN_OK
    assert gs.gdn_pool_apply(cp, plan, 2) == gs.GDN_OK
    assert cp.refcount[2] == 0 and cp.free_list()[-1] == 2
    assert cp.release(2) == gs.GDN_ERR_ARG           # duplicate release refused
    assert cp.refcount[2] == 0 and cp.free_list()[-1] == 2
    bad = gs.gdn_plan_limits(64, 64, 16)              # k_max above the kernels' limit
    assert gs.plan_transaction(to_c(reqs), 2, bad, cp, plan) == gs.GDN_ERR_ARG
