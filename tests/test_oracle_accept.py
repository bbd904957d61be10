"""Pins for the oracle's greedy choice, acceptance rule and commit rule (CPU only)."""
import itertools

import numpy as np
import pytest
import torch

import gdnsynth as sy
import oracle


def _bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return oracle.bf16_bits(t)


def test_argmax_matches_numpy_on_random_rows():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((37, 1000)).astype(np.float32) * 2
    b = _bits(x)
    ref = np.argmax(torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy(), axis=1)
    assert np.array_equal(oracle.argmax_bf16(b), ref.astype(np.int32))


def test_argmax_ties_nan_signed_zero_and_stride():
    rows = np.zeros((6, 12), dtype=np.float32)
    rows[0] = -1.0
    rows[0, [3, 7, 9]] = 5.0                      # ties: first index wins
    rows[1] = -np.inf
    rows[1, 11] = -np.inf                         # all -inf: index 0
    rows[2, :] = -1.0
    rows[2, 2] = -0.0                             # -0 and +0 compare equal:
    rows[2, 5] = 0.0                              # the first of them wins
    rows[3, :] = 1.0
    rows[3, [4, 8]] = np.nan                      # first NaN wins
    rows[4] = np.arange(12)[::-1]                 # strictly decreasing: 0
    rows[5] = np.arange(12)                       # increasing: last
    b = _bits(rows)
    got = oracle.argmax_bf16(b)
    with np.errstate(invalid="ignore"):
        ref = np.argmax(rows, axis=1)
    assert list(got) == [3, 0, 2, 4, 0, 11]
    assert np.array_equal(got, ref.astype(np.int32))
    # only the first 8 entries of each row are logits (row stride 12)
    got8 = oracle.argmax_bf16(b, vocab=8)
    assert list(got8) == [3, 0, 2, 4, 0, 7]


def _brute_accept(argmax, toks, K):
    """Definition by enumeration: the largest j such that every draft i <= j
    equals the greedy choice of the row before it."""
    best = 0
    for j in range(K + 1):
        if all(toks[i] == argmax[i - 1] for i in range(1, j + 1)):
            best = j
    return best


def test_accept_exhaustive_small_vocab():
    V = 3
    for K in range(0, 4):
        for am in itertools.product(range(V), repeat=K + 1):
            for dr in itertools.product(range(-1, V + 1), repeat=K):
                toks = np.array([0] + list(dr), dtype=np.int32)
                res = oracle.greedy_accept(np.array(am, np.int32), toks, np.array([0, K + 1]), V)
                j = _brute_accept(am, toks, K)
                assert res.accept_len[0] == j
                assert res.bonus[0] == am[j]
                assert list(res.out_tokens) == list(am[:j + 1]) + [-1] * (K - j)
                assert res.stats["accepted"] == j and res.stats["emitted"] == j + 1
                assert res.stats["proposed"] == K
                assert res.stats["evaluated"] == min(j + 1, K)
                oor = any(not (0 <= d < V) for d in dr)
                assert bool(res.status & oracle.STATUS_TOKEN_OOR) == oor


def test_accept_ragged_batch_and_empty_request():
    am = np.array([5, 6, 7, 1, 2, 9], np.int32)
    toks = np.array([0, 5, 6, 0, 1, 2], np.int32)
    cu = np.array([0, 3, 3, 4, 6])   # request 1 has no rows
    res = oracle.greedy_accept(am, toks, cu, 10)
    assert list(res.accept_len) == [2, -1, 0, 1]
    assert list(res.bonus) == [7, -1, 1, 9]
    assert res.status & oracle.STATUS_ROWS_BAD
    assert res.stats == dict(proposed=3, evaluated=3, accepted=3, emitted=6, steps=1)


def test_tiny_workload_accepts_two_drafts():
    """The tiny workload fixes drafts that match the greedy choice for the
    first two rows and miss on the third, so j = 2 and bonus = argmax of row 2."""
    spec = sy.SPECS["tiny"]
    lg, tgt = sy.ring_logits(spec, 0, 4)
    am = oracle.argmax_bf16(oracle.bf16_bits(lg))
    assert list(am) == tgt.tolist()
    toks = sy.step_drafts(spec, 0, [3], tgt.tolist())[0]
    res = oracle.greedy_accept(am, np.array(toks, np.int32), np.array([0, 4]), spec.vocab)
    assert res.accept_len[0] == 2 and res.bonus[0] == am[2]


def test_commit_moves_and_refusals():
    cu = [0, 4, 5, 9]
    acc = [2, 0, 3]
    rows = [[4, 1, 4], [4, 1, 2]]          # layer 1: request 2 wrote only 2 rows
    txn = [[7, 7, 7], [7, 6, 7]]           # layer 1: request 1's tag is stale
    moves, st = oracle.commit_plan(acc, cu, rows, txn, 7, [3, 0, 5], 6)
    assert moves[0] == [2, 4, 8]
    assert moves[1] == [2, None, None]
    assert st & oracle.STATUS_CKPT_UNWRITTEN and st & oracle.STATUS_ACCEPT_BAD
    moves, st = oracle.commit_plan([0], [0, 1], [[1]], [[1]], 1, [9], 6)
    assert moves[0] == [None] and st == oracle.STATUS_SLOT_OOR
