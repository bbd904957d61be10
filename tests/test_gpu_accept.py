"""GPU parity of mtp_greedy_accept: argmax ids, accept lengths, bonus tokens,
emitted tokens and telemetry must equal the oracle's bit for bit."""
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


def run_accept(gs, dev, logits, vocab, tokens, cu, stats=None, cap=None):
    rows = logits.shape[0]
    cap = rows if cap is None else cap
    B = len(cu) - 1
    ws_bytes = gs.mtp_accept_workspace_bytes(cap, vocab)
    ws = torch.empty(max(ws_bytes, 8), dtype=torch.uint8, device=dev)
    am = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)
    acc = torch.full((max(B, 1),), -7, dtype=torch.int32, device=dev)
    bon = torch.full((max(B, 1),), -7, dtype=torch.int32, device=dev)
    out = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stats = torch.zeros(5, dtype=torch.int64, device=dev) if stats is None else stats
    gs.mtp_greedy_accept(B, cap, torch.tensor(cu, dtype=torch.int32, device=dev), logits, vocab, logits.stride(0),
                         torch.tensor(tokens, dtype=torch.int32, device=dev), am, acc, bon, out, stats, ws,
                         ws_bytes, st)
    torch.cuda.synchronize()
    return am.cpu().numpy(), acc.cpu().numpy()[:B], bon.cpu().numpy()[:B], out.cpu().numpy(), int(st.item()), stats


def check_against_oracle(gs, dev, logits_cpu, vocab, tokens, cu, cap=None):
    am, acc, bon, out, st, stats = run_accept(gs, dev, logits_cpu.to(dev), vocab, tokens, cu, cap=cap)
    bits = oracle.bf16_bits(logits_cpu)[:, :vocab]
    am_ref = oracle.argmax_bf16(np.ascontiguousarray(bits))
    R = cu[-1]
    assert np.array_equal(am[:R], am_ref[:R])
    res = oracle.greedy_accept(am_ref, np.array(tokens, np.int32), np.array(cu), vocab)
    assert np.array_equal(acc, res.accept_len)
    assert np.array_equal(bon, res.bonus)
    assert np.array_equal(out[:R], res.out_tokens)
    s = stats.cpu().numpy().astype(np.uint64)
    assert [int(x) for x in s] == [res.stats[k] for k in ("proposed", "evaluated", "accepted", "emitted", "steps")]
    assert st == res.status
    return res


def test_full_vocab_bernoulli_drafts(gs, cuda_dev):
    spec = sy.SPECS["paged256"]
    ks = [3, 0, 2, 3, 1, 3, 3, 2]
    R = sum(k + 1 for k in ks)
    lg, tgt = sy.logits(sy.generator(4), R, spec.vocab, 2.0)
    toks = sy.drafts(sy.generator(5), tgt.tolist(), ks, spec.vocab, 0.85)
    cu = [0]
    for k in ks:
        cu.append(cu[-1] + k + 1)
    check_against_oracle(gs, cuda_dev, lg, spec.vocab, sum(toks, []), cu)


def test_ties_nan_and_split_boundaries(gs, cuda_dev):
    V = 151936
    R = 7
    lg = torch.randn((R, V), generator=sy.generator(9)).to(torch.bfloat16)
    # row 0: ties at three places, spanning several CTA splits: the lowest index wins
    for i in (149000, 70001, 70000):
        lg[0, i] = 9.0
    # row 1: NaNs -- the first one wins; row 2: every value equal; row 3: -0 before +0 at the top
    lg[1, 5000] = float("nan")
    lg[1, 4000] = float("nan")
    lg[1, 100] = 30.0
    lg[2] = -3.0
    lg[3] = -1.0
    lg[3, 77777] = -0.0
    lg[3, 77778] = 0.0
    lg[4] = float("-inf")
    lg[4, V - 1] = -1e30
    lg[5, V - 1] = 50.0
    lg[6] = float("-inf")     # row 6: nothing but -inf, so the first index wins
    toks = [0, 1, 2, 3, 4, 5, 6]
    cu = [0, 2, 4, 7]
    toks[1] = 70000           # draft equals row 0's greedy choice
    check_against_oracle(gs, cuda_dev, lg, V, toks, cu)


def test_whole_row_scans_adversarial_orders(gs, cuda_dev):
    """A row capacity of 1,024 gives one CTA per row (no vocabulary split), so
    every thread streams ~74 vectors through the grouped scan whose exact key
    search a warp skips when the group's largest value does not beat the
    largest it has recorded.  Orders that defeat or test that skip: a rising
    ramp (every group beats the last; bf16 rounding makes plateaus, so the
    first index of the top plateau must win), a falling ramp, a constant row,
    the maximum repeated in many groups, the maximum only in the per-lane tail,
    an equal value earlier than that tail, a NaN after a large value, and
    -0 / +0 as the top in either order."""
    V = 151936
    R = 10
    lg = (torch.randn((R, V), generator=sy.generator(31)) * 2.0).to(torch.bfloat16)
    ramp = torch.linspace(-40.0, 40.0, V)
    lg[0] = ramp.to(torch.bfloat16)
    lg[1] = ramp.flip(0).to(torch.bfloat16)
    lg[2] = 1.5
    for i in range(5003, V, 997):
        lg[3, i] = 20.0
    lg[4, V - 1] = 25.0
    lg[5, V - 2] = 25.0
    lg[5, 12345] = 25.0
    lg[6, 300] = 40.0
    lg[6, 140000] = float("nan")
    lg[7] = -2.0
    lg[7, 100000] = -0.0
    lg[7, 50000] = 0.0
    lg[8] = -2.0
    lg[8, 50000] = -0.0
    lg[8, 100000] = 0.0
    lg[9] = float("-inf")
    toks = list(range(R))
    cu = [0, 4, 10]
    check_against_oracle(gs, cuda_dev, lg, V, toks, cu, cap=1024)


@pytest.mark.parametrize("vocab,stride", [(64, 64), (1001, 1001), (1001, 1008), (5000, 5003), (151936, 151936)])
def test_vocab_sizes_and_strides(gs, cuda_dev, vocab, stride):
    R = 7
    full = torch.randn((R, stride), generator=sy.generator(vocab)).to(torch.bfloat16)
    full[:, vocab:] = 100.0                  # padding beyond the vocabulary must be ignored
    tgt = full[:, :vocab].float().argmax(dim=1).tolist()
    toks = [0, tgt[0], tgt[1], 5, 0, tgt[4], 9]
    cu = [0, 4, 7]
    check_against_oracle(gs, cuda_dev, full, vocab, toks, cu)


def test_bad_rows_token_range_and_counters(gs, cuda_dev):
    V = 4096
    lg = torch.randn((8, V), generator=sy.generator(3)).to(torch.bfloat16)
    tgt = lg.float().argmax(dim=1).tolist()
    toks = [0, tgt[0], -5, 0, 0, V + 3, 1, 2]
    cu = [0, 3, 3, 6, 8]                     # request 1 has no rows
    res = check_against_oracle(gs, cuda_dev, lg, V, toks, cu)
    assert res.status & oracle.STATUS_ROWS_BAD and res.status & oracle.STATUS_TOKEN_OOR
    # counters accumulate over calls
    stats = torch.zeros(5, dtype=torch.int64, device=cuda_dev)
    cu2 = [0, 3, 6, 8]
    for _ in range(3):
        run_accept(gs, cuda_dev, lg.to(cuda_dev), V, toks, cu2, stats=stats)
    ref = oracle.greedy_accept(oracle.argmax_bf16(oracle.bf16_bits(lg)), np.array(toks, np.int32), np.array(cu2), V)
    s = [int(x) for x in stats.cpu().numpy().astype(np.uint64)]
    assert s == [3 * ref.stats[k] for k in ("proposed", "evaluated", "accepted", "emitted", "steps")]
    # rows past the capacity are refused
    am, acc, bon, out, st, _ = run_accept(gs, cuda_dev, lg.to(cuda_dev), V, toks, [0, 4, 8], cap=6)
    assert acc[1] == -1 and st & gs.DEV_ROWS_BAD
    # a workspace that is too small is refused on the host
    with pytest.raises(gs.GdnError):
        gs.mtp_greedy_accept(1, 8, torch.zeros(2, dtype=torch.int32, device=cuda_dev), lg.to(cuda_dev), V, V,
                             torch.zeros(8, dtype=torch.int32, device=cuda_dev), *([torch.zeros(8, dtype=torch.int32,
                                                                                                device=cuda_dev)] * 4),
                             None, torch.zeros(8, dtype=torch.uint8, device=cuda_dev), 8,
                             torch.zeros(1, dtype=torch.int32, device=cuda_dev))
