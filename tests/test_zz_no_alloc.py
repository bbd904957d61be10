"""The allocation-free accept entry point (mtp_greedy_accept_noalloc) gives
the same results as mtp_greedy_accept with a caller workspace.

Some callers cannot allocate device memory where they accept drafts (a plugin
whose host engine owns all device memory, a loop that cannot afford a
cudaMalloc); this variant uses a fixed scratch array inside the library.
Two calls in a row check that the scratch's leftover contents do not leak
into a later result.  The file sorts last so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import gdnsynth as sy
from gpu_util import build_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs(cuda_dev):
    build_lib()
    from speculative_decoding_hybrid_gb300 import binding
    return binding


def _case(dev, seed, ks, vocab):
    R = sum(k + 1 for k in ks)
    lg, tgt = sy.logits(sy.generator(seed), R, vocab, 2.0)
    toks = sum(sy.drafts(sy.generator(seed + 1), tgt.tolist(), ks, vocab, 0.85), [])
    cu = [0]
    for k in ks:
        cu.append(cu[-1] + k + 1)
    return (lg.to(dev), torch.tensor(toks, dtype=torch.int32, device=dev),
            torch.tensor(cu, dtype=torch.int32, device=dev), R)


def _outputs(dev, B, R):
    z = lambda n: torch.full((max(n, 1),), -9, dtype=torch.int32, device=dev)
    return dict(argmax=z(R), accept_len=z(B), bonus=z(B), out_tokens=z(R),
                stats=torch.zeros(5, dtype=torch.int64, device=dev), status=torch.zeros(1, dtype=torch.int32,
                                                                                         device=dev))


def test_noalloc_accept_matches_the_workspace_call(gs, cuda_dev):
    cases = [(11, [3, 0, 2, 3, 1, 3, 2, 3, 3, 1, 0, 2, 3, 3, 2, 1], 151936),   # ragged, 16 requests
             (12, [3] * 8, 151936)]                                              # next call, new inputs
    for seed, ks, vocab in cases:
        lg, toks, cu, R = _case(cuda_dev, seed, ks, vocab)
        B = len(ks)
        ref = _outputs(cuda_dev, B, R)
        ws_bytes = gs.mtp_accept_workspace_bytes(R, vocab)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda_dev)
        gs.mtp_greedy_accept(B, R, cu, lg, vocab, lg.stride(0), toks, ref["argmax"], ref["accept_len"],
                             ref["bonus"], ref["out_tokens"], ref["stats"], ws, ws_bytes, ref["status"])
        got = _outputs(cuda_dev, B, R)
        gs.mtp_greedy_accept_noalloc(B, R, cu, lg, vocab, lg.stride(0), toks, got["argmax"], got["accept_len"],
                                     got["bonus"], got["out_tokens"], got["stats"], got["status"])
        torch.cuda.synchronize()
        for key in ref:
            assert torch.equal(ref[key], got[key]), key


def test_noalloc_refuses_requests_beyond_its_scratch(gs, cuda_dev):
    # 65537 rows need more than the 512 KiB of partial maxima the scratch holds
    rows = 70000
    assert gs.mtp_accept_workspace_bytes(rows, 151936) > 512 * 1024
    z = torch.zeros(8, dtype=torch.int32, device=cuda_dev)
    with pytest.raises(gs.GdnError) as e:
        gs.mtp_greedy_accept_noalloc(1, rows, z, z, 151936, 151936, z, z, z, z, z, None, z)
    assert e.value.status == gs.GDN_ERR_WORKSPACE
