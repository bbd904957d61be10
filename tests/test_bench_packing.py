"""The end-to-end arm's packed input buffer (host side, no GPU): every
layer's row inputs and the logits get disjoint, 256-byte-aligned byte ranges,
and the typed views written through one buffer read back exactly."""
import types

import torch

import bench


def _fake_bench(layers=3, rows=5, h_qk=2, h_v=4, d=8, vocab=37):
    from dataclasses import dataclass

    @dataclass
    class R:
        q: torch.Tensor
        k: torch.Tensor
        v: torch.Tensor
        g: torch.Tensor
        beta: torch.Tensor

    g = torch.Generator().manual_seed(0)
    mk = lambda *s, dt=torch.float32: torch.randn(*s, generator=g).to(dt)
    ring = [[R(mk(rows, h_qk, d, dt=torch.bfloat16), mk(rows, h_qk, d, dt=torch.bfloat16),
               mk(rows, h_v, d, dt=torch.bfloat16), mk(rows, h_v), mk(rows, h_v)) for _ in range(layers)]]
    return types.SimpleNamespace(rows=ring, logits=[mk(rows, vocab, dt=torch.bfloat16)])


def test_pieces_are_disjoint_aligned_and_cover_every_tensor():
    b = _fake_bench()
    pieces, total = bench._packed_layout(b)
    assert len(pieces) == 3 * 5 + 1
    end = 0
    for off, dt, shape in pieces:
        assert off % 256 == 0 and off >= end
        n = 1
        for s in shape:
            n *= s
        end = off + n * torch.empty((), dtype=dt).element_size()
    assert end <= total and total % 256 == 0


def test_views_round_trip_through_one_buffer():
    b = _fake_bench()
    pieces, total = bench._packed_layout(b)
    buf = torch.zeros((total,), dtype=torch.uint8)
    src = [x for r in b.rows[0] for x in (r.q, r.k, r.v, r.g, r.beta)] + [b.logits[0]]
    for v, x in zip(bench._views(buf, pieces), src):
        assert v.dtype == x.dtype and v.shape == x.shape
        v.copy_(x)
    copy = buf.clone()
    for v, x in zip(bench._views(copy, pieces), src):
        assert torch.equal(v, x)
