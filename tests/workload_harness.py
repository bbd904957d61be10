"""Runs a multi-step verification workload through the library and, beside
it, through the oracle (planner model, greedy choice, acceptance rule and
FP64 recurrence), comparing every step."""
import numpy as np
import torch

import gdnsynth as sy
import oracle
from gpu_util import noted, out_err, state_err


class Workload:
    def __init__(self, spec: sy.Spec, steps: int, fp_requests, dev, gen_device=None):
        from speculative_decoding_hybrid_gb300 import binding as gs
        from speculative_decoding_hybrid_gb300.step import DecodeLoop, LayerRows, VerifyStep
        self.gs = gs
        self.spec = spec
        self.steps = steps
        self.dev = dev
        gdev = dev if gen_device is None else gen_device
        d = spec.dims
        self.cap = spec.batch * (spec.k_max + 1)
        self.ks = sy.k_table(spec, steps)
        slot_of, free, ref = sy.initial_slots(spec)
        self.slot_of0 = list(slot_of)
        # native pool and the oracle's model, set up identically
        order = list(free)
        taken = []
        for s in slot_of:
            if s not in taken:
                taken.append(s)
        full_order = taken + order
        self.pool_c = gs.Pool(spec.num_slots, full_order)
        self.pool_m = oracle.PoolModel(spec.num_slots, full_order)
        seen = set()
        for s in slot_of:
            if s in seen:
                self.pool_c.share(s)
                self.pool_m.share(s)
            else:
                assert self.pool_c.alloc() == s
                assert self.pool_m.alloc() == (0, s)
                seen.add(s)
        pool = torch.empty((spec.num_slots, spec.layers, d.h_v, d.d_v, d.d_k), dtype=torch.float32, device=dev)
        sy.pool_state(spec, dev, out=pool)
        self.vs = VerifyStep(gs.dims(d.h_qk, d.h_v, d.d_k, d.d_v), spec.layers, spec.num_slots, self.cap,
                             spec.batch, spec.vocab, dev, pool=pool)
        self.loop = DecodeLoop(self.vs, slot_of, self.pool_c, k_max=spec.k_max)
        self.ring_rows = [[sy.ring_rows(spec, l, i, self.cap, gdev) for l in range(spec.layers)]
                          for i in range(spec.ring)]
        self.ring_rows_dev = [[LayerRows(*(t.to(dev) for t in (r.q, r.k, r.v, r.g, r.beta))) for r in ring]
                              for ring in self.ring_rows]
        self.ring_rows_host = [[[t.detach().to("cpu") for t in (r.q, r.k, r.v, r.g, r.beta)] for r in ring]
                               for ring in self.ring_rows]
        self.ring_logits = []
        self.ring_targets = []
        self.ring_argmax = []
        for i in range(spec.ring):
            lg, tgt = sy.ring_logits(spec, i, self.cap, gdev)
            self.ring_logits.append(lg.to(dev))
            self.ring_targets.append(tgt.tolist())
            self.ring_argmax.append(oracle.argmax_bf16(oracle.bf16_bits(lg)))
        self.fp = list(fp_requests)
        # oracle states of the requests followed in FP64: [layers][h_v, d_v, d_k]
        self.S = {r: pool[slot_of[r]].detach().cpu().numpy().astype(np.float64) for r in self.fp}
        self.slots_m = list(slot_of)
        self.cur_len_m = [1] * spec.batch
        self.worst_state = 0.0
        self.worst_out = 0.0

    def step(self, s):
        gs, spec, loop, vs = self.gs, self.spec, self.loop, self.vs
        B = spec.batch
        ks = self.ks[s].tolist()
        p = loop.plan_step(ks)
        reqs_m = [oracle.Req(oracle.DECODE, ks[i], cur_len=self.cur_len_m[i], slot=self.slots_m[i])
                  for i in range(B)]
        pm = oracle.plan_transaction(reqs_m, self.cap, B, spec.k_max, self.pool_m)
        assert pm.status == 0
        assert p.dec_cu == pm.dec_cu and p.dec_src == pm.dec_src and p.dec_dst == pm.dec_dst and p.k == pm.k
        ring = s % spec.ring
        cu = pm.dec_cu
        total = cu[-1]
        drafts = sy.step_drafts(spec, s, pm.k, self.ring_targets[ring])
        tokens = [t for d in drafts for t in d]
        tok_d = torch.tensor(tokens + [0] * (self.cap - total), dtype=torch.int32, device=self.dev)
        shared_before = {}
        for i in range(B):
            if pm.dst[i] != pm.src[i]:
                shared_before[pm.src[i]] = vs.pool[pm.src[i]].clone()
        loop.upload_tables()
        loop.run(self.ring_rows_dev[ring], self.ring_logits[ring], tok_d)
        acc, bon, out = loop.readback()
        assert int(vs.status.item()) == 0
        # integers: argmax, acceptance, bonus, emitted tokens -- bit-exact for every request
        am_ref = self.ring_argmax[ring][:total]
        assert np.array_equal(vs.argmax[:total].cpu().numpy(), am_ref)
        res = oracle.greedy_accept(am_ref, np.array(tokens, np.int32), np.array(cu), spec.vocab)
        assert np.array_equal(acc.numpy(), res.accept_len)
        assert np.array_equal(bon.numpy(), res.bonus)
        assert np.array_equal(out.numpy()[:total], res.out_tokens)
        # commit: every (request, layer) slot equals its accepted checkpoint, bit for bit
        for i in range(B):
            assert torch.equal(vs.pool[pm.dst[i]], vs.ckpt[:, cu[i] + int(res.accept_len[i])])
        # shared (copy-on-write) sources were never written
        for src, snap in shared_before.items():
            assert torch.equal(vs.pool[src], snap)
        # FP64 recurrence for the followed requests
        host = self.ring_rows_host[ring]
        units, keys = [], []
        for r in self.fp:
            a, b = cu[r], cu[r + 1]
            for l in range(spec.layers):
                q, k, v, g, beta = host[l]
                units += oracle.head_units(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], self.S[r][l])
                keys.append((r, l))
        _, o_list, ck_list = oracle.recurrent_units(units, want_ckpt=True)
        H = spec.dims.h_v
        o_gpu = vs.o.detach().cpu()
        for n, (r, l) in enumerate(keys):
            a, b = cu[r], cu[r + 1]
            j = int(res.accept_len[r])
            o_ref = np.stack(o_list[n * H:(n + 1) * H], axis=1)
            self.worst_out = max(self.worst_out, out_err(o_gpu[l, a:b], o_ref))
            self.S[r][l] = np.stack([ck_list[n * H + h][j] for h in range(H)])
        assert noted("workload %s: outputs" % self.spec.name, self.worst_out) <= 1.0, self.worst_out
        loop.finish(acc)
        assert oracle.pool_apply(self.pool_m, reqs_m, pm) == 0
        for i in range(B):
            self.slots_m[i] = pm.dst[i]
            self.cur_len_m[i] += int(res.accept_len[i]) + 1
        assert list(self.pool_c.refcount) == self.pool_m.ref
        assert self.pool_c.free_list() == self.pool_m.free
        return res

    def check_states(self):
        for r in self.fp:
            gpu = self.vs.pool[self.slots_m[r]].detach().cpu().numpy()
            e = state_err(gpu, self.S[r])
            self.worst_state = max(self.worst_state, e)
        assert noted("workload %s: state" % self.spec.name, self.worst_state) <= 1.0, self.worst_state
