"""The continuous-batching mix driven through ContinuousBatcher and checked,
step for step, against the oracle's scheduler, append and decode (shared by
the GPU test and the CPU test of the batcher's host logic)."""
import numpy as np
import torch

import workloads as W
from oracle import admission as OA, int8_kv as OI, paged_kv as OP, rope as OR
from tests._util import bf16_to_f64, bits, check_close, check_close_int8


class Source:
    """Seeded K/V/q of the mix, memoised per (request, layer, position)."""

    def __init__(self, case):
        self.case = case
        self.q_cache = {}
        self.kv_cache = {}

    def prompt_kv(self, rid, layer):
        return W.request_kv(self.case.seed, rid, layer, 0, int(self.case.prompt_lens[rid]))

    def token_kv(self, rid, layer, pos):
        key = (rid, layer, pos)
        if key not in self.kv_cache:
            k, v = W.request_kv(self.case.seed, rid, layer, pos, 1)
            self.kv_cache[key] = (k[0], v[0])
        return self.kv_cache[key]

    def token_q(self, rid, layer, pos):
        key = (rid, layer, pos)
        if key not in self.q_cache:
            self.q_cache[key] = W.request_q(self.case.seed, rid, layer, pos)
        return self.q_cache[key]


def run_mix(lib, dev, case, fused, cos_d, sin_d, static=False, int8=False,
            sample_every=16, sample_layers=(0, 15)):
    """Run the mix through ContinuousBatcher and, step for step, through the
    oracle's scheduler, append and decode; returns the number of steps.

    lib provides new_int8_pool (INT8 pools only); the batcher's kernels are
    whatever paged_kv_gqa_append_gb300.serving calls.
    """
    from paged_kv_gqa_append_gb300.serving import ContinuousBatcher
    src = Source(case)
    if int8:
        pool = lib.new_int8_pool(case.num_pages, dev)
        ocodes, oscales = OI.new_pools(case.num_pages)
    else:
        pool = torch.zeros((case.num_pages, 2, 8, 16, 64), dtype=torch.bfloat16, device=dev)
    cb = ContinuousBatcher(pool, case.num_layers, cos_d, sin_d, W.DEFAULT_SCALE,
                           max_slots=64, fused=fused, static=static)
    for p in case.prompt_lens:
        assert cb.submit(int(p), case.allowed_new_tokens) >= 0
    # oracle side
    osch = OA.Scheduler(case.num_pages, case.num_layers, W.MAX_BLOCKS, 64,
                        OA.Scheduler.STATIC if static else OA.Scheduler.CONTINUOUS)
    for p in case.prompt_lens:
        assert osch.submit(int(p), case.allowed_new_tokens)[0] == OA.Scheduler.OK
    opool = OP.new_pool(case.num_pages)
    cos_o, sin_o = OR.table(OR.inv_freq_llama3(), W.MAX_CONTEXT)
    orun, olen, odone = [], {}, {}
    step = 0
    checked = 0
    while cb.sched.stats()["queued"] or cb.running:
        adm = cb.admit(src.prompt_kv)
        oadm = osch.admit()
        assert adm == oadm, (step, adm, oadm)
        for rid in oadm:
            P = int(case.prompt_lens[rid])
            assert osch.grow(rid, P) == osch.OK
            for l in range(case.num_layers):
                k, v = src.prompt_kv(rid, l)
                row = np.array([osch.block_table_row(rid, l)], np.int32)
                if int8:
                    _, _, _, e = OI.append_rope_int8(ocodes, oscales, bits(k), bits(v), np.arange(P),
                                                     np.zeros(P, np.int32), row, cos_o, sin_o,
                                                     inplace=True)
                else:
                    _, _, e = OP.append_rope(opool, bits(k), bits(v), np.arange(P),
                                             np.zeros(P, np.int32), row, cos_o, sin_o, inplace=True)
                assert not e
            olen[rid], odone[rid] = P, 0
        orun += oadm
        ids, lens, out = cb.step(src.token_kv, src.token_q)
        assert ids == orun
        sample = step % sample_every == 0
        outs = out[list(sample_layers)].cpu() if sample else None
        for rid in orun:
            assert osch.grow(rid, olen[rid] + 1) == osch.OK
        for l in range(case.num_layers):
            for b, rid in enumerate(orun):
                pos = olen[rid]
                k, v = src.token_kv(rid, l, pos)
                row = np.array([osch.block_table_row(rid, l)], np.int32)
                q = src.token_q(rid, l, pos)
                if int8:
                    _, _, qr, e = OI.append_rope_int8(ocodes, oscales, bits(k[None]), bits(v[None]),
                                                      [pos], [0], row, cos_o, sin_o, bits(q[None]),
                                                      inplace=True)
                else:
                    _, qr, e = OP.append_rope(opool, bits(k[None]), bits(v[None]), [pos], [0], row,
                                              cos_o, sin_o, bits(q[None]), inplace=True)
                assert not e
                if sample and l in sample_layers:
                    got = bf16_to_f64(outs[sample_layers.index(l), b])[None]
                    if int8:
                        ref, e2 = OI.decode_int8(qr, ocodes, oscales, row, [pos + 1], W.DEFAULT_SCALE)
                        check_close_int8(got, ref, f"INT8 step {step} layer {l} request {rid}")
                    else:
                        ref, e2 = OP.decode(qr, opool, row, [pos + 1], W.DEFAULT_SCALE)
                        check_close(got, ref, f"step {step} layer {l} request {rid}")
                    assert not e2
                    checked += 1
        for rid in orun:
            olen[rid] += 1
            odone[rid] += 1
        done = cb.retire(case.decode_steps)
        odone_ids = [r for r in orun if odone[r] == case.decode_steps]
        assert done == odone_ids
        for rid in odone_ids:
            osch.finish(rid)
        orun = [r for r in orun if r not in odone_ids]
        step += 1
    assert cb.error() == 0
    assert cb.sched.events() == osch.events
    if int8:
        assert np.array_equal(pool.cpu().numpy(), OI.pack_pages(ocodes, oscales))
    else:
        assert np.array_equal(bits(pool), opool)
    assert checked >= len(case.prompt_lens)     # every request sampled at least once
    return step
