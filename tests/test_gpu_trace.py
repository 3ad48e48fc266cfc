"""GPU parity of the continuous-batching trace driver, through the C ABI.

A scaled-down version of the trace workload on the 0.1B shape: 10 requests
through 6 state slots (slots are reset and reused as requests finish), a
prefill phase every 5 decode rounds admitting up to 2 requests, one prompt
short enough to be fed through single-token steps, seeded sampling with the
adapter's defaults.  Two requests are followed by the oracle through their
whole life (prefill, then every decode round they take part in), teacher-forced
on the GPU's tokens: logits within the tolerance, and the oracle sampler, given
the GPU's fp32 logits and the request's occurrence counts and draw index,
draws the GPU's token every round.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from _harness import assert_logits_close

pytestmark = pytest.mark.gpu


def test_trace_driver_against_oracle():
    import torch
    import recurrent_decode_gb300 as rd
    from recurrent_decode_gb300.trace import Request, run_trace
    dims = synth.Dims("0.1b")
    W = synth.make_weights("0.1b")
    ctx = rd.Rwkv7(dims, 6)
    ctx.set_weights(W)
    lens = synth.trace_requests(10, 12, 40, 8, 20, seed=5)
    lens[3] = (6, lens[3][1])  # decode-fed prompt (shorter than min_forward_seq_len)
    reqs = []
    for i, (pl, ol) in enumerate(lens):
        sp = dict(temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0, penalty_decay=0.996,
                  seed=synth.SAMPLING_SEED_BASE + i, greedy=False)
        reqs.append(Request(prompt=synth.prompt_tokens(dims.vocab, 1, pl, seed=100 + i)[0], n_out=ol, sampling=sp))
    tracked = [3, 8]
    oracle.set_threads(os.cpu_count() or 1)
    m = oracle.Model(W, dims)
    sts = {i: m.new_state() for i in tracked}
    for i in tracked:
        sts[i].prefill_chunked(reqs[i].prompt[:-1], want_logits=False)
    occ = {i: np.zeros(dims.vocab, np.float32) for i in tracked}
    seen = {i: 0 for i in tracked}

    def on_round(slots, toks, logits, got):
        rows = None
        for i in tracked:
            r = reqs[i]
            if r.slot < 0 or r.t_done >= 0 or r.slot not in slots.tolist():
                continue
            if rows is None:
                rows = logits.cpu().numpy()
            k = slots.tolist().index(r.slot)
            ref = sts[i].step(int(toks[k]))
            assert_logits_close(rows[k], ref, f"request {i} token {seen[i]}")
            tok, _ = oracle.sample(rows[k], occ[i], r.sampling, seen[i])
            assert tok == int(got[k]), (i, seen[i], tok, int(got[k]))
            seen[i] += 1

    stats = run_trace(ctx, reqs, 6, decode_prefill_ratio=5, max_prefill_count=2, on_round=on_round,
                      want_logits=True)
    assert all(len(r.out) == r.n_out for r in reqs)
    assert seen == {i: reqs[i].n_out for i in tracked}
    assert stats.generated == sum(r.n_out for r in reqs)
    assert stats.decode_fed_tokens == 5 and stats.prefill_tokens == sum(len(r.prompt) - 1 for r in reqs) - 5
    ctx.close()
