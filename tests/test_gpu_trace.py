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


def _shared_prefix_requests(dims, n, prefix_len, seed):
    """n requests whose prompts share their first prefix_len tokens, then differ."""
    prefix = synth.prompt_tokens(dims.vocab, 1, prefix_len, seed=seed)[0]
    lens = synth.trace_requests(n, 15, 40, 4, 8, seed=seed + 1)
    reqs = []
    for i, (pl, ol) in enumerate(lens):
        tail = synth.prompt_tokens(dims.vocab, 1, pl, seed=seed + 10 + i)[0]
        sp = dict(temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0, penalty_decay=0.996,
                  seed=synth.SAMPLING_SEED_BASE + i, greedy=False)
        reqs.append((np.concatenate([prefix, tail]).astype(np.int32), ol, sp))
    return reqs


def _run(ctx, specs, n_slots, **kw):
    from recurrent_decode_gb300.trace import Request, run_trace
    reqs = [Request(prompt=p, n_out=o, sampling=dict(sp)) for p, o, sp in specs]
    seen = {}

    def on_round(slots, toks, logits, got):
        rows = logits.cpu().numpy()
        for k, s in enumerate(slots.tolist()):
            i = next(j for j, r in enumerate(reqs) if r.slot == s and r.status == "running")
            seen.setdefault(i, []).append((rows[k].copy(), int(got[k])))

    stats = run_trace(ctx, reqs, n_slots, decode_prefill_ratio=5, max_prefill_count=2, on_round=on_round,
                      want_logits=True, **kw)
    return reqs, seen, stats


def test_prefix_cache_results_bit_identical():
    """Requests sharing a 600-token prompt prefix: with the prefix-state cache
    every request after the first restores the state after 512 tokens (two
    256-token blocks) and prefills only the rest, yet every logit and sampled
    token equals the uncached run bit for bit (the restored state is a byte
    copy, and the rest is prefilled in the same chunks as without the cache)."""
    import recurrent_decode_gb300 as rd
    from recurrent_decode_gb300.prefix_cache import PrefixStateCache
    dims = synth.Dims("0.1b")
    W = synth.make_weights("0.1b")
    specs = _shared_prefix_requests(dims, 6, 600, seed=40)
    n_run, n_cache = 3, 4
    ctx = rd.Rwkv7(dims, n_run + n_cache)
    ctx.set_weights(W)
    ref_reqs, ref_seen, ref_stats = _run(ctx, specs, n_run)
    for s in range(n_run + n_cache):
        ctx.slot_reset(s)
    cache = PrefixStateCache(ctx, range(n_run, n_run + n_cache))
    reqs, seen, stats = _run(ctx, specs, n_run, prefix_cache=cache)
    assert [r.out for r in reqs] == [r.out for r in ref_reqs]
    assert seen.keys() == ref_seen.keys()
    for i in seen:
        assert len(seen[i]) == len(ref_seen[i])
        for (a, ta), (b, tb) in zip(seen[i], ref_seen[i]):
            assert ta == tb
            assert np.array_equal(a, b), f"request {i}: logits differ with the prefix cache"
    # the first request stores states at 256, 512 and its full body; the other
    # five restore the 512-token prefix (their full bodies differ)
    assert cache.hits == 5 and stats.prefix_hit_tokens == 5 * 512
    assert [r.prefix_hit for r in reqs] == [0] + [512] * 5
    assert stats.prefill_tokens == ref_stats.prefill_tokens - 5 * 512
    ctx.close()


def test_abort_ends_only_that_request():
    """Request-level abort: request 1 is aborted at round 3 while running and
    request 4 before it is admitted; both free their slot, and every other
    request's tokens and logits equal the run without aborts bit for bit (a
    slot's results do not depend on the other rows of its step)."""
    import recurrent_decode_gb300 as rd
    dims = synth.Dims("0.1b")
    W = synth.make_weights("0.1b")
    specs = _shared_prefix_requests(dims, 7, 20, seed=70)
    ctx = rd.Rwkv7(dims, 3)
    ctx.set_weights(W)
    ref_reqs, ref_seen, _ = _run(ctx, specs, 3)
    reqs, seen, stats = _run(ctx, specs, 3, abort_at={1: 3, 4: 0})
    assert reqs[1].status == "aborted" and 0 < len(reqs[1].out) <= 3
    assert reqs[4].status == "aborted" and reqs[4].out == [] and reqs[4].slot == -1
    assert stats.aborted == 2
    for i, r in enumerate(reqs):
        if i in (1, 4):
            continue
        assert r.status == "finished" and r.out == ref_reqs[i].out, i
        for (a, _), (b, _) in zip(seen[i], ref_seen[i]):
            assert np.array_equal(a, b), f"request {i}: logits changed by another request's abort"
    for (a, _), (b, _) in zip(seen[1], ref_seen[1]):  # the aborted request's rounds before the abort
        assert np.array_equal(a, b)
    ctx.close()
