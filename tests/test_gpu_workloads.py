"""GPU parity on the named decode workloads, through the C ABI.

- The 0.1B-shape workload in full: 32 slots, 64-token prompts (63 consumed by
  batched steps, the 64th by the first decode step), 256 sampled decode steps
  with the adapter's sampling defaults (temperature 1, top_p 0.3, frequency 1,
  penalty decay 0.996) and per-slot seeds.  Two slots are followed by the
  oracle, teacher-forced on the GPU's tokens: logits stay within the tolerance
  for all 256 steps, and the oracle's sampler, given the GPU's fp32 logits, the
  same occurrence counts and draw counters, draws the GPU's token every step.
- The 2.9B and 7.2B shapes at their benchmark batch (64 and 256 slots), in the
  benchmark's launch configuration (CUDA-graph replay of the fused step) and
  sampling (2.9B greedy; 7.2B the adapter's defaults, top_p 0.3, seeded per
  slot): 8-token prompts, 8 decode steps; three rows are followed by the
  oracle, teacher-forced, and checked within the tolerance; greedy tokens are
  the GPU logits' argmax and the oracle's up to near ties, sampled tokens are
  the oracle sampler's draw on the GPU's logits with the same occurrence counts
  and draw index.

Tolerances as in _harness: logits max-abs <= 2e-2, cosine >= 0.9999; greedy
tokens equal to the oracle's argmax unless the oracle's margin is within it.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from _harness import assert_logits_close, greedy_consistent

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def test_sampled_workload_0p1b_full():
    torch = _torch()
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    wl = synth.WORKLOADS["0.1b"]
    dims = synth.Dims(wl["shape"])
    B, P, steps = wl["B"], wl["prompt"], wl["steps"]
    W = synth.make_weights(wl["shape"])
    ctx = rd.Rwkv7(dims, B)
    ctx.set_weights(W)
    params = []
    for s in range(B):
        sp = dict(temperature=wl["temperature"], top_p=wl["top_p"], top_k=wl["top_k"], presence=wl["presence"],
                  frequency=wl["frequency"], penalty_decay=wl["penalty_decay"], seed=synth.SAMPLING_SEED_BASE + s,
                  greedy=False)
        ctx.set_sampling(s, **sp)
        params.append(sp)
    prompts = synth.prompt_tokens(dims.vocab, B, P)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    dprompts = torch.from_numpy(prompts).to(dev)
    for t in range(P - 1):
        ctx.decode_step(slots, dprompts[:, t].contiguous())
    tracked = [3, 26]
    oracle.set_threads(os.cpu_count() or 1)
    m = oracle.Model(W, dims)
    sts = [m.new_state() for _ in tracked]
    for st, s in zip(sts, tracked):
        st.prefill_chunked(prompts[s, :P - 1], want_logits=False)
    occ = [np.zeros(dims.vocab, np.float32) for _ in tracked]
    cur = dprompts[:, P - 1].contiguous()
    logits = torch.empty(B, dims.vocab, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    for step in range(steps):
        ctx.decode_step(slots, cur, logits, nxt)
        ctx.synchronize()
        tok_in = cur.cpu().numpy()
        got = nxt.cpu().numpy()
        rows = logits[tracked].cpu().numpy()
        for k, s in enumerate(tracked):
            ref = sts[k].step(int(tok_in[s]))
            assert_logits_close(rows[k], ref, f"slot {s} step {step}")
            tok, _ = oracle.sample(rows[k], occ[k], params[s], step)
            assert tok == int(got[s]), (s, step, tok, int(got[s]))
        cur = nxt.clone()
    ctx.close()


@pytest.mark.parametrize("shape", ["2.9b", "7.2b"])
def test_full_shape_bench_batch_teacher_forced(shape):
    torch = _torch()
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    dims = synth.Dims(shape)
    wl = synth.WORKLOADS[shape]
    B = wl["B"]
    W = synth.make_weights(shape)
    ctx = rd.Rwkv7(dims, B)
    ctx.set_weights(W)
    ctx.set_mode(0)  # the benchmark's configuration: graph replay
    greedy = bool(wl.get("greedy"))
    params = []
    for s in range(B):
        sp = dict(greedy=True) if greedy else dict(
            temperature=wl["temperature"], top_p=wl["top_p"], top_k=wl["top_k"], presence=wl["presence"],
            frequency=wl["frequency"], penalty_decay=wl["penalty_decay"], seed=synth.SAMPLING_SEED_BASE + s,
            greedy=False)
        ctx.set_sampling(s, **sp)
        params.append(sp)
    P = 8
    prompts = synth.prompt_tokens(dims.vocab, B, P, seed=31)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    dprompts = torch.from_numpy(prompts).to(dev)
    for t in range(P - 1):
        ctx.decode_step(slots, dprompts[:, t].contiguous())
    tracked = [0, B // 2 + 1, B - 1]
    oracle.set_threads(os.cpu_count() or 1)
    m = oracle.Model(W, dims)
    sts = [m.new_state() for _ in tracked]
    for st, s in zip(sts, tracked):
        st.prefill_chunked(prompts[s, :P - 1], want_logits=False)
    occ = [np.zeros(dims.vocab, np.float32) for _ in tracked]
    cur = dprompts[:, P - 1].contiguous()
    logits = torch.empty(B, dims.vocab, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    for step in range(8):
        ctx.decode_step(slots, cur, logits, nxt)
        ctx.synchronize()
        tok_in = cur.cpu().numpy()
        got = nxt.cpu().numpy()
        rows = logits[tracked].cpu().numpy()
        for k, s in enumerate(tracked):
            ref = sts[k].step(int(tok_in[s]))
            assert_logits_close(rows[k], ref, f"{shape} slot {s} step {step}")
            if greedy:
                assert int(got[s]) == int(np.argmax(rows[k]))
                assert greedy_consistent(int(got[s]), ref, f"{shape} slot {s} step {step}")
            else:
                tok, _ = oracle.sample(rows[k], occ[k], params[s], step)
                assert tok == int(got[s]), (shape, s, step, tok, int(got[s]))
        cur = nxt.clone()
    ctx.close()
