"""GPU parity of the decode path against the CPU oracle, through the C ABI.

Tolerances (fp16 weights, fp32 state): logits max-abs <= 2e-2, cosine >= 0.9999;
greedy tokens equal to the oracle argmax unless the oracle's margin is within
the tolerance; sampled tokens bit-exact given the same logits and seed."""
import numpy as np
import pytest

import oracle
import synth
from _harness import assert_logits_close, gpu_ctx, greedy_consistent, oracle_states

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


@pytest.fixture(scope="module")
def tiny():
    return synth.make_weights("tiny")


@pytest.mark.parametrize("mode", [2, 1, 0])
def test_tiny_workload_greedy(tiny, mode):
    """Tiny config: B=1, 8-token prompt (prefill 7, first decode consumes the 8th),
    16 greedy decode steps; oracle teacher-forced on the GPU's tokens."""
    torch = _torch()
    ctx, W, dims = gpu_ctx("tiny", 1, tiny, mode)
    ctx.set_sampling(0, greedy=True)
    prompt = synth.prompt_tokens(dims.vocab, 1, 8)[0]
    _, (st,) = oracle_states(W, dims, 1)
    st.prefill_chunked(prompt[:-1], want_logits=False)
    dev = torch.device("cuda")
    ctx.prefill_seq(0, torch.from_numpy(prompt[:-1]).to(dev))
    slots = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = torch.tensor([int(prompt[-1])], dtype=torch.int32, device=dev)
    logits = torch.empty(1, dims.vocab, device=dev)
    nxt = torch.empty(1, dtype=torch.int32, device=dev)
    cur = int(prompt[-1])
    for s in range(16):
        ctx.decode_step(slots, tok, logits, nxt)
        ctx.synchronize()
        ref = st.step(cur)
        g = logits[0].cpu().numpy()
        assert_logits_close(g, ref, f"mode {mode} step {s}")
        t = int(nxt.item())
        assert t == int(np.argmax(g))
        assert greedy_consistent(t, ref)
        cur = t
        tok.fill_(t)


@pytest.mark.parametrize("mode", [2, 0])
def test_tiny_ragged_batch_permuted_slots(tiny, mode):
    """B=37 of 48 slots (three N tiles of 16 with a ragged tail), slots in a
    random order, per-slot prompts of different lengths, 4 decode steps."""
    torch = _torch()
    dev = torch.device("cuda")
    ctx, W, dims = gpu_ctx("tiny", 48, tiny, mode)
    g = np.random.default_rng(11)
    slots = g.permutation(48)[:37].astype(np.int32)
    lens = g.integers(1, 6, size=37)
    prompts = synth.prompt_tokens(dims.vocab, 37, 6, seed=21)
    m, sts = oracle_states(W, dims, 37)
    for i, s in enumerate(slots):
        p = prompts[i][:lens[i]]
        if len(p) > 1:
            ctx.prefill_seq(int(s), torch.from_numpy(p[:-1].copy()).to(dev))
            sts[i].prefill_chunked(p[:-1], want_logits=False)
    cur = np.array([prompts[i][lens[i] - 1] for i in range(37)], np.int32)
    d_slots = torch.from_numpy(slots).to(dev)
    logits = torch.empty(37, dims.vocab, device=dev)
    for step in range(4):
        ctx.decode_step(d_slots, torch.from_numpy(cur).to(dev), logits)
        ctx.synchronize()
        got = logits.cpu().numpy()
        for i in range(37):
            assert_logits_close(got[i], sts[i].step(int(cur[i])), f"slot {slots[i]} step {step}")
        cur = synth.prompt_tokens(dims.vocab, 37, 1, seed=100 + step)[:, 0]


def test_wide_batch_graph_vs_cuda_core(tiny):
    """150 of 160 slots (an MMA N side of 160, a ragged tail of the 16-wide
    padding): the tensor-core step replayed as a graph (mode 0) matches the
    CUDA-core cross-check (mode 2) within the tolerance on every row and the
    oracle on a sampled row; the states written back match too."""
    torch = _torch()
    dev = torch.device("cuda")
    g = np.random.default_rng(5)
    slots = g.permutation(160)[:150].astype(np.int32)
    outs, states = [], []
    for mode in (2, 0):
        ctx, W, dims = gpu_ctx("tiny", 160, tiny, mode)
        lg = torch.empty(150, dims.vocab, device=dev)
        res = []
        for t in range(3):
            toks = synth.prompt_tokens(dims.vocab, 150, 1, seed=80 + t)[:, 0]
            ctx.decode_step(torch.from_numpy(slots).to(dev), torch.from_numpy(toks).to(dev), lg)
            res.append(lg.cpu().numpy().copy())
        ctx.synchronize()
        outs.append(res)
        states.append(ctx.get_state(int(slots[7])))
        ctx.close()
    for t in range(3):
        for i in range(150):
            assert_logits_close(outs[1][t][i], outs[0][t][i], f"step {t} row {i}")
    for a, b in zip(states[0], states[1]):
        np.testing.assert_allclose(a, b, atol=1e-3, rtol=1e-3)
    m, (st,) = oracle_states(tiny, synth.Dims("tiny"), 1)
    for t in range(3):
        ref = st.step(int(synth.prompt_tokens(1024, 150, 1, seed=80 + t)[7, 0]))
        assert_logits_close(outs[1][t][7], ref, f"oracle step {t}")


def test_2p9b_layer_sizes_graph_vs_cuda_core():
    """The 2.9B layer sizes (d=2560, F=10240, V=65536, LoRA 96/96/64/320) cut to
    2 layers, B=64 of 72 permuted slots, 3 steps: k-split projections whose
    slabs the consumers add, the fused r, k, v + LoRA launch (LoRA-down tiles
    split in four and finished by their last split, LoRA-up after the
    in-kernel counter), the 512-tile head.  Every row of the graph-replayed
    tensor-core step (mode 0) matches the CUDA-core cross-check (mode 2) within
    the tolerance and four rows match the oracle."""
    torch = _torch()
    dev = torch.device("cuda")
    W = synth.make_weights("2.9b", n_layer=2)
    dims = synth.Dims("2.9b", 2)
    slots = np.random.default_rng(9).permutation(72)[:64].astype(np.int32)
    outs = []
    for mode in (2, 0):
        ctx, _, _ = gpu_ctx("2.9b", 72, W, mode, n_layer=2)
        lg = torch.empty(64, dims.vocab, device=dev)
        res = []
        for t in range(3):
            toks = synth.prompt_tokens(dims.vocab, 64, 1, seed=90 + t)[:, 0]
            ctx.decode_step(torch.from_numpy(slots).to(dev), torch.from_numpy(toks).to(dev), lg)
            ctx.synchronize()
            res.append(lg.cpu().numpy().copy())
        outs.append(res)
        ctx.close()
    for t in range(3):
        for i in range(64):
            assert_logits_close(outs[1][t][i], outs[0][t][i], f"step {t} row {i}")
    rows = [0, 17, 40, 63]
    m, sts = oracle_states(W, dims, len(rows))
    for t in range(3):
        toks = synth.prompt_tokens(dims.vocab, 64, 1, seed=90 + t)[:, 0]
        for k, i in enumerate(rows):
            assert_logits_close(outs[1][t][i], sts[k].step(int(toks[i])), f"oracle step {t} row {i}")


def test_fused_and_three_launch_lora_paths_bit_identical_2p9b():
    """At the 2.9B layer sizes the LoRA-down tiles are k-split.  A narrow batch
    runs r, k, v and both LoRA stages as one two-phase launch (each tile's
    last split adds the slabs); a batch wider than half the SMs runs them as
    three launches (the finalize kernel adds them).  Both add the same slabs
    in the same order with the same activations, so a slot fed the same
    tokens gives bit-identical logits either way."""
    torch = _torch()
    dev = torch.device("cuda")
    W = synth.make_weights("2.9b", n_layer=2)
    dims = synth.Dims("2.9b", 2)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    wide = min(256, nsm // 2 + 24)
    ctx, _, _ = gpu_ctx("2.9b", wide + 1, W, 0, n_layer=2)
    if ctx.step_kernel_count(1, False) == ctx.step_kernel_count(wide, False):
        ctx.close()
        pytest.skip("both batch widths take the same path on this device")
    toks = synth.prompt_tokens(dims.vocab, wide + 1, 3, seed=77)
    one = torch.empty(1, dims.vocab, device=dev)
    many = torch.empty(wide, dims.vocab, device=dev)
    batch_slots = torch.arange(1, wide + 1, dtype=torch.int32, device=dev)
    pos = wide // 2
    for t in range(3):
        ctx.decode_step(torch.zeros(1, dtype=torch.int32, device=dev),
                        torch.tensor([int(toks[0, t])], dtype=torch.int32, device=dev), one)
        bt = toks[1:wide + 1, t].copy()
        bt[pos] = toks[0, t]
        ctx.decode_step(batch_slots, torch.from_numpy(bt).to(dev), many)
        ctx.synchronize()
        assert torch.equal(one[0], many[pos]), f"step {t}"
    ctx.close()


def test_batch_beyond_one_fused_step(tiny):
    """B = 300 slots (more than one fused step of 256): the step runs as two
    sub-steps; rows from both match the oracle, and the host-buffer entry point
    gives the device-buffer path's logits and tokens bit for bit."""
    torch = _torch()
    dev = torch.device("cuda")
    B = 300
    ctxs = []
    for _ in range(2):
        ctx, W, dims = gpu_ctx("tiny", B, tiny, 0)
        for s in range(B):
            ctx.set_sampling(s, greedy=True)
        ctxs.append(ctx)
    slots = np.random.default_rng(17).permutation(B).astype(np.int32)
    rows = [0, 131, 255, 256, 299]
    m, sts = oracle_states(tiny, dims, len(rows))
    lg = torch.empty(B, dims.vocab, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    h_lg = np.zeros((B, dims.vocab), np.float32)
    h_nx = np.zeros(B, np.int32)
    toks = synth.prompt_tokens(dims.vocab, B, 1, seed=140)[:, 0]
    for step in range(2):
        ctxs[0].decode_step(torch.from_numpy(slots).to(dev), torch.from_numpy(toks).to(dev), lg, nxt)
        ctxs[0].synchronize()
        ctxs[1].decode_step_host(slots, toks, h_lg, h_nx)
        got = lg.cpu().numpy()
        assert np.array_equal(got, h_lg) and np.array_equal(nxt.cpu().numpy(), h_nx)
        for k, i in enumerate(rows):
            assert_logits_close(got[i], sts[k].step(int(toks[i])), f"step {step} row {i}")
        toks = nxt.cpu().numpy().copy()
    for ctx in ctxs:
        ctx.close()


def _zero(a):
    a[...] = 0


def test_sparse_value_projection():
    """Channel-mix key weights zero: ReLU^2 input is zero everywhere, the value
    projection skips every block (union 0 of all) and the logits still match the
    oracle's dense channel mix; with the seeded weights nearly every block is
    read."""
    torch = _torch()
    dev = torch.device("cuda")
    dims = synth.Dims("tiny")
    ov = {f"blocks.{l}.ffn.key": _zero for l in range(dims.n_layer)}
    for W, expect_zero in ((synth.make_weights("tiny", overrides=ov), True), (synth.make_weights("tiny"), False)):
        ctx, _, _ = gpu_ctx("tiny", 4, W, 0)
        m, sts = oracle_states(W, dims, 3)
        lg = torch.empty(3, dims.vocab, device=dev)
        ctx.ffn_union_stats()
        for t in range(3):
            toks = synth.prompt_tokens(dims.vocab, 3, 1, seed=130 + t)[:, 0]
            ctx.decode_step(torch.arange(3, dtype=torch.int32, device=dev), torch.from_numpy(toks).to(dev), lg)
            ctx.synchronize()
            got = lg.cpu().numpy()
            for i in range(3):
                assert_logits_close(got[i], sts[i].step(int(toks[i])), f"step {t} row {i}")
        nz, tot = ctx.ffn_union_stats()
        assert tot == 3 * dims.n_layer * (dims.d_ffn // 64)
        if expect_zero:
            assert nz == 0
        else:
            assert nz >= 0.9 * tot
        ctx.close()


def test_batch_invariance_bit_exact(tiny):
    """A slot's logits do not depend on B or on its position in the batch."""
    torch = _torch()
    dev = torch.device("cuda")
    ctx, W, dims = gpu_ctx("tiny", 40, tiny, 0)
    toks = synth.prompt_tokens(dims.vocab, 40, 3, seed=5)
    one = torch.empty(1, dims.vocab, device=dev)
    many = torch.empty(37, dims.vocab, device=dev)
    batch_slots = torch.arange(3, 40, dtype=torch.int32, device=dev)
    for t in range(3):
        # slot 0 alone; slot 20 inside a batch of 37, both fed the same tokens
        ctx.decode_step(torch.zeros(1, dtype=torch.int32, device=dev),
                        torch.tensor([int(toks[0, t])], dtype=torch.int32, device=dev), one)
        bt = toks[3:40, t].copy()
        bt[20 - 3] = toks[0, t]
        ctx.decode_step(batch_slots, torch.from_numpy(bt).to(dev), many)
        ctx.synchronize()
        assert torch.equal(one[0], many[20 - 3])


def test_graph_replay_equals_direct_launch(tiny):
    torch = _torch()
    dev = torch.device("cuda")
    outs = []
    for mode in (0, 1):
        ctx, W, dims = gpu_ctx("tiny", 8, tiny, mode)
        lg = torch.empty(8, dims.vocab, device=dev)
        res = []
        for t in range(3):
            toks = torch.from_numpy(synth.prompt_tokens(dims.vocab, 8, 1, seed=40 + t)[:, 0]).to(dev)
            ctx.decode_step(torch.arange(8, dtype=torch.int32, device=dev), toks, lg)
            res.append(lg.clone())
        ctx.synchronize()
        outs.append(torch.stack(res))
        ctx.close()
    assert torch.equal(outs[0], outs[1])


def test_prefill_matches_decode_steps(tiny):
    """prefill_seq (chunked: the tokens of a chunk are the N side of every
    projection) against the same tokens fed as T single-token decode steps:
    logits within the tolerance, states within fp32 reassociation."""
    torch = _torch()
    dev = torch.device("cuda")
    ctx, W, dims = gpu_ctx("tiny", 4, tiny, 0)
    toks = synth.prompt_tokens(dims.vocab, 1, 20, seed=8)[0]
    a = torch.empty(dims.vocab, device=dev)
    ctx.prefill_seq(0, torch.from_numpy(toks).to(dev), a)
    b = torch.empty(1, dims.vocab, device=dev)
    for t in toks:
        ctx.decode_step(torch.ones(1, dtype=torch.int32, device=dev),
                        torch.tensor([int(t)], dtype=torch.int32, device=dev), b)
    ctx.synchronize()
    assert_logits_close(a.cpu().numpy(), b[0].cpu().numpy(), "prefill vs steps")
    for x, y in zip(ctx.get_state(0), ctx.get_state(1)):
        np.testing.assert_allclose(x, y, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("T", [1, 5, 37, 300])
def test_prefill_chunked_against_oracle(tiny, T):
    """prefill_seq of T tokens (T=300 spans two 256-token chunks) from a
    non-zero state, against the oracle's chunked prefill: last-token logits
    within the tolerance, recurrent and shift states close."""
    torch = _torch()
    dev = torch.device("cuda")
    ctx, W, dims = gpu_ctx("tiny", 4, tiny, 0)
    pre = synth.prompt_tokens(dims.vocab, 1, 6, seed=51)[0]
    toks = synth.prompt_tokens(dims.vocab, 1, T, seed=52 + T)[0]
    m, (st,) = oracle_states(W, dims, 1)
    st.prefill_chunked(pre, want_logits=False)
    ref = st.prefill_chunked(toks, want_logits=True)[-1]
    ctx.prefill_seq(2, torch.from_numpy(pre).to(dev))
    lg = torch.empty(dims.vocab, device=dev)
    ctx.prefill_seq(2, torch.from_numpy(toks).to(dev), lg)
    ctx.synchronize()
    assert_logits_close(lg.cpu().numpy(), ref, f"T={T}")
    for name, gx, wx in zip(("wkv", "shift_att", "shift_ffn"), ctx.get_state(2), st.get()):
        wx = np.asarray(wx, np.float64).reshape(gx.shape)
        err = np.max(np.abs(gx - wx))
        assert err <= 1e-2 * max(1.0, float(np.max(np.abs(wx)))), (name, T, err)


def test_prefill_at_2p9b_layer_sizes():
    """Chunked prefill on the 2.9B layer sizes cut to 2 layers, 280 tokens
    (two chunks), then two decode steps, against the oracle."""
    torch = _torch()
    dev = torch.device("cuda")
    ctx, W, dims = gpu_ctx("2.9b", 4, None, 0, n_layer=2)
    toks = synth.prompt_tokens(dims.vocab, 1, 282, seed=61)[0]
    m, (st,) = oracle_states(W, dims, 1)
    ref = st.prefill_chunked(toks[:280], want_logits=True)[-1]
    lg = torch.empty(dims.vocab, device=dev)
    ctx.prefill_seq(1, torch.from_numpy(toks[:280]).to(dev), lg)
    ctx.synchronize()
    assert_logits_close(lg.cpu().numpy(), ref, "prefill 280")
    out = torch.empty(1, dims.vocab, device=dev)
    for t in toks[280:]:
        ctx.decode_step(torch.ones(1, dtype=torch.int32, device=dev),
                        torch.tensor([int(t)], dtype=torch.int32, device=dev), out)
        ctx.synchronize()
        assert_logits_close(out[0].cpu().numpy(), st.step(int(t)), "decode after prefill")


def test_slot_reset_copy_swap_and_checkpoint(tiny):
    torch = _torch()
    dev = torch.device("cuda")
    ctx, W, dims = gpu_ctx("tiny", 4, tiny, 0)
    for s in range(3):
        ctx.prefill_seq(s, torch.from_numpy(synth.prompt_tokens(dims.vocab, 1, 5, seed=60 + s)[0]).to(dev))
    ctx.synchronize()
    s0, s1 = ctx.get_state(0), ctx.get_state(1)
    assert np.abs(s0[0]).max() > 0
    ctx.slot_swap(0, 1)
    ctx.synchronize()
    for x, y in zip(ctx.get_state(0), s1):
        assert np.array_equal(x, y)
    ctx.slot_copy(1, 3)  # slot 1 now holds the old slot 0
    ctx.synchronize()
    for x, y in zip(ctx.get_state(3), s0):
        assert np.array_equal(x, y)
    ctx.slot_reset(2)
    ctx.synchronize()
    for x in ctx.get_state(2):
        assert not np.any(x)
    # checkpoint: save, run, restore, run again -> identical
    saved = ctx.get_state(3)
    toks = synth.prompt_tokens(dims.vocab, 1, 4, seed=70)[0]
    runs = []
    for _ in range(2):
        ctx.set_state(3, *saved)
        lg = torch.empty(dims.vocab, device=dev)
        ctx.prefill_seq(3, torch.from_numpy(toks).to(dev), lg)
        runs.append(lg.clone())
    ctx.synchronize()
    assert torch.equal(runs[0], runs[1])


SAMPLER_CASES = [
    dict(temperature=1.0, top_p=0.3, frequency=1.0, penalty_decay=0.996),
    dict(temperature=0.7, top_p=0.9, presence=0.5, frequency=0.3, penalty_decay=0.99),
    dict(temperature=1.3, top_p=0.5, top_k=20, frequency=0.5, penalty_decay=0.996),
    dict(temperature=1.0, top_p=1.0, top_k=1),
    dict(greedy=True),
    dict(temperature=1.0, top_p=1.0, frequency=0.0, penalty_decay=1.0),
    dict(temperature=1.0, top_p=1e-6),
    dict(temperature=2.0, top_p=0.95, top_k=200, presence=0.2, frequency=0.2, penalty_decay=0.9),
]


def test_sampler_bit_exact_against_oracle():
    """sample_batch on random logits at V=65536 equals the oracle sampler token
    for token over 25 rounds (occurrence counts and draw counters evolving)."""
    torch = _torch()
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    dims = synth.Dims("0.1b")
    ctx = rd.Rwkv7(dims, len(SAMPLER_CASES))
    occ, full = [], []
    for s, p in enumerate(SAMPLER_CASES):
        f = dict(temperature=1.0, top_p=1.0, top_k=0, presence=0.0, frequency=0.0, penalty_decay=1.0,
                 greedy=False, seed=1000 + s)
        f.update(p)
        full.append(f)
        ctx.set_sampling(s, **f)
        occ.append(np.zeros(dims.vocab, np.float32))
    slots = torch.arange(len(SAMPLER_CASES), dtype=torch.int32, device=dev)
    nxt = torch.empty(len(SAMPLER_CASES), dtype=torch.int32, device=dev)
    draws = [0] * len(SAMPLER_CASES)
    for rnd in range(25):
        lg = synth.random_logits(len(SAMPLER_CASES), dims.vocab, seed=500 + rnd, scale=1.0 + (rnd % 4))
        ctx.sample_batch(slots, torch.from_numpy(lg).to(dev), nxt)
        ctx.synchronize()
        got = nxt.cpu().numpy()
        for s, p in enumerate(full):
            tok, _ = oracle.sample(lg[s], occ[s], p, draws[s])
            if not p["greedy"]:
                draws[s] += 1
            assert got[s] == tok, (rnd, s, got[s], tok)


def test_sampler_wide_batch_bit_exact_against_oracle():
    """A batch with more rows than SMs takes the sampler's two-CTAs-per-SM build:
    its tokens equal the oracle sampler's, row for row, over a few rounds."""
    torch = _torch()
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    dims = synth.Dims("0.1b")
    B = torch.cuda.get_device_properties(0).multi_processor_count + 8
    ctx = rd.Rwkv7(dims, B)
    occ, full = [], []
    for s in range(B):
        f = dict(temperature=1.0, top_p=1.0, top_k=0, presence=0.0, frequency=0.0, penalty_decay=1.0,
                 greedy=False, seed=3000 + s)
        f.update(SAMPLER_CASES[s % len(SAMPLER_CASES)])
        full.append(f)
        ctx.set_sampling(s, **f)
        occ.append(np.zeros(dims.vocab, np.float32))
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    draws = [0] * B
    for rnd in range(4):
        lg = synth.random_logits(B, dims.vocab, seed=900 + rnd, scale=1.0 + rnd)
        ctx.sample_batch(slots, torch.from_numpy(lg).to(dev), nxt)
        ctx.synchronize()
        got = nxt.cpu().numpy()
        for s, p in enumerate(full):
            tok, _ = oracle.sample(lg[s], occ[s], p, draws[s])
            if not p["greedy"]:
                draws[s] += 1
            assert got[s] == tok, (rnd, s, got[s], tok)
    ctx.close()


def test_device_side_argument_errors_are_reported(tiny):
    torch = _torch()
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    ctx, W, dims = gpu_ctx("tiny", 4, tiny, 0)
    lg = torch.empty(2, dims.vocab, device=dev)
    bad_cases = [([0, 4], [1, 2]), ([0, 1], [1, dims.vocab]), ([2, 2], [1, 2]), ([-1, 1], [1, 2])]
    for s, t in bad_cases:
        ctx.decode_step(torch.tensor(s, dtype=torch.int32, device=dev),
                        torch.tensor(t, dtype=torch.int32, device=dev), lg)
        with pytest.raises(rd.RWKV7Error) as ei:
            ctx.synchronize()
        assert ei.value.code == rd.EINVAL
    # the context still works afterwards
    ctx.decode_step(torch.tensor([0, 1], dtype=torch.int32, device=dev),
                    torch.tensor([1, 2], dtype=torch.int32, device=dev), lg)
    ctx.synchronize()
    assert torch.isfinite(lg).all()


def test_host_api_errors(tiny):
    import recurrent_decode_gb300 as rd
    dims = synth.Dims("tiny")
    ctx = rd.Rwkv7(dims, 4)
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.decode_step_host(np.array([0], np.int32), np.array([1], np.int32))
    assert ei.value.code == -6  # weights not set
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.set_weight("emb", np.zeros((3, 3), np.float16))
    assert ei.value.code == -2
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.set_weight("blocks.9.att.key", np.zeros((128, 128), np.float16))
    assert ei.value.code == -2
    ctx.set_weights(tiny)
    for s, t in (([0, 0], [1, 2]), ([0, 5], [1, 2]), ([0, 1], [1, 5000])):
        with pytest.raises(rd.RWKV7Error) as ei:
            ctx.decode_step_host(np.array(s, np.int32), np.array(t, np.int32))
        assert ei.value.code == -1
    nxt = np.zeros(2, np.int32)
    ctx.set_sampling(0, greedy=True)
    ctx.set_sampling(1, greedy=True)
    ctx.decode_step_host(np.array([0, 1], np.int32), np.array([1, 2], np.int32), None, nxt)
    assert np.all((nxt >= 0) & (nxt < dims.vocab))


def test_weight_file_roundtrip(tiny, tmp_path):
    torch = _torch()
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    path = str(tmp_path / "tiny.rwkv7")
    synth.write_weight_file(path, tiny)
    dims = synth.Dims("tiny")
    a = rd.Rwkv7(dims, 1)
    a.load_weights(path)
    b, _, _ = gpu_ctx("tiny", 1, tiny, 0)
    la = torch.empty(dims.vocab, device=dev)
    lb = torch.empty(dims.vocab, device=dev)
    toks = torch.tensor([3, 14, 15], dtype=torch.int32, device=dev)
    a.prefill_seq(0, toks, la)
    b.prefill_seq(0, toks, lb)
    a.synchronize()
    b.synchronize()
    assert torch.equal(la, lb)
