"""GPU parity of the int8 weight variant (W = q * per-row fp16 scale), through
the C ABI: the library's int8 GEMM (int8 tiles widened to fp16 in shared
memory, row scale in the epilogue) against the oracle's int8 model on the same
synthetic int8 weights, with the fp16 variant's tolerances.

- tiny shape, 16 greedy steps over a ragged batch of permuted slots, graph
  replay and direct launches (bit-identical to each other);
- the 2.9B layer sizes (2 layers) at B = 64 (two k-blocks per ring stage) and
  B = 200 (one k-block per stage), rows teacher-forced against the oracle;
- chunked prefill of 300 tokens (a 256-token chunk: N = 256) against the
  oracle's chunked prefill;
- the channel-mix value projection skipping all-zero blocks (zero key rows);
- the API refuses fp16 uploads of int8 matrices and the CUDA-core mode.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from _harness import assert_logits_close, greedy_consistent

pytestmark = pytest.mark.gpu


def _ctx(shape, n_slots, n_layer=None, pow2=False, zero_key=False):
    import recurrent_decode_gb300 as rd
    dims = synth.Dims(shape, n_layer)
    w16, i8 = synth.make_weights_i8(shape, n_layer=n_layer, pow2_scales=pow2)
    if zero_key:
        for l in range(dims.n_layer):
            i8[f"blocks.{l}.ffn.key"][0][...] = 0
    ctx = rd.Rwkv7(dims, n_slots, weight_bits=8)
    ctx.set_weights(w16, i8)
    oracle.set_threads(os.cpu_count() or 1)
    m = oracle.Model(w16, dims, int8=i8)
    return ctx, m, dims


@pytest.mark.parametrize("mode", [0, 1])
def test_tiny_int8_ragged_batch(mode):
    import torch
    dev = torch.device("cuda")
    ctx, m, dims = _ctx("tiny", 12)
    ctx.set_mode(mode)
    slots = np.array([7, 2, 11, 0, 5], np.int32)
    B = len(slots)
    for s in slots:
        ctx.set_sampling(int(s), greedy=True)
    sts = [m.new_state() for _ in range(B)]
    toks = synth.prompt_tokens(dims.vocab, B, 1, seed=61)[:, 0]
    lg = torch.empty(B, dims.vocab, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    d_slots = torch.from_numpy(slots).to(dev)
    for step in range(16):
        ctx.decode_step(d_slots, torch.from_numpy(toks.astype(np.int32)).to(dev), lg, nxt)
        ctx.synchronize()
        got, nt = lg.cpu().numpy(), nxt.cpu().numpy()
        for i in range(B):
            ref = sts[i].step(int(toks[i]))
            assert_logits_close(got[i], ref, f"mode {mode} step {step} row {i}")
            assert greedy_consistent(int(nt[i]), ref)
        toks = nt.copy()
    ctx.close()


def test_tiny_int8_graph_equals_direct():
    import torch
    dev = torch.device("cuda")
    outs = []
    for mode in (0, 1):
        ctx, _, dims = _ctx("tiny", 4)
        ctx.set_mode(mode)
        lg = torch.empty(3, dims.vocab, device=dev)
        seq = []
        for t in range(4):
            toks = synth.prompt_tokens(dims.vocab, 3, 1, seed=70 + t)[:, 0]
            ctx.decode_step(torch.arange(3, dtype=torch.int32, device=dev), torch.from_numpy(toks).to(dev), lg)
            ctx.synchronize()
            seq.append(lg.cpu().numpy().copy())
        outs.append(seq)
        ctx.close()
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("B", [64, 200])
def test_int8_at_2p9b_layer_sizes(B):
    import torch
    dev = torch.device("cuda")
    ctx, m, dims = _ctx("2.9b", B, n_layer=2)
    tracked = [0, B // 2, B - 1]
    sts = [m.new_state() for _ in tracked]
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    lg = torch.empty(B, dims.vocab, device=dev)
    for step in range(3):
        toks = synth.prompt_tokens(dims.vocab, B, 1, seed=80 + step)[:, 0]
        ctx.decode_step(slots, torch.from_numpy(toks).to(dev), lg)
        ctx.synchronize()
        got = lg[tracked].cpu().numpy()
        for k, s in enumerate(tracked):
            assert_logits_close(got[k], sts[k].step(int(toks[s])), f"B={B} step {step} slot {s}")
    ctx.close()


def test_int8_prefill_against_oracle():
    import torch
    dev = torch.device("cuda")
    ctx, m, dims = _ctx("0.1b", 2)
    toks = synth.prompt_tokens(dims.vocab, 1, 300, seed=90)[0]
    lg = torch.empty(dims.vocab, device=dev)
    ctx.prefill_seq(1, torch.from_numpy(toks).to(dev), lg)
    ctx.synchronize()
    st = m.new_state()
    ref = st.prefill_chunked(toks, chunk=64)
    assert_logits_close(lg.cpu().numpy(), ref[-1], "prefill last token")
    ctx.close()


def test_int8_sparse_value_projection():
    import torch
    dev = torch.device("cuda")
    ctx, m, dims = _ctx("tiny", 4, zero_key=True)
    sts = [m.new_state() for _ in range(3)]
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
    assert nz == 0 and tot == 3 * dims.n_layer * (dims.d_ffn // 64)
    ctx.close()


def test_int8_api_errors():
    import recurrent_decode_gb300 as rd
    dims = synth.Dims("tiny")
    w16, i8 = synth.make_weights_i8("tiny")
    ctx = rd.Rwkv7(dims, 2, weight_bits=8)
    assert ctx.lib.rwkv7_weight_bits(ctx.h) == 8
    full16 = synth.make_weights("tiny")
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.set_weight("blocks.0.att.key", full16["blocks.0.att.key"])
    assert ei.value.code == rd.ESHAPE
    q, sc = i8["blocks.0.att.key"]
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.set_weight_i8("blocks.0.att.key", q[:, :-1], sc)
    assert ei.value.code == rd.ESHAPE
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.set_weight_i8("blocks.0.ln1.w", q, sc)  # not an int8 matrix
    assert ei.value.code == rd.ESHAPE
    for mode in (2, 3):
        with pytest.raises(rd.RWKV7Error) as ei:
            ctx.set_mode(mode)
        assert ei.value.code == rd.EINVAL
    ctx.close()
    ctx16 = rd.Rwkv7(dims, 2)
    assert ctx16.lib.rwkv7_weight_bits(ctx16.h) == 16
    with pytest.raises(rd.RWKV7Error):
        ctx16.set_weight_i8("blocks.0.att.key", q, sc)
    ctx16.close()
