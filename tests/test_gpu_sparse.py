"""The sparse channel-mix value projection at mixed unions, against the oracle.

The RWKV-Server page ("RWKV 批量推理中 Prefill 的正确打开方式", section "cmix_sparse_one
vs cmix_sparse_rows 的调用") makes skipping the value rows whose ReLU^2 input is
zero the point of the B > 1, T = 1 path.  Here the key rows of a chosen share of
the 64-row hidden blocks are zero in every layer, so those blocks of ReLU^2
output are exactly zero for every slot and the value projection skips them,
while the other blocks are read.  The oracle computes the channel mix densely;
logits must agree within the tolerance, and the library's union count must
equal the number of kept blocks exactly, in decode steps and in prefill."""
import numpy as np
import pytest

import synth
from _harness import assert_logits_close, oracle_states

pytestmark = pytest.mark.gpu


def _sparse_weights(shape, n_layer, zero_frac, seed):
    dims = synth.Dims(shape, n_layer)
    nblk = dims.d_ffn // 64
    rng = np.random.default_rng(seed)
    zero = np.zeros(nblk, bool)
    zero[rng.permutation(nblk)[:int(round(zero_frac * nblk))]] = True

    def zap(a):
        a.reshape(nblk, 64, dims.d_model)[zero] = 0

    ov = {f"blocks.{l}.ffn.key": zap for l in range(dims.n_layer)}
    return dims, synth.make_weights(shape, n_layer=n_layer, overrides=ov), int((~zero).sum())


@pytest.mark.parametrize("shape,n_layer", [("tiny", None), ("2.9b", 2)])
@pytest.mark.parametrize("zero_frac", [0.5, 0.9])
@pytest.mark.parametrize("B", [1, 3, 64])
def test_mixed_union_matches_oracle_and_counts_kept_blocks(shape, n_layer, zero_frac, B):
    import torch
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    dims, W, kept = _sparse_weights(shape, n_layer, zero_frac, seed=B + int(100 * zero_frac))
    L, nblk = dims.n_layer, dims.d_ffn // 64
    ctx = rd.Rwkv7(dims, B)
    ctx.set_weights(W)
    tracked = sorted({0, B // 2, B - 1})
    _, sts = oracle_states(W, dims, len(tracked))
    # prefill of one slot's prompt body (chunked path), then batched decode steps
    prompt = synth.prompt_tokens(dims.vocab, 1, 9, seed=77)[0]
    ctx.ffn_union_stats()
    ctx.prefill_seq(tracked[0], torch.from_numpy(prompt[:-1].copy()).to(dev))
    sts[0].prefill_chunked(prompt[:-1], want_logits=False)
    nz, tot = ctx.ffn_union_stats()
    assert tot == L * nblk and nz == L * kept, (nz, tot, kept)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    logits = torch.empty(B, dims.vocab, device=dev)
    steps = 3
    for t in range(steps):
        toks = synth.prompt_tokens(dims.vocab, B, 1, seed=300 + t)[:, 0].copy()
        if t == 0:
            toks[tracked[0]] = prompt[-1]
        ctx.decode_step(slots, torch.from_numpy(toks).to(dev), logits)
        ctx.synchronize()
        got = logits.cpu().numpy()
        for k, s in enumerate(tracked):
            assert_logits_close(got[s], sts[k].step(int(toks[s])), f"{shape} B={B} step {t} slot {s}")
    nz, tot = ctx.ffn_union_stats()
    assert tot == steps * L * nblk
    assert nz == steps * L * kept, (nz, steps * L * kept)
    ctx.close()
