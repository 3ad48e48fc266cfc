"""Pins of the oracle's whole-model step.

The pages print no logits, so these pins are internal: the chunked-vs-stepwise
identity (two formulations of the recurrence), closed forms of models with parts
switched off (computed here with torch primitives and a dense transition matrix
instead of the oracle's rank-1 update), and the parameter counts of the pages'
model names."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

TINY = synth.Dims("tiny")


def _zero(a):
    a[...] = 0


@pytest.fixture(scope="module")
def tiny_weights():
    return synth.make_weights("tiny")


def test_param_counts_match_page_model_names():
    assert round(synth.n_params(synth.Dims("2.9b")) / 1e9, 1) == 2.9
    assert round(synth.n_params(synth.Dims("7.2b")) / 1e9, 1) == 7.2


@pytest.mark.parametrize("T,chunk", [(1, 64), (2, 64), (7, 5), (64, 64), (513, 64)])
def test_chunked_prefill_equals_stepwise(tiny_weights, T, chunk):
    m = oracle.Model(tiny_weights, TINY)
    toks = synth.prompt_tokens(TINY.vocab, 1, T, seed=31)[0]
    s1 = m.new_state()
    step_logits = np.stack([s1.step(int(t)) for t in toks])
    s2 = m.new_state()
    chunk_logits = s2.prefill_chunked(toks, chunk=chunk)
    np.testing.assert_allclose(chunk_logits, step_logits, rtol=1e-8, atol=1e-8)
    for a, b in zip(s1.get(), s2.get()):
        np.testing.assert_allclose(a, b, rtol=1e-8, atol=1e-8)


def test_chunked_prefill_from_nonzero_state(tiny_weights):
    m = oracle.Model(tiny_weights, TINY)
    toks = synth.prompt_tokens(TINY.vocab, 2, 40, seed=32)
    s1 = m.new_state()
    for t in toks[0]:
        s1.step(int(t))
    s2 = s1.copy()
    ref = np.stack([s1.step(int(t)) for t in toks[1]])
    got = s2.prefill_chunked(toks[1], chunk=16)
    np.testing.assert_allclose(got, ref, rtol=1e-8, atol=1e-8)


# ---------------------------------------------------------------- closed forms
def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def _r16(x: torch.Tensor) -> torch.Tensor:
    return torch.from_numpy(x.numpy().astype(np.float16).astype(np.float64))


def _ln(x, w, b):
    return F.layer_norm(x, (x.shape[-1],), _t(w), _t(b), eps=1e-5)


def _head(W, x):
    return _t(W["head"]) @ _r16(_ln(x, W["ln_out.w"], W["ln_out.b"]))


def test_residual_off_closed_form(tiny_weights):
    """All output projections zero: logits = head . r16(LNout(LN0(emb[tok])))."""
    ov = {}
    for l in range(TINY.n_layer):
        ov[f"blocks.{l}.att.output"] = _zero
        ov[f"blocks.{l}.ffn.value"] = _zero
    W = synth.make_weights("tiny", overrides=ov)
    m = oracle.Model(W, TINY)
    s = m.new_state()
    for tok in (5, 999, 0):
        x0 = _ln(_t(W["emb"][tok]), W["ln0.w"], W["ln0.b"])
        np.testing.assert_allclose(s.step(tok), _head(W, x0).numpy(), rtol=1e-10, atol=1e-10)


def _att_only_sequence(W, toks):
    """Closed form of a model whose channel mixes are all off, for a token
    sequence from the zero state, with each head's state carried as a dense
    matrix: S_t = S_{t-1} A_t + vp_t kp_t^T, A_t = diag(decay_t) - kh_t (a_t kh_t)^T."""
    d, N, L = TINY.d_model, 64, TINY.n_layer
    H = d // N
    S = torch.zeros(L, H, N, N, dtype=torch.float64)
    prev = torch.zeros(L, d, dtype=torch.float64)
    outs = []
    for tok in toks:
        x = _ln(_t(W["emb"][tok]), W["ln0.w"], W["ln0.b"])
        v_first = None
        for l in range(L):
            p = f"blocks.{l}.att."
            xl = _ln(x, W[f"blocks.{l}.ln1.w"], W[f"blocks.{l}.ln1.b"])
            mix = {n: _r16(xl + (prev[l] - xl) * _t(W[p + "x_" + n])) for n in "rwkvag"}
            prev[l] = xl
            r = _t(W[p + "receptance"]) @ mix["r"]
            k = _t(W[p + "key"]) @ mix["k"]
            v = _t(W[p + "value"]) @ mix["v"]
            hw = _r16(torch.tanh(_t(W[p + "w1"]) @ mix["w"]))
            ha = _r16(_t(W[p + "a1"]) @ mix["a"])
            hv = _r16(_t(W[p + "v1"]) @ mix["v"])
            hg = _r16(torch.sigmoid(_t(W[p + "g1"]) @ mix["g"]))
            dw = _t(W[p + "w0"]) + _t(W[p + "w2"]) @ hw
            decay = torch.exp(-np.exp(-0.5) * torch.sigmoid(dw))
            a = torch.sigmoid(_t(W[p + "a0"]) + _t(W[p + "a2"]) @ ha)
            g = _t(W[p + "g2"]) @ hg
            if l == 0:
                v_first = v
            else:
                vg = torch.sigmoid(_t(W[p + "v0"]) + _t(W[p + "v2"]) @ hv)
                v = torch.lerp(v, v_first, vg)
            kh = F.normalize((k * _t(W[p + "k_k"])).view(H, N), dim=-1, eps=1e-12)
            kp = (k * (1 + (a - 1) * _t(W[p + "k_a"]))).view(H, N)
            vp = v.view(H, N)
            y = torch.zeros(H, N, dtype=torch.float64)
            for h in range(H):
                A = torch.diag(decay.view(H, N)[h]) - torch.outer(kh[h], a.view(H, N)[h] * kh[h])
                S[l, h] = S[l, h] @ A + torch.outer(vp[h], kp[h])
                y[h] = S[l, h] @ r.view(H, N)[h]
            yn = F.group_norm(y.reshape(1, d), H, _t(W[p + "ln_x.w"]), _t(W[p + "ln_x.b"]),
                              eps=64e-5)[0].view(H, N)
            bonus = (r.view(H, N) * kp * _t(W[p + "r_k"]).view(H, N)).sum(-1, keepdim=True)
            z = _r16(((yn + bonus * vp).reshape(d)) * g)
            x = x + _t(W[p + "output"]) @ z
        outs.append(x)
    return outs


def test_attention_only_model_closed_form(tiny_weights):
    """Channel mixes off (value matrices zero): logits follow from the
    dense-transition closed form above over 5 tokens, both layers active
    (layer 1 exercises the mix toward the layer-0 value)."""
    ov = {f"blocks.{l}.ffn.value": _zero for l in range(TINY.n_layer)}
    W = synth.make_weights("tiny", overrides=ov)
    m = oracle.Model(W, TINY)
    s = m.new_state()
    toks = [17, 400, 3, 1023, 17]
    xs = _att_only_sequence(W, toks)
    for tok, x1 in zip(toks, xs):
        np.testing.assert_allclose(s.step(tok), _head(W, x1).numpy(), rtol=1e-9, atol=1e-9)


def test_single_channel_mix_layer_closed_form(tiny_weights):
    """Only layer 0's channel mix active: x1 = x0 + Wv r16(relu(Wk xk)^2) with the
    token-shifted channel-mix input, over 3 tokens."""
    ov = {"blocks.0.att.output": _zero, "blocks.1.att.output": _zero, "blocks.1.ffn.value": _zero}
    W = synth.make_weights("tiny", overrides=ov)
    m = oracle.Model(W, TINY)
    s = m.new_state()
    prev = torch.zeros(TINY.d_model, dtype=torch.float64)
    for tok in (8, 8, 512):
        x0 = _ln(_t(W["emb"][tok]), W["ln0.w"], W["ln0.b"])
        xl2 = _ln(x0, W["blocks.0.ln2.w"], W["blocks.0.ln2.b"])
        xk = _r16(xl2 + (prev - xl2) * _t(W["blocks.0.ffn.x_k"]))
        prev = xl2
        h = _r16(torch.relu(_t(W["blocks.0.ffn.key"]) @ xk) ** 2)
        x1 = x0 + _t(W["blocks.0.ffn.value"]) @ h
        np.testing.assert_allclose(s.step(tok), _head(W, x1).numpy(), rtol=1e-9, atol=1e-9)


def test_state_roundtrip_and_copy(tiny_weights):
    m = oracle.Model(tiny_weights, TINY)
    s = m.new_state()
    for t in (1, 2, 3):
        s.step(t)
    c = s.copy()
    a = s.step(77)
    b = c.step(77)
    assert np.array_equal(a, b)


def test_state_stays_finite_over_long_run(tiny_weights):
    m = oracle.Model(tiny_weights, TINY)
    s = m.new_state()
    toks = synth.prompt_tokens(TINY.vocab, 1, 2000, seed=33)[0]
    s.prefill_chunked(toks, chunk=64, want_logits=False)
    for a in s.get():
        assert np.all(np.isfinite(a))
    assert np.abs(s.get()[0]).max() < 1e4
