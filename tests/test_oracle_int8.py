"""Pins of the oracle's int8 weight variant (W[o][i] = q[o][i] * scale[o]).

With power-of-two scales every q * scale is exact in fp16, so the int8 form
must reproduce the fp16 form on that exact matrix bit for bit: the matrix-vector
product against the pinned fp16 one, and the whole model (every int8 matrix
wired in its place, the scale of the right row) against the fp16 model.  With
general scales the product is checked against numpy's matmul on the
dequantised matrix."""
import numpy as np

import oracle
import synth

TINY = synth.Dims("tiny")


def _dequant16(q, sc):
    w = q.astype(np.float64) * sc.astype(np.float64)[:, None]
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)  # exact for power-of-two scales
    return w16


def test_gemv_i8_equals_fp16_gemv_on_exact_matrix():
    g = np.random.default_rng(3)
    for rows, cols in [(1, 1), (5, 7), (64, 256), (300, 130)]:
        q = g.integers(-127, 128, (rows, cols)).astype(np.int8)
        sc = (2.0 ** -g.integers(9, 15, rows)).astype(np.float16)
        x = g.standard_normal(cols)
        assert np.array_equal(oracle.gemv_i8(q, sc, x), oracle.gemv(_dequant16(q, sc), x))


def test_gemv_i8_matches_numpy_with_general_scales():
    g = np.random.default_rng(4)
    q = g.integers(-127, 128, (96, 200)).astype(np.int8)
    sc = (g.random(96) * 1e-3 + 1e-4).astype(np.float16)
    x = g.standard_normal(200)
    ref = (q.astype(np.float64) * sc.astype(np.float64)[:, None]) @ x
    np.testing.assert_allclose(oracle.gemv_i8(q, sc, x), ref, rtol=1e-12, atol=1e-15)
    # the scale belongs to the output row: swapping two rows' scales changes exactly those rows
    sc2 = sc.copy()
    sc2[[0, 1]] = sc2[[1, 0]]
    y = oracle.gemv_i8(q, sc2, x)
    assert not np.allclose(y[:2], ref[:2]) and np.allclose(y[2:], ref[2:], rtol=1e-12)


def test_int8_model_equals_fp16_model_on_exact_weights():
    w16, i8 = synth.make_weights_i8("tiny", pow2_scales=True)
    full = dict(w16)
    for name, (q, sc) in i8.items():
        full[name] = _dequant16(q, sc)
    assert set(i8) == set(synth.i8_matrix_names(TINY))
    m8 = oracle.Model(w16, TINY, int8=i8)
    m16 = oracle.Model(full, TINY)
    toks = synth.prompt_tokens(TINY.vocab, 1, 12, seed=41)[0]
    s8, s16 = m8.new_state(), m16.new_state()
    a = s8.prefill_chunked(toks[:7], chunk=4)
    b = s16.prefill_chunked(toks[:7], chunk=4)
    assert np.array_equal(a, b)
    for t in toks[7:]:
        assert np.array_equal(s8.step(int(t)), s16.step(int(t)))
    for x, y in zip(s8.get(), s16.get()):
        assert np.array_equal(x, y)


def test_int8_weights_spread_like_fp16_variant():
    _, i8 = synth.make_weights_i8("tiny")
    q, sc = i8["blocks.0.att.key"]
    w = q.astype(np.float64) * sc.astype(np.float64)[:, None]
    assert 0.015 < w.std() < 0.025 and q.min() >= -127 and q.max() <= 127


def test_int8_weights_independent_of_thread_count():
    a16, a8 = synth.make_weights_i8("0.1b", threads=1, n_layer=1)
    b16, b8 = synth.make_weights_i8("0.1b", threads=8, n_layer=1)
    assert a16.keys() == b16.keys() and a8.keys() == b8.keys()
    assert all(np.array_equal(a16[k], b16[k]) for k in a16)
    assert all(np.array_equal(a8[k][0], b8[k][0]) and np.array_equal(a8[k][1], b8[k][1]) for k in a8)
