"""Pins of the oracle's primitives against things other than the oracle itself:
library routines (numpy, torch), closed forms and invariants of the state update,
and published known-answer vectors."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp16
def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_f16_round_to_nearest_even_matches_numpy():
    g = np.random.default_rng(5)
    xs = np.concatenate([
        g.standard_normal(4000) * 10.0 ** g.integers(-9, 5, 4000),
        # exact ties between neighbours (1 + (2m+1)/2048) and subnormal ties
        (1.0 + (2 * np.arange(64) + 1) / 2048.0),
        (2 * np.arange(64) + 1) * 2.0 ** -25,
        [65504.0, 65519.9, 65520.0, 1e6, -1e6, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8, 0.0, -0.0],
    ])
    for x in xs:
        want = int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.f64_to_f16(float(x)) == want, x


# ---------------------------------------------------------------- GEMV / norms
def test_gemv_matches_numpy_matmul():
    g = np.random.default_rng(1)
    W = (g.standard_normal((300, 517)) * 0.02).astype(np.float16)
    x = g.standard_normal(517)
    ref = W.astype(np.float64) @ x
    np.testing.assert_allclose(oracle.gemv(W, x), ref, rtol=1e-12, atol=1e-13)


def test_layernorm_matches_torch_and_invariants():
    g = np.random.default_rng(2)
    x = g.standard_normal(768) * 3 + 1.5
    gam = g.uniform(0.5, 1.5, 768)
    bet = g.uniform(-0.3, 0.3, 768)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (768,), torch.from_numpy(gam),
                                         torch.from_numpy(bet), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.layernorm(x, gam, bet), ref, rtol=1e-12, atol=1e-12)
    y = oracle.layernorm(x, np.ones(768), np.zeros(768), eps=0.0)
    assert abs(y.mean()) < 1e-12 and abs(y.var() - 1.0) < 1e-12


def test_groupnorm_matches_torch():
    g = np.random.default_rng(3)
    x = g.standard_normal(4 * 64) * 2
    gam = g.uniform(0.5, 1.5, 256)
    bet = g.uniform(-0.3, 0.3, 256)
    ref = torch.nn.functional.group_norm(torch.from_numpy(x)[None], 4, torch.from_numpy(gam),
                                         torch.from_numpy(bet), eps=64e-5)[0].numpy()
    np.testing.assert_allclose(oracle.groupnorm(x, gam, bet, 64), ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- state update
def _rand_head(g, N, T=None):
    shp = (N,) if T is None else (T, N)
    r = g.standard_normal(shp)
    decay = g.uniform(0.5, 1.0, shp)
    kk = g.standard_normal(shp)
    kh = kk / np.linalg.norm(kk, axis=-1, keepdims=True)
    a = g.uniform(0.0, 1.0, shp)
    kp = g.standard_normal(shp)
    vp = g.standard_normal(shp)
    return r, decay, kh, a, kp, vp


@pytest.mark.parametrize("N", [2, 4, 64])
def test_wkv_step_equals_dense_transition_matrix(N):
    """Brute-force dense re-derivation: S' = S A + vp kp^T with the explicit
    transition A = diag(decay) - kh (a*kh)^T, then y = S' r (general matmuls)."""
    g = np.random.default_rng(N)
    S = g.standard_normal((N, N))
    for _ in range(5):
        r, decay, kh, a, kp, vp = _rand_head(g, N)
        A = np.diag(decay) - np.outer(kh, a * kh)
        S_ref = S @ A + np.outer(vp, kp)
        S_got, y = oracle.wkv_step(S, r, decay, kh, a, kp, vp)
        np.testing.assert_allclose(S_got, S_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(y, S_ref @ r, rtol=1e-12, atol=1e-12)
        S = S_got


def test_wkv_pure_accumulation_invariant():
    """Zero state, decay = 1, a = 0: the state is exactly sum_t vp_t kp_t^T."""
    g = np.random.default_rng(7)
    N, T = 64, 9
    S = np.zeros((N, N))
    acc = np.zeros((N, N))
    for _ in range(T):
        r, _, kh, _, kp, vp = _rand_head(g, N)
        # small-integer values make every product and sum exact in fp64
        kp = np.round(kp * 4); vp = np.round(vp * 4)
        S, y = oracle.wkv_step(S, r, np.ones(N), kh, np.zeros(N), kp, vp)
        acc += np.outer(vp, kp)
        assert np.array_equal(S, acc)


def test_wkv_forget_all_invariant():
    """decay = 0, a = 0: the state is the last outer product vp kp^T."""
    g = np.random.default_rng(8)
    N = 64
    S = g.standard_normal((N, N))
    for _ in range(3):
        r, _, kh, _, kp, vp = _rand_head(g, N)
        S, y = oracle.wkv_step(S, r, np.zeros(N), kh, np.zeros(N), kp, vp)
        assert np.array_equal(S, np.outer(vp, kp))
        np.testing.assert_allclose(y, vp * (kp @ r), rtol=1e-13)


def test_wkv_delta_rule_recall():
    """decay = 1, a = 1, kp = kh (unit): after the update S kh = vp exactly
    (up to rounding): the write replaces what the state held at key kh."""
    g = np.random.default_rng(9)
    N = 64
    S = g.standard_normal((N, N))
    for _ in range(5):
        r, _, kh, _, _, vp = _rand_head(g, N)
        S, _ = oracle.wkv_step(S, r, np.ones(N), kh, np.ones(N), kh, vp)
        np.testing.assert_allclose(S @ kh, vp, rtol=1e-11, atol=1e-11)


def test_wkv_removal_is_non_expansive():
    """decay = 1, scalar a in [0,1], unit kh: A = I - a kh kh^T has eigenvalues
    {1, 1-a}, so ||S A||_F <= ||S||_F (checked with vp = 0, no write)."""
    g = np.random.default_rng(10)
    N = 64
    S = g.standard_normal((N, N))
    for _ in range(20):
        r, _, kh, _, kp, _ = _rand_head(g, N)
        a = np.full(N, g.uniform())
        n0 = np.linalg.norm(S)
        S, _ = oracle.wkv_step(S, r, np.ones(N), kh, a, kp, np.zeros(N))
        assert np.linalg.norm(S) <= n0 * (1 + 1e-13)


@pytest.mark.parametrize("T", [1, 2, 7, 64])
def test_wkv_chunked_equals_stepwise(T):
    g = np.random.default_rng(100 + T)
    N = 64
    S0 = g.standard_normal((N, N))
    r, decay, kh, a, kp, vp = _rand_head(g, N, T)
    S = S0.copy()
    ys = []
    for t in range(T):
        S, y = oracle.wkv_step(S, r[t], decay[t], kh[t], a[t], kp[t], vp[t])
        ys.append(y)
    Sc, yc = oracle.wkv_chunk(S0, r, decay, kh, a, kp, vp)
    np.testing.assert_allclose(Sc, S, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(yc, np.array(ys), rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------- RNG, exp2
def test_philox_known_answer_vectors():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for row in rows:
        w = [int(v, 16) for v in row]
        assert oracle.philox4x32_10(w[0:4], w[4:6]) == w[6:10]


def test_exp2_within_two_ulp_of_libm():
    es = np.concatenate([-np.linspace(0, 125.9, 20001), -np.random.default_rng(4).uniform(0, 30, 5000),
                         [-0.5, -0.49999997, -1.5, -1e-8]]).astype(np.float32)
    for e in es:
        got = oracle.exp2(float(e))
        ref = math.pow(2.0, float(e))
        ulp = 2.0 ** (math.frexp(ref)[1] - 24) if ref >= 2.0 ** -126 else 2.0 ** -149
        assert abs(got - ref) <= 2 * ulp * (1 + 1e-9), (e, got, ref)
    assert oracle.exp2(0.0) == 1.0
    assert oracle.exp2(-200.0) == 0.0
