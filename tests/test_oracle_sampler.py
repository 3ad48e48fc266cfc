"""Pins of the oracle's sampler: reductions to greedy, the top-p set's defining
properties, exhaustive enumeration of the selection step, the empirical
histogram, the penalty (through top-k = 1) and the decayed-count closed form."""
import math

import numpy as np
import pytest

import oracle
import synth


def _logits(V, seed, scale=2.0):
    return synth.random_logits(1, V, seed, scale)[0]


def test_pick_enumeration_gives_weights_as_histogram():
    g = np.random.default_rng(0)
    for V in (1, 3, 8):
        for _ in range(10):
            w = g.integers(0, 6, V).astype(np.uint32)
            if w.sum() == 0:
                w[g.integers(0, V)] = 1
            hist = np.zeros(V, np.int64)
            for r in range(int(w.sum())):
                hist[oracle.pick(w, r)] += 1
            assert np.array_equal(hist, w.astype(np.int64))


def test_integer_weights_match_closed_form():
    V = 4096
    lg = _logits(V, 1)
    for T in (1.0, 0.7, 1.6):
        q1, qT, kept = oracle.sample_weights(lg, np.zeros(V, np.float32),
                                             dict(temperature=T, top_p=1.0))
        m = float(lg.max())
        ref1 = np.floor(2.0 ** 24 * np.exp(lg.astype(np.float64) - m))
        refT = np.floor(2.0 ** 24 * np.exp((lg.astype(np.float64) - m) / T))
        assert np.max(np.abs(q1.astype(np.float64) - ref1)) <= 1.0
        assert q1[np.argmax(lg)] == 2 ** 24
        assert np.max(np.abs(qT[kept].astype(np.float64) - refT[kept])) <= 1.0
        assert np.all(qT[~kept] == 0)


@pytest.mark.parametrize("top_p", [0.05, 0.3, 0.5, 0.9, 1.0])
def test_top_p_set_is_minimal_upward_closed_set(top_p):
    V = 2048
    lg = _logits(V, 2)
    q1, _, kept = oracle.sample_weights(lg, np.zeros(V, np.float32), dict(top_p=top_p))
    q = q1.astype(np.int64)
    target = max(1, math.ceil(top_p * q.sum()))
    target = min(target, q.sum())
    # upward closed: every value above the smallest kept value is kept
    tp = q[kept].min()
    assert np.array_equal(kept, q >= tp)
    # it reaches the mass, and dropping its smallest value class does not
    assert q[kept].sum() >= target
    assert q[q > tp].sum() < target


def test_top_k_one_and_tiny_top_p_are_greedy():
    V = 65536
    for s in range(5):
        lg = _logits(V, 10 + s)
        want = int(np.argmax(lg))
        occ = np.zeros(V, np.float32)
        t1, _ = oracle.sample(lg, occ.copy(), dict(top_k=1, top_p=1.0, seed=s), 3)
        t2, kept = oracle.sample(lg, occ.copy(), dict(top_p=1e-9, seed=s), 4)
        assert t1 == want and t2 == want and kept.sum() == 1


def test_greedy_ties_take_lowest_index():
    lg = np.zeros(16, np.float32)
    lg[[3, 7, 11]] = 1.0
    occ = np.zeros(16, np.float32)
    assert oracle.sample(lg, occ, dict(greedy=True), 0)[0] == 3


def test_penalty_applied_through_top_k_one():
    """With top-k = 1 the draw is the argmax of the penalised logits
    l_i - ((occ_i > 0) * presence + occ_i * frequency)."""
    V = 512
    g = np.random.default_rng(3)
    for s in range(20):
        lg = _logits(V, 40 + s, scale=0.5)
        occ = np.where(g.uniform(size=V) < 0.3, g.uniform(0, 2, V), 0).astype(np.float32)
        pres, freq = float(g.uniform(0, 1)), float(g.uniform(0, 1))
        pen = lg.astype(np.float64) - ((occ > 0) * pres + occ.astype(np.float64) * freq)
        tok, _ = oracle.sample(lg, occ.copy(), dict(top_k=1, presence=pres, frequency=freq,
                                                    penalty_decay=0.9), s)
        assert tok == int(np.argmax(pen))


def test_decayed_occurrence_closed_form():
    """After n draws occ_i = sum over draws s that picked i of decay^(n-1-s)."""
    V = 64
    decay = 0.996
    occ = np.zeros(V, np.float32)
    picks = []
    lg = _logits(V, 5, scale=0.3)
    params = dict(top_p=1.0, temperature=1.0, penalty_decay=decay, frequency=0.2, seed=9)
    for n in range(300):
        tok, _ = oracle.sample(lg, occ, params, n)
        picks.append(tok)
    ref = np.zeros(V)
    for s, t in enumerate(picks):
        ref[t] += decay ** (len(picks) - 1 - s)
    np.testing.assert_allclose(occ, ref, rtol=2e-4, atol=1e-6)


def test_empirical_histogram_on_tiny_vocab():
    """Many draws from an 8-token vocabulary follow qT / sum(qT) over the kept set."""
    V = 8
    lg = np.array([0.0, -0.3, -1.0, -0.2, -2.5, -0.05, -4.0, -0.7], np.float32)
    params = dict(top_p=0.85, temperature=1.3, seed=77, penalty_decay=1.0)
    q1, qT, kept = oracle.sample_weights(lg, np.zeros(V, np.float32), params)
    p = qT / qT.sum()
    n = 20000
    hist = np.zeros(V)
    for i in range(n):
        occ = np.zeros(V, np.float32)
        hist[oracle.sample(lg, occ, params, i)[0]] += 1
    assert np.all(hist[~kept] == 0)
    sd = np.sqrt(n * p * (1 - p)) + 1e-9
    assert np.all(np.abs(hist - n * p) <= 5 * sd)


def test_draw_stream_depends_on_seed_and_index():
    a = [oracle.draw_u64(1000, i) for i in range(4)]
    b = [oracle.draw_u64(1001, i) for i in range(4)]
    assert len(set(a)) == 4 and not set(a) & set(b)


def _kept_by_definition(q1, top_p, top_k):
    """The kept set written out from the reading of the worker's per-slot top_p /
    top_k (RWKV-Runner Albatross page, worker main loop): the top-p set is every
    token whose T=1 weight is at least the cut value, the cut being the largest
    weight value whose class and every heavier class together hold at least
    ceil(top_p * total) (at least 1, at most the total); then top-k keeps the
    first k tokens of the order (weight descending, index ascending); the result
    is the intersection.  Plain loops over the integer weights."""
    q = [int(x) for x in q1]
    total = sum(q)
    target = min(max(1, math.ceil(float(np.float32(top_p)) * total)), total)
    mass_at = {}
    for x in q:
        mass_at[x] = mass_at.get(x, 0) + x
    acc, cut = 0, None
    for val in sorted(mass_at, reverse=True):
        acc += mass_at[val]
        if acc >= target:
            cut = val
            break
    keep = [x >= cut for x in q]
    if 0 < top_k < len(q):
        order = sorted(range(len(q)), key=lambda i: (-q[i], i))
        allowed = set(order[:top_k])
        keep = [keep[i] and i in allowed for i in range(len(q))]
    return np.array(keep)


def _tied_logits(V, seed, n_levels):
    """Logits drawn from a few distinct values, so that ties fall at the top-k
    boundary and at the top-p cut."""
    g = np.random.default_rng(seed)
    levels = np.sort(g.normal(0, 1.5, n_levels)).astype(np.float32)
    return levels[g.integers(0, n_levels, V)].astype(np.float32)


@pytest.mark.parametrize("V", [16, 257, 4096])
@pytest.mark.parametrize("top_p", [0.05, 0.3, 0.9, 1.0])
@pytest.mark.parametrize("top_k", [2, 5, 20, 200])
def test_top_k_intersect_top_p_matches_definition(V, top_p, top_k):
    """top-k > 1 together with top-p: the oracle's kept set equals the set built
    from the definition, on continuous logits, on logits with many exact ties,
    and with a penalty in effect (the integer weights then come from the
    penalised logits)."""
    cases = [(_logits(V, 100 + V + top_k), np.zeros(V, np.float32)),
             (_tied_logits(V, 200 + V + top_k, 5), np.zeros(V, np.float32)),
             (_tied_logits(V, 300 + V + top_k, 17), np.zeros(V, np.float32))]
    g = np.random.default_rng(V * 7 + top_k)
    occ = np.where(g.uniform(size=V) < 0.2, g.integers(1, 4, V), 0).astype(np.float32)
    cases.append((_logits(V, 400 + V + top_k, scale=1.0), occ))
    for lg, oc in cases:
        params = dict(top_p=top_p, top_k=top_k, temperature=1.0, presence=0.3, frequency=0.5)
        q1, qT, kept = oracle.sample_weights(lg, oc, params)
        want = _kept_by_definition(q1, top_p, top_k)
        assert np.array_equal(kept, want)
        assert kept.sum() <= top_k
        assert np.all(qT[~kept] == 0) and np.all(qT[kept] == q1[kept])


def test_top_k_boundary_ties_keep_lowest_indices():
    """Equal weights straddling the k-th place: the lower indices are kept, and
    the set size is exactly k when the top-p set holds at least k tokens."""
    lg = np.zeros(12, np.float32)
    lg[[2, 5, 8, 11]] = 1.0  # four tokens tie for the top
    for k in (1, 2, 3, 4):
        _, _, kept = oracle.sample_weights(lg, np.zeros(12, np.float32), dict(top_p=1.0, top_k=k))
        assert list(np.flatnonzero(kept)) == [2, 5, 8, 11][:k]
    _, _, kept = oracle.sample_weights(lg, np.zeros(12, np.float32), dict(top_p=1.0, top_k=6))
    assert list(np.flatnonzero(kept)) == [0, 1, 2, 5, 8, 11]


def test_top_p_mass_is_taken_over_the_whole_vocabulary():
    """The top-p cut is computed on all tokens, before top-k: with a long flat
    tail, top_p = 0.9 keeps many tokens, so top-k = 3 keeps three of them.  (If
    the mass were taken over the top-k tokens only, a dominant first token would
    be kept alone.)"""
    V = 64
    lg = np.full(V, -1.0, np.float32)
    lg[0] = 3.0
    _, _, kept = oracle.sample_weights(lg, np.zeros(V, np.float32), dict(top_p=0.9, top_k=3))
    assert list(np.flatnonzero(kept)) == [0, 1, 2]
    _, _, kept_p = oracle.sample_weights(lg, np.zeros(V, np.float32), dict(top_p=0.3, top_k=3))
    assert list(np.flatnonzero(kept_p)) == [0]


def test_sample_draws_only_from_the_top_k_top_p_set():
    V = 1024
    lg = _tied_logits(V, 55, 9)
    params = dict(top_p=0.6, top_k=20, temperature=0.8, seed=5, penalty_decay=1.0)
    _, _, kept = oracle.sample_weights(lg, np.zeros(V, np.float32), params)
    for i in range(300):
        tok, kk = oracle.sample(lg, np.zeros(V, np.float32), params, i)
        assert kept[tok] and np.array_equal(kk, kept)
