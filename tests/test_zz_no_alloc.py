"""GPU test of rwkv7_sample_rows_static, the sampler entry point that allocates
no device memory.

Callers that cannot allocate -- a serving process whose HBM already belongs to
its own arena, or a loop that cannot take the device-wide synchronisation that
cudaMalloc / cudaFree may cause -- own every buffer of this call themselves;
the sampler's scratch is a fixed array inside the library.  The test checks
that, on the same logits, parameters and starting counts, it returns exactly
the tokens of rwkv7_sample_batch (the tokens are integers decided by the same
kernel, so the tolerance is equality) on two calls in a row, the second one
depending on the occurrence counts and draw counters the first one left; and
that a batch larger than the fixed scratch is refused with a clear error.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

CASES = [
    dict(),                                   # the adapter's defaults: T=1, top_p 0.3, frequency 1, decay 0.996
    dict(greedy=True),
    dict(temperature=0.7, top_p=0.9, presence=0.5, frequency=0.5),
    dict(temperature=1.3, top_p=1.0, top_k=40),
    dict(top_p=1e-6),
    dict(temperature=2.0, top_p=0.95, top_k=200, presence=0.2, frequency=0.2, penalty_decay=0.9),
]


def test_static_sampler_matches_sample_batch():
    torch = pytest.importorskip("torch")
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    V = synth.Dims("0.1b").vocab
    B = rd.SAMPLE_STATIC_MAX_ELEMS // V      # a batch that fills the fixed scratch exactly
    assert B * V == rd.SAMPLE_STATIC_MAX_ELEMS
    params = []
    for s in range(B):
        p = dict(CASES[s % len(CASES)])
        p["seed"] = 7000 + s
        params.append(p)

    # existing entry point: a ctx whose slot s carries params[s]
    ctx = rd.Rwkv7(synth.Dims("0.1b"), B)
    for s, p in enumerate(params):
        ctx.set_sampling(s, **{**dict(temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0,
                                      penalty_decay=0.996, greedy=False), **p})
    # new entry point: caller-owned per-sequence arrays, same starting state
    table = torch.from_numpy(rd.sampling_table(params)).to(dev)
    occ = torch.zeros(B, V, dtype=torch.float32, device=dev)
    ndraw = torch.zeros(B, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    rows = torch.from_numpy(np.random.default_rng(3).permutation(B).astype(np.int32)).to(dev)
    got_ctx = torch.empty(B, dtype=torch.int32, device=dev)
    got_static = torch.empty(B, dtype=torch.int32, device=dev)
    for call in range(2):
        lg = torch.from_numpy(synth.random_logits(B, V, seed=900 + call, scale=2.0 + call)).to(dev)
        ctx.sample_batch(rows, lg, got_ctx)
        ctx.synchronize()
        rd.sample_rows_static(lg, rows, occ, table, ndraw, got_static, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        a, b = got_ctx.cpu().numpy(), got_static.cpu().numpy()
        assert np.array_equal(a, b), (call, np.nonzero(a != b)[0][:8])
        assert ((b >= 0) & (b < V)).all()

    # each non-greedy row drew twice and counted its two tokens
    greedy = np.array([bool(p.get("greedy", False)) for p in params])
    nd = ndraw.cpu().numpy()
    assert (nd[~greedy] == 2).all() and (nd[greedy] == 0).all()
    o = occ.cpu().numpy()
    assert (o[greedy] == 0).all()
    assert np.allclose(o[~greedy].sum(axis=1), [1.0 + d for d, g in
                                                zip([p.get("penalty_decay", 0.996) for p in params], greedy) if not g],
                       rtol=1e-6)


def test_static_sampler_rejects_a_batch_beyond_its_scratch():
    torch = pytest.importorskip("torch")
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    V = 65536
    B = rd.SAMPLE_STATIC_MAX_ELEMS // V + 1
    lg = torch.zeros(B, V, dtype=torch.float32, device=dev)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    occ = torch.zeros(B, V, dtype=torch.float32, device=dev)
    table = torch.from_numpy(rd.sampling_table([dict()] * B)).to(dev)
    ndraw = torch.zeros(B, dtype=torch.int64, device=dev)
    nxt = torch.full((B,), -1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(rd.RWKV7Error) as ei:
        rd.sample_rows_static(lg, rows, occ, table, ndraw, nxt, err)
    assert ei.value.code == rd.EINVAL and "exceeds" in str(ei.value)
    torch.cuda.synchronize()
    assert (nxt.cpu().numpy() == -1).all()   # nothing was launched


def test_static_sampler_flags_bad_rows_on_a_side_stream():
    """n_rows larger than B, one row index out of range, the call on a
    non-default stream: that row gets token 0 and error flag 1; every other row
    equals rwkv7_sample_batch's token for the same logits and parameters."""
    torch = pytest.importorskip("torch")
    import recurrent_decode_gb300 as rd
    dev = torch.device("cuda")
    V, B, n_rows = synth.Dims("tiny").vocab, 6, 11  # the comparison context samples V-wide rows
    params = [dict(CASES[s % len(CASES)], seed=8100 + s) for s in range(n_rows)]
    table = torch.from_numpy(rd.sampling_table(params)).to(dev)
    occ = torch.zeros(n_rows, V, dtype=torch.float32, device=dev)
    ndraw = torch.zeros(n_rows, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rows_np = np.array([9, 2, n_rows + 3, 0, 10, 5], np.int32)  # row 2 is out of range
    rows = torch.from_numpy(rows_np).to(dev)
    lg = torch.from_numpy(synth.random_logits(B, V, seed=811, scale=2.5)).to(dev)
    nxt = torch.full((B,), -1, dtype=torch.int32, device=dev)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    rd.sample_rows_static(lg, rows, occ, table, ndraw, nxt, err, stream=side)
    side.synchronize()
    got = nxt.cpu().numpy()
    assert int(err.item()) & 1
    assert got[2] == 0

    # the same rows through a context whose slot s carries params[s]
    ctx = rd.Rwkv7(synth.Dims("tiny"), n_rows)
    for s, p in enumerate(params):
        ctx.set_sampling(s, **{**dict(temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0,
                                      penalty_decay=0.996, greedy=False), **p})
    good = [i for i in range(B) if rows_np[i] < n_rows]
    want = torch.empty(len(good), dtype=torch.int32, device=dev)
    ctx.sample_batch(torch.from_numpy(rows_np[good].copy()).to(dev), lg[good].contiguous(), want)
    ctx.synchronize()
    assert np.array_equal(got[good], want.cpu().numpy())
    ctx.close()
