"""Shared helpers of the GPU parity tests: build a library context and an oracle
model on the same seeded weights, and compare their outputs.

Acceptance (fp16 weights, fp32 state): logits max-abs <= 2e-2 and cosine
>= 0.9999 against the oracle; greedy tokens identical wherever the oracle's
top-1/top-2 margin exceeds the logit tolerance (below it both picks are correct
readings of the same logits); sampled tokens bit-exact given identical logits."""
from __future__ import annotations

import numpy as np

import oracle
import synth

LOGIT_ATOL = 2e-2
LOGIT_COS = 0.9999


def gpu_ctx(shape: str, n_slots: int, weights: dict | None = None, mode: int = 0, n_layer: int | None = None):
    import recurrent_decode_gb300 as rd
    dims = synth.Dims(shape, n_layer)
    if weights is None:
        weights = synth.make_weights(shape, n_layer=n_layer)
    ctx = rd.Rwkv7(dims, n_slots)
    ctx.set_weights(weights)
    ctx.set_mode(mode)
    return ctx, weights, dims


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def assert_logits_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.max(np.abs(gpu - ref))
    cos = cosine(gpu, ref)
    assert err <= LOGIT_ATOL and cos >= LOGIT_COS, f"{what}: max|d|={err:.3e} cos={cos:.7f}"
    return err, cos


# Greedy checks of this test session, and those accepted only by the near-tie
# rule (oracle margin, where); the summary at the end of the run reports them.
GREEDY_CHECKS = [0]
ESCAPES = []


def greedy_consistent(gpu_token: int, ref_logits, where: str = "") -> bool:
    """The GPU's greedy token is the oracle's argmax, or within the tolerance of it
    (a near tie, counted in ESCAPES with the oracle's margin)."""
    GREEDY_CHECKS[0] += 1
    ref = np.asarray(ref_logits, np.float64)
    best = int(np.argmax(ref))
    if gpu_token == best:
        return True
    margin = float(ref[best] - ref[gpu_token])
    if margin <= 2 * LOGIT_ATOL:
        ESCAPES.append((margin, where))
        return True
    return False


def oracle_states(weights, dims, n):
    m = oracle.Model(weights, dims)
    return m, [m.new_state() for _ in range(n)]
