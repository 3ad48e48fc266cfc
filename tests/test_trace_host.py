"""Host scheduling of the continuous-batching trace driver (no GPU): the
worker loop's admission policy, decode-fed short prompts, token feedback, slot
reuse, request abort and the prefix-cache hookup, run against a fake context
on CPU tensors that records every call and produces deterministic tokens."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from recurrent_decode_gb300.prefix_cache import PrefixStateCache
from recurrent_decode_gb300.trace import Request, run_trace

V = 1000


class Dims:
    vocab = V


class FakeCtx:
    def __init__(self):
        self.dims = Dims()
        self.calls = []
        self.state = {}

    def slot_reset(self, s):
        self.calls.append(("reset", s))
        self.state[s] = ()

    def set_sampling(self, s, **kw):
        self.calls.append(("sampling", s, kw.get("seed")))

    def slot_copy(self, src, dst):
        self.calls.append(("copy", src, dst))
        self.state[dst] = self.state.get(src, ())

    def prefill_seq(self, s, tokens):
        t = tuple(int(x) for x in tokens.cpu().numpy())
        self.calls.append(("prefill", s, len(t)))
        self.state[s] = self.state.get(s, ()) + t

    def decode_step(self, slots, tokens, logits=None, next_out=None):
        sl = slots.cpu().numpy().tolist()
        tk = tokens.cpu().numpy().tolist()
        self.calls.append(("step", tuple(sl), tuple(tk), next_out is not None))
        for s, t in zip(sl, tk):
            self.state[s] = self.state.get(s, ()) + (t,)
        if next_out is not None:  # a deterministic function of the slot's whole history
            nxt = [hash(self.state[s]) % V for s in sl]
            next_out[: len(sl)] = torch.tensor(nxt, dtype=torch.int32)

    def synchronize(self):
        pass


def _requests(lens, seed=0):
    g = np.random.default_rng(seed)
    return [Request(prompt=g.integers(0, V, pl).astype(np.int32), n_out=ol, sampling={"seed": i})
            for i, (pl, ol) in enumerate(lens)]


def _rounds_of_admission(ctx):
    """Index (in decode rounds with sampling) before which each reset happened."""
    out, rounds = [], 0
    for c in ctx.calls:
        if c[0] == "step" and c[3]:
            rounds += 1
        elif c[0] == "reset":
            out.append(rounds)
    return out


def test_admission_policy_and_token_feedback():
    ctx = FakeCtx()
    reqs = _requests([(30, 4), (25, 12), (40, 3), (6, 5), (50, 7), (20, 2), (33, 9)])
    st = run_trace(ctx, reqs, 3, decode_prefill_ratio=5, max_prefill_count=2, device="cpu")
    # admissions only every 5th round (or when nothing runs), at most 2 at a time
    adm = _rounds_of_admission(ctx)
    assert all(r % 5 == 0 for r in adm)
    for r in set(adm):
        assert adm.count(r) <= 2
    # every request generated exactly n_out tokens, in a slot of its own while running
    assert all(r.status == "finished" and len(r.out) == r.n_out for r in reqs)
    assert st.generated == sum(r.n_out for r in reqs)
    # prompt bodies >= 10 tokens are prefilled, shorter ones fed by single-token steps
    assert st.prefill_tokens == sum(len(r.prompt) - 1 for r in reqs if len(r.prompt) - 1 >= 10)
    assert st.decode_fed_tokens == 5
    # each request's slot saw: its prompt body, its last prompt token, then its own outputs fed back
    # (the fake's tokens are a function of that history, so a mixed-up feed changes them)
    for r in reqs:
        h = tuple(int(x) for x in r.prompt)
        outs = []
        for _ in range(r.n_out):
            tok = hash(h) % V
            outs.append(tok)
            h = h + (tok,)
        assert r.out == outs


def test_abort_running_and_waiting():
    ctx = FakeCtx()
    reqs = _requests([(30, 8), (30, 8), (30, 8), (30, 8)])
    st = run_trace(ctx, reqs, 2, decode_prefill_ratio=5, max_prefill_count=2, abort_at={0: 2, 3: 0},
                   device="cpu")
    assert reqs[0].status == "aborted" and len(reqs[0].out) == 2  # rounds 0 and 1 ran, aborted at round 2
    assert reqs[3].status == "aborted" and reqs[3].out == [] and reqs[3].slot == -1
    assert reqs[1].status == reqs[2].status == "finished"
    assert st.aborted == 2 and st.generated == 2 + 8 + 8
    # the aborted request's slot was reused by request 2 after the next admission round (5)
    assert reqs[2].slot == reqs[0].slot
    assert _rounds_of_admission(ctx) == [0, 0, 5]


def test_prefix_cache_hookup():
    ctx = FakeCtx()
    g = np.random.default_rng(5)
    prefix = g.integers(0, V, 300).astype(np.int32)
    reqs = [Request(prompt=np.concatenate([prefix, g.integers(0, V, 20 + i)]).astype(np.int32), n_out=3,
                    sampling={"seed": i}) for i in range(4)]
    cache = PrefixStateCache(ctx, [10, 11, 12], block=256)
    st = run_trace(ctx, reqs, 2, decode_prefill_ratio=5, max_prefill_count=2, prefix_cache=cache, device="cpu")
    assert [r.prefix_hit for r in reqs] == [0, 256, 256, 256]
    assert st.prefix_hit_tokens == 3 * 256
    assert st.prefill_tokens == sum(len(r.prompt) - 1 for r in reqs) - 3 * 256
    assert all(r.status == "finished" and len(r.out) == 3 for r in reqs)
