"""Failure paths of the library, made on the host: a latched device error
becomes the documented return code and is cleared, and a refused device
allocation makes context creation fail cleanly with the process still usable.
No kernel is made to fail, wait out or fault.

The articles' failure handling is a per-request abort and an engine-init error
(RWKV-Runner Albatross page, "断开中止与性能画像" and "适配器Runner 与异步引擎之间的桥");
here every call returns a status and device-side problems are latched in an
error word that the next rwkv7_synchronize reports."""
import numpy as np
import pytest

import synth
from _harness import assert_logits_close, oracle_states

pytestmark = pytest.mark.gpu


def _tiny_decode_matches_oracle(ctx, W, dims, steps=3):
    import torch
    dev = torch.device("cuda")
    ctx.slot_reset(0)
    ctx.set_sampling(0, greedy=True)
    _, (st,) = oracle_states(W, dims, 1)
    prompt = synth.prompt_tokens(dims.vocab, 1, 5)[0]
    ctx.prefill_seq(0, torch.from_numpy(prompt[:-1].copy()).to(dev))
    st.prefill_chunked(prompt[:-1], want_logits=False)
    slots = torch.zeros(1, dtype=torch.int32, device=dev)
    logits = torch.empty(1, dims.vocab, device=dev)
    nxt = torch.empty(1, dtype=torch.int32, device=dev)
    cur = int(prompt[-1])
    for s in range(steps):
        ctx.decode_step(slots, torch.tensor([cur], dtype=torch.int32, device=dev), logits, nxt)
        ctx.synchronize()
        assert_logits_close(logits[0].cpu().numpy(), st.step(cur), f"step {s}")
        cur = int(nxt.item())


def test_latched_timeout_is_reported_once_and_cleared():
    import recurrent_decode_gb300 as rd
    dims = synth.Dims("tiny")
    W = synth.make_weights("tiny")
    ctx = rd.Rwkv7(dims, 2)
    ctx.set_weights(W)
    ctx.synchronize()
    ctx.debug_latch_error(8)  # the bit a bounded in-kernel wait latches when it gives up
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.synchronize()
    assert ei.value.code == rd.ETIMEOUT
    assert "bounded wait" in str(ei.value)
    ctx.synchronize()  # cleared: the next call is clean
    ctx.debug_latch_error(1 | 2)  # argument errors map to RWKV7_EINVAL
    with pytest.raises(rd.RWKV7Error) as ei:
        ctx.synchronize()
    assert ei.value.code == rd.EINVAL
    assert "slot out of range" in str(ei.value) and "token out of range" in str(ei.value)
    ctx.synchronize()
    _tiny_decode_matches_oracle(ctx, W, dims)  # the context keeps working
    ctx.close()


def test_refused_device_allocation_returns_enomem_and_releases_everything():
    import torch
    import recurrent_decode_gb300 as rd
    dims = synth.Dims("tiny")
    W = synth.make_weights("tiny")
    live = {}
    calls = {"n": 0}

    def alloc(nbytes, fail_at):
        calls["n"] += 1
        if fail_at is not None and calls["n"] == fail_at:
            return 0
        p = torch.cuda.caching_allocator_alloc(nbytes)
        live[p] = nbytes
        return p

    def free(p):
        assert p in live, "released a pointer the allocator never gave out"
        del live[p]
        torch.cuda.caching_allocator_delete(p)

    try:
        for fail_at in (1, 7, 40):
            calls["n"] = 0
            rd.set_device_allocator(lambda n, f=fail_at: alloc(n, f), free)
            with pytest.raises(rd.RWKV7Error) as ei:
                rd.Rwkv7(dims, 2)
            assert ei.value.code == rd.ENOMEM
            assert "refused" in str(ei.value)
            assert not live, f"{len(live)} allocations not returned after the failed create"
        # the same process creates a working context through the hook
        calls["n"] = 0
        rd.set_device_allocator(lambda n: alloc(n, None), free)
        ctx = rd.Rwkv7(dims, 2)
        assert calls["n"] > 40 and len(live) == calls["n"]
        ctx.set_weights(W)
        _tiny_decode_matches_oracle(ctx, W, dims)
        ctx.close()
        assert not live
    finally:
        rd.set_device_allocator()
    # and with the default allocator again
    ctx = rd.Rwkv7(dims, 2)
    ctx.set_weights(W)
    _tiny_decode_matches_oracle(ctx, W, dims)
    ctx.close()


def test_allocator_hook_needs_both_functions():
    import recurrent_decode_gb300 as rd
    lib = rd.load_library()
    assert lib.rwkv7_set_device_allocator(rd.ALLOC_FN(lambda u, n, o: 1), rd.FREE_FN(), None) == rd.EINVAL
    assert lib.rwkv7_set_device_allocator(rd.ALLOC_FN(), rd.FREE_FN(), None) == rd.OK
