"""Continuous-batching trace driver over the C ABI.

The worker loop of the RWKV-Runner Albatross article ("连续批处理Worker 主循环")
keeps one state slot per running request, decodes all running slots together,
and admits waiting requests between decode rounds: a prefill phase every
`decode_prefill_ratio` (5) rounds admits up to `max_prefill_count`
(max(batch/8, 1)) requests, each prefilled as a single sequence; prompts
shorter than `min_forward_seq_len` (10) are fed through single-token steps
instead.  A request prefills prompt[:-1] and its first decode round consumes
prompt[-1] (RWKV-Server article, "RWKV 批量推理中 Prefill 的正确打开方式" §五).
Slots are reused as requests finish; a reused slot is reset first.  Each round
first checks every running slot for an abort: the worker loop's request-level
abort ends that request only (FINISHED_ABORTED) and frees its slot, and a
waiting request aborted before admission is never admitted.  Optionally the
prompt bodies go through a PrefixStateCache (prefix_cache.py): an admitted
request starts from the longest stored prefix state and prefills the rest.

Host scheduling only: every computation runs in the library's kernels through
the binding (rwkv7_prefill_seq, rwkv7_decode_step, rwkv7_slot_reset,
rwkv7_slot_copy).
"""
from __future__ import annotations

import time
from dataclasses import dataclass, field

import numpy as np


@dataclass
class Request:
    prompt: np.ndarray            # int32 token ids
    n_out: int                    # tokens to generate
    sampling: dict                # Rwkv7.set_sampling keyword arguments
    out: list = field(default_factory=list)
    slot: int = -1
    status: str = "waiting"       # waiting -> running -> finished | aborted
    prefix_hit: int = 0           # prompt tokens restored from the prefix cache
    t_first: float = -1.0         # seconds from the trace start to the first generated token
    t_done: float = -1.0


@dataclass
class TraceStats:
    generated: int = 0
    prefill_tokens: int = 0
    decode_fed_tokens: int = 0
    prefix_hit_tokens: int = 0
    aborted: int = 0
    rounds: int = 0
    wall_s: float = 0.0
    ttft_s: list = field(default_factory=list)


def run_trace(ctx, requests, n_slots: int, decode_prefill_ratio: int = 5, max_prefill_count: int | None = None,
              min_forward_seq_len: int = 10, on_round=None, want_logits: bool = False, abort_at=None,
              prefix_cache=None, device: str = "cuda") -> TraceStats:
    """Run every request to completion (or abort).  on_round(slots, tokens_in, logits,
    next_tokens) is called after each decode round with host int32 arrays (logits: a
    CUDA tensor [B][V] when want_logits, else None).  abort_at: {request index: round}
    -- the request is aborted at the start of that round.  prefix_cache: a
    PrefixStateCache over slots outside [0, n_slots).  device: where the token
    and slot tensors handed to ctx live (the library takes CUDA tensors)."""
    import torch
    dev = torch.device(device)
    if max_prefill_count is None:
        max_prefill_count = max(int(n_slots * 0.125), 1)
    abort_at = dict(abort_at or {})
    waiting = list(range(len(requests)))
    free = list(range(n_slots))
    running = {}                  # slot -> request index
    next_in = {}                  # slot -> next input token
    stats = TraceStats()
    V = ctx.dims.vocab
    logits = torch.empty(n_slots, V, device=dev) if want_logits else None
    nxt = torch.empty(n_slots, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)

    def admit():
        k = 0
        while waiting and free and k < max_prefill_count:
            i = waiting.pop(0)
            s = free.pop(0)
            r = requests[i]
            r.slot = s
            r.status = "running"
            ctx.slot_reset(s)
            ctx.set_sampling(s, **r.sampling)
            body = r.prompt[:-1]
            start = prefix_cache.restore(body, s) if prefix_cache is not None else 0
            r.prefix_hit = start
            stats.prefix_hit_tokens += start
            rest = body[start:]
            if len(rest) >= min_forward_seq_len:
                if prefix_cache is not None:
                    prefix_cache.prefill(s, body, start, to_dev)
                else:
                    ctx.prefill_seq(s, to_dev(rest))
                stats.prefill_tokens += len(rest)
            else:
                for tok in rest:  # short rest: single-token steps without the head
                    ctx.decode_step(torch.tensor([s], dtype=torch.int32, device=dev),
                                    torch.tensor([int(tok)], dtype=torch.int32, device=dev))
                stats.decode_fed_tokens += len(rest)
                if prefix_cache is not None and len(rest) > 0:
                    prefix_cache.store(body, s)
            running[s] = i
            next_in[s] = int(r.prompt[-1])
            k += 1

    def apply_aborts(now):
        for s in [s for s, i in running.items() if abort_at.get(i, 1 << 62) <= stats.rounds]:
            r = requests[running.pop(s)]
            del next_in[s]
            r.status = "aborted"
            r.t_done = now
            stats.aborted += 1
            free.append(s)
        for i in [i for i in waiting if abort_at.get(i, 1 << 62) <= stats.rounds]:
            waiting.remove(i)
            requests[i].status = "aborted"
            requests[i].t_done = now
            stats.aborted += 1

    while waiting or running:
        apply_aborts(time.perf_counter() - t0)
        if not waiting and not running:
            break
        if not running or stats.rounds % decode_prefill_ratio == 0:
            admit()
        slots = np.array(sorted(running), np.int32)
        toks = np.array([next_in[s] for s in slots], np.int32)
        B = len(slots)
        d_slots = torch.from_numpy(slots).to(dev)
        d_toks = torch.from_numpy(toks).to(dev)
        ctx.decode_step(d_slots, d_toks, logits[:B] if want_logits else None, nxt[:B])
        got = nxt[:B].cpu().numpy()
        now = time.perf_counter() - t0
        stats.rounds += 1
        if on_round is not None:
            on_round(slots, toks, logits[:B] if want_logits else None, got)
        for s, tok in zip(slots.tolist(), got.tolist()):
            r = requests[running[s]]
            if not r.out:
                r.t_first = now
                stats.ttft_s.append(now)
            r.out.append(int(tok))
            stats.generated += 1
            next_in[s] = int(tok)
            if len(r.out) >= r.n_out:
                r.status = "finished"
                r.t_done = now
                del running[s]
                del next_in[s]
                free.append(s)
    ctx.synchronize()
    stats.wall_s = time.perf_counter() - t0
    return stats
