#!/usr/bin/env python
"""Batched RWKV-7 decode benchmark on one GB300 (or N replicas under torchrun).

A step is one batched decode step of B slots through the whole path (embedding,
every layer's time mix / state update / channel mix, head, sampling) on
synthetic random-init weights of the named shape.  Prints one JSON line.

  python bench.py [--config 2.9b|7.2b|0.1b|tiny] [--steps K] [--warmup W] [--gpus N]
  python bench.py --impl reference ...   # the CPU oracle on the same workload
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "batched decode tok/s on 1 GB300 (2.9B/7.2B shapes) and % of HBM weight-stream roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# dram bytes per launch from ncu captures, valid only while the kernel source is
# unchanged: kernel -> (source files, sha256 prefix of their concatenation at
# capture, workload, bytes)
NCU_TRAFFIC = {
    ("gemm_tc_kernel", "2.9b"): (("recurrent_decode_gb300/csrc/gemm.cu", "recurrent_decode_gb300/csrc/gemm_common.cuh"),
                                  "4a26b728954c9d79",
                                  "2.9B shape, B=64: DRAM read+write of the 11 GEMM launches of one step of "
                                  "a 2-layer cut (profiles/gemm_traffic_2.9b_b64.md), scaled to 32 layers + head, "
                                  "per launch", 35823045),
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _sha(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def class_bytes(dm: synth.Dims, B: int):
    """Algorithmic bytes per step of each kernel class: fp16 weights streamed
    once, activations read/written once, fp32 state read and written once."""
    d, F, V, L, H = dm.d_model, dm.d_ffn, dm.vocab, dm.n_layer, dm.n_head
    rs = dm.lora_w + dm.lora_a + dm.lora_v + dm.lora_g
    f32, f16 = 4, 2
    return {
        "embed": B * d * (f16 + f32),
        "ln_mix": L * B * d * (f32 + 2 * f32 + 6 * f16) + L * B * d * (f32 + 2 * f32 + f16),
        "gemm_proj": L * ((3 * d * d + d * rs) * f16 + B * 6 * d * f16 + B * (3 * d + rs) * f32),
        "gemm_lora": L * (d * rs * f16 + B * rs * f16 + B * 4 * d * f32),
        "wkv": L * B * (H * 64 * 64 * f32 * 2 + 9 * d * f32 + d * f16),
        "gemm_out": L * (d * d * f16 + B * d * f16 + 2 * B * d * f32),
        "gemm_key": L * (F * d * f16 + B * d * f16 + B * F * f16),
        "gemm_value": L * (d * F * f16 + B * F * f16 + 2 * B * d * f32),
        "ln_out": B * d * (f32 + f16),
        "gemm_head": V * d * f16 + B * d * f16 + B * V * f32,
        "sampler": B * V * f32,
        "lora_fin": L * B * rs * (f32 + f16),
    }


def step_bytes(dm: synth.Dims, B: int) -> int:
    """Weight + state bytes per step (the roofline's numerator): fp16 weights of
    every matrix but the gathered embedding, plus fp32 wkv and shift states
    read and written for B slots."""
    d, F, V, L, H = dm.d_model, dm.d_ffn, dm.vocab, dm.n_layer, dm.n_head
    rs = dm.lora_w + dm.lora_a + dm.lora_v + dm.lora_g
    w = L * (4 * d * d + 2 * d * F + 2 * d * rs) * 2 + V * d * 2
    s = 2 * B * L * (H * 64 * 64 + 2 * d) * 4
    return w + s


def step_bytes_i8(dm: synth.Dims, B: int) -> int:
    """step_bytes for the int8 weight variant: one byte per matrix weight plus
    an fp16 scale per matrix row, the same states."""
    d, F, V, L, H = dm.d_model, dm.d_ffn, dm.vocab, dm.n_layer, dm.n_head
    rs = dm.lora_w + dm.lora_a + dm.lora_v + dm.lora_g
    w = L * (4 * d * d + 2 * d * F + 2 * d * rs) + V * d
    scales = (L * (4 * d + F + d + rs + 4 * d) + V) * 2  # rows of r,k,v,o, key, value, LoRA down and up, head
    s = 2 * B * L * (H * 64 * 64 + 2 * d) * 4
    return w + scales + s


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_id: str | None):
        self.proc = None
        self.path = os.path.join("/tmp", f"rwkv7_clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100"]
        if dev_id:
            cmd += ["-i", dev_id]
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for ln in fh:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_baseline(weights, dm, wl, seconds=15.0):
    """The oracle, as it stands, on a bounded sample of the workload: decode
    tokens of one slot (after a short prompt) until ~`seconds` have passed."""
    import oracle
    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    m = oracle.Model(weights, dm)
    st = m.new_state()
    toks = synth.prompt_tokens(dm.vocab, 1, 64)[0]
    st.step(int(toks[0]), want_logits=False)
    n, t0 = 0, time.perf_counter()
    cur = int(toks[1])
    while True:
        lg = st.step(cur)
        cur = int(np.argmax(lg))
        n += 1
        if time.perf_counter() - t0 >= seconds or n >= 2000:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} greedy decode tokens of 1 slot of the {dm.name} shape (fp64 oracle, OpenMP over "
                      f"matrix rows, {threads} threads), {dt:.1f} s"}


def run_reference(args, wl, dm):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    weights = synth.make_weights(wl["shape"], n_layer=dm.n_layer)
    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    m = oracle.Model(weights, dm)
    st = m.new_state()
    toks = synth.prompt_tokens(dm.vocab, 1, 2)[0]
    st.step(int(toks[0]), want_logits=False)
    cur = int(toks[1])
    for _ in range(args.warmup):
        cur = int(np.argmax(st.step(cur)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cur = int(np.argmax(st.step(cur)))
    dt = time.perf_counter() - t0
    val = args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(wl, dm, args),
            "cpu_baseline": {"value": val, "unit": "tok/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step = 1 greedy decode token of 1 slot of the {dm.name} shape"},
            "e2e": {"value": val, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def _config(wl, dm, args):
    return {"workload": f"RWKV-7 {dm.name} shape batched greedy decode" if wl.get("greedy")
            else f"RWKV-7 {dm.name} shape batched sampled decode (top_p {wl.get('top_p')})",
            "shape": dm.name, "n_layer": dm.n_layer, "B": wl.get("B", wl.get("n_slots")),
            "prompt_tokens": wl.get("prompt", wl.get("prompt_range")), "decode_steps_timed": args.steps,
            "weights": "random-init fp16 (seed 0)", "state": "fp32",
            "l2": "inputs larger than L2 (weights + states per step >> 126 MB), no flush"}


def run_trace_bench(args, wl):
    """The continuous-batching trace: every request to completion through the
    worker loop (recurrent_decode_gb300.trace); value = generated tokens per
    second of wall time, prefills included."""
    import torch
    import recurrent_decode_gb300 as rd
    from recurrent_decode_gb300.trace import Request, run_trace
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    from recurrent_decode_gb300.prefix_cache import PrefixStateCache
    dm = synth.Dims(wl["shape"])
    weights = synth.make_weights(wl["shape"])
    n_cache = wl.get("cache_slots", 0)
    ctx = rd.Rwkv7(dm, wl["n_slots"] + n_cache)
    ctx.set_weights(weights)
    del weights
    if args.mode >= 0:
        ctx.set_mode(args.mode)
    lens = synth.trace_requests(wl["n_req"], *wl["prompt_range"], *wl["out_range"])
    prefix = (synth.prompt_tokens(dm.vocab, 1, wl["shared_prefix"], seed=9999)[0]
              if wl.get("shared_prefix") else np.zeros(0, np.int32))

    def make_requests():
        reqs = []
        for i, (pl, ol) in enumerate(lens):
            sp = dict(temperature=wl["temperature"], top_p=wl["top_p"], top_k=wl["top_k"],
                      presence=wl["presence"], frequency=wl["frequency"], penalty_decay=wl["penalty_decay"],
                      seed=synth.SAMPLING_SEED_BASE + i, greedy=False)
            tail = synth.prompt_tokens(dm.vocab, 1, pl, seed=10000 + i)[0]
            reqs.append(Request(prompt=np.concatenate([prefix, tail]).astype(np.int32), n_out=ol, sampling=sp))
        return reqs

    dev_id = None
    try:
        dev_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass

    def one_run(cache):
        for s in range(wl["n_slots"] + n_cache):
            ctx.slot_reset(s)
        torch.cuda.synchronize()
        reqs = make_requests()
        clk = ClockSampler(dev_id)
        st = run_trace(ctx, reqs, wl["n_slots"], decode_prefill_ratio=wl["decode_prefill_ratio"],
                       min_forward_seq_len=wl["min_forward_seq_len"], prefix_cache=cache)
        return st, clk.stop()

    uncached = None
    if n_cache:  # the same requests without the cache first, for comparison
        uncached, _ = one_run(None)
    cache = PrefixStateCache(ctx, range(wl["n_slots"], wl["n_slots"] + n_cache)) if n_cache else None
    stats, clocks = one_run(cache)
    ctx.close()
    ttft = np.array(stats.ttft_s)
    total_in = stats.prefill_tokens + stats.decode_fed_tokens + stats.generated
    line = {"metric": METRIC, "value": world * stats.generated / stats.wall_s, "unit": "tok/s", "n_gpus": world,
            "steps": stats.rounds, "warmup": 0, "ms_per_step": stats.wall_s * 1e3 / max(1, stats.rounds),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": f"continuous-batching trace on the {dm.name} shape ({args.config})",
                       "shape": dm.name, "slots": wl["n_slots"], "requests": wl["n_req"],
                       "prompt_range": list(wl["prompt_range"]), "output_range": list(wl["out_range"]),
                       "decode_prefill_ratio": wl["decode_prefill_ratio"],
                       "weights": "random-init fp16 (seed 0)"},
            "trace": {"generated_tokens": stats.generated, "prefill_tokens": stats.prefill_tokens,
                      "decode_fed_tokens": stats.decode_fed_tokens, "rounds": stats.rounds,
                      "wall_s": stats.wall_s, "prefill_share": stats.prefill_tokens / max(1, total_in),
                      "ttft_s_p50": float(np.percentile(ttft, 50)), "ttft_s_p90": float(np.percentile(ttft, 90))},
            "clocks": clocks}
    if uncached is not None:
        ut = np.array(uncached.ttft_s)
        line["config"]["shared_prefix"] = wl["shared_prefix"]
        line["config"]["cache_slots"] = n_cache
        line["prefix_cache"] = {
            "hits": cache.hits, "misses": cache.misses, "hit_tokens": cache.hit_tokens,
            "evictions": cache.evictions,
            "uncached": {"value": uncached.generated / uncached.wall_s, "wall_s": uncached.wall_s,
                         "prefill_tokens": uncached.prefill_tokens,
                         "ttft_s_p50": float(np.percentile(ut, 50)), "ttft_s_p90": float(np.percentile(ut, 90))},
            "note": "value / trace: the run with the cache; the same requests without it under 'uncached'"}
    if rank == 0:
        print(json.dumps(line))
    return 0


def secondary(config, steps, args, dev, world, int8=False):
    """The same timed decode loop on another named workload (graph replay,
    CUDA events, clocks sampled): throughput and whole-step roofline.  int8:
    the int8 weight variant (synth.make_weights_i8) of the workload."""
    import torch
    import recurrent_decode_gb300 as rd
    wl = synth.WORKLOADS[config]
    dm = synth.Dims(wl["shape"])
    B = wl["B"]
    if int8:
        w16, i8 = synth.make_weights_i8(wl["shape"])
        ctx = rd.Rwkv7(dm, B, weight_bits=8)
        ctx.set_weights(w16, i8)
        del w16, i8
    else:
        weights = synth.make_weights(wl["shape"])
        ctx = rd.Rwkv7(dm, B)
        ctx.set_weights(weights)
        del weights
    if args.mode >= 0:
        ctx.set_mode(args.mode)
    for s in range(B):
        if wl.get("greedy"):
            ctx.set_sampling(s, greedy=True)
        else:
            ctx.set_sampling(s, temperature=wl["temperature"], top_p=wl["top_p"], top_k=wl["top_k"],
                             presence=wl["presence"], frequency=wl["frequency"],
                             penalty_decay=wl["penalty_decay"], seed=synth.SAMPLING_SEED_BASE + s)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    prompts = torch.from_numpy(synth.prompt_tokens(dm.vocab, B, wl["prompt"])).to(dev)
    for t in range(wl["prompt"] - 1):
        ctx.decode_step(slots, prompts[:, t].contiguous())
    tokens = prompts[:, -1].contiguous()
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    for _ in range(max(3, args.warmup)):
        ctx.decode_step(slots, tokens, None, nxt)
        tokens.copy_(nxt)
    ctx.synchronize()
    dev_id = None
    try:
        dev_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    clk = ClockSampler(dev_id)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        ctx.decode_step(slots, tokens, None, nxt)
        tokens.copy_(nxt)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1)
    ctx.synchronize()
    ctx.close()
    peak, peak_kind = _peaks()
    sb = step_bytes_i8(dm, B) if int8 else step_bytes(dm, B)
    gbs = sb / (ms / steps / 1e3) / 1e9
    cfg = _config(wl, dm, argparse.Namespace(steps=steps))
    if int8:
        cfg["workload"] += ", int8 weights"
        cfg["weights"] = "random-init int8 matrices (uniform on [-127, 127]) with fp16 row scales (seed 0)"
    return {"config": cfg, "value": world * B * steps / (ms / 1e3),
            "unit": "tok/s", "steps": steps, "ms_per_step": ms / steps,
            "step_roofline": {"bytes_per_step": sb, "achieved_GBps": gbs, "frac_of_peak": gbs / peak,
                              "peak_kind": peak_kind, "frac_of_8TBps": gbs / NOMINAL_HBM_GBS},
            "clocks": clocks}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="2.9b", choices=list(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run a model with this many layers of the shape's sizes")
    ap.add_argument("--prompt", type=int, default=0, help="profiling only: override the prompt length")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the 7.2B-shape measurement added to the 2.9B line")
    ap.add_argument("--mode", type=int, default=-1,
                    help="implementation: 0 multi-kernel CUDA graph, 3 persistent kernel (default: library default)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = dict(synth.WORKLOADS[args.config])
    if args.config.startswith("trace") and args.impl != "reference":
        return run_trace_bench(args, wl)
    if args.prompt:
        wl["prompt"] = max(2, args.prompt)
    dm = synth.Dims(wl["shape"], args.layers or None)
    if args.impl == "reference":
        return run_reference(args, wl, dm)

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import recurrent_decode_gb300 as rd

    B = wl["B"]
    weights = synth.make_weights(wl["shape"], n_layer=args.layers or None)
    ctx = rd.Rwkv7(dm, B)
    ctx.set_weights(weights)
    if args.mode >= 0:
        ctx.set_mode(args.mode)
    for s in range(B):
        if wl.get("greedy"):
            ctx.set_sampling(s, greedy=True)
        else:
            ctx.set_sampling(s, temperature=wl["temperature"], top_p=wl["top_p"], top_k=wl["top_k"],
                             presence=wl["presence"], frequency=wl["frequency"],
                             penalty_decay=wl["penalty_decay"], seed=synth.SAMPLING_SEED_BASE + s)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    prompts = torch.from_numpy(synth.prompt_tokens(dm.vocab, B, wl["prompt"])).to(dev)
    # prompts: all but the last token consumed through batched steps without the head
    for t in range(wl["prompt"] - 1):
        ctx.decode_step(slots, prompts[:, t].contiguous())
    tokens = prompts[:, -1].contiguous()
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ctx.decode_step(slots, tokens, None, nxt)
        tokens.copy_(nxt)

    for _ in range(args.warmup):
        step()
    ctx.synchronize()
    dev_id = None
    try:
        dev_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ctx.ffn_union_stats()  # reset: count the timed steps only
    clk = ClockSampler(dev_id)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1)
    ctx.synchronize()
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    value = world * B * args.steps / (ms / 1e3)
    nzb, totb = ctx.ffn_union_stats()

    # end to end through the host-buffer entry point (pinned host memory)
    h_slots = torch.arange(B, dtype=torch.int32).pin_memory()
    h_tok = tokens.cpu().pin_memory()
    h_next = torch.empty(B, dtype=torch.int32).pin_memory()
    for _ in range(3):
        ctx.decode_step_host(h_slots, h_tok, None, h_next)
        h_tok.copy_(h_next)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        ctx.decode_step_host(h_slots, h_tok, None, h_next)
        h_tok.copy_(h_next)
    e2e_s = time.perf_counter() - t0
    e2e_val = world * B * args.e2e_steps / e2e_s

    # prefill throughput: one slot consumes a 1024-token prompt (4 chunks of 256)
    pre = None
    if not args.layers and not args.prompt:
        ptoks = torch.from_numpy(synth.prompt_tokens(dm.vocab, 1, 1024, seed=7)[0]).to(dev)
        plog = torch.empty(dm.vocab, device=dev)
        ctx.prefill_seq(0, ptoks, plog)  # warm-up
        ctx.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        ctx.prefill_seq(0, ptoks, plog)
        p1.record(stream)
        ctx.synchronize()
        pms = p0.elapsed_time(p1)
        body = synth.n_params(dm) - 2 * dm.vocab * dm.d_model  # all but the embedding and the head
        flops = 2.0 * body * 1024 + 2.0 * dm.vocab * dm.d_model
        pre = {"tokens": 1024, "ms": pms, "tok_per_s": 1024 / (pms / 1e3), "tflops": flops / (pms / 1e3) / 1e12,
               "note": "one slot, 4 chunks of 256 tokens; FLOPs = 2 x non-embedding, non-head parameters x tokens "
                       "+ the head for the last token"}

    # per-kernel-class device time of one directly launched step (events)
    prof = ctx.profile_step(slots, tokens, with_sampling=True)
    cb = class_bytes(dm, B)
    peak, peak_kind = _peaks()
    gemm_cls = [k for k in prof if k.startswith("gemm") and k in cb]
    gemm_ms = sum(prof[k][0] for k in gemm_cls)
    gemm_n = sum(prof[k][1] for k in gemm_cls)
    gemm_bytes = sum(cb[k] for k in gemm_cls)
    kern = {
        "gemm_tc_kernel": (gemm_ms, gemm_n, gemm_bytes),
        "wkv_kernel": (prof["wkv"][0], prof["wkv"][1], cb["wkv"]),
    }
    dom = max(kern, key=lambda k: kern[k][0])
    dms, dn, dbytes = kern[dom]
    achieved = (dbytes / dn) / ((dms / dn) / 1e3) / 1e9
    tr = NCU_TRAFFIC.get((dom, wl["shape"])) if not args.layers else None
    traffic = None
    if tr is not None:
        src, sha, _, nbytes = tr
        if _sha([os.path.join(ROOT, f) for f in src]) == sha:
            traffic = nbytes
    sb = step_bytes(dm, B)
    step_gbs = sb / (ms / args.steps / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": _config(wl, dm, args),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes_per_launch": dbytes / dn, "launches_per_step": dn},
        "step_roofline": {"bytes_per_step": sb, "achieved_GBps": step_gbs,
                          "frac_of_8TBps": step_gbs / NOMINAL_HBM_GBS, "frac_of_peak": step_gbs / peak},
        "kernel_ms_per_step": {k: round(v[0], 4) for k, v in prof.items()},
        "e2e": {"value": e2e_val, "unit": "tok/s", "h2d_bytes_per_step": 2 * B * 4, "d2h_bytes_per_step": B * 4,
                "steps": args.e2e_steps},
        "gpu_launches": ctx.step_kernel_count(B, True) * args.steps,
        "prefill": pre,
        "ffn_union": {"nonzero_blocks": nzb, "blocks": totb, "fraction": nzb / max(1, totb),
                      "note": "64-row blocks of the channel-mix value matrix read by the sparse value projection "
                              "over the timed steps; the roofline counts the dense bytes"},
        "clocks": clocks,
    }
    ctx.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(weights, dm, wl, args.cpu_seconds)
    if args.config == "2.9b" and world == 1 and not args.layers and not args.prompt and not args.no_secondary:
        # the metric names both shapes: the 7.2B workload rides along on the same line
        line["secondary"] = secondary("7.2b", max(16, min(64, args.steps)), args, dev, world)
        # the int8 weight variant of the headline workload (a separate row, not the headline)
        line["int8"] = secondary("2.9b", max(16, min(256, args.steps)), args, dev, world, int8=True)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
