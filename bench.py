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
import re
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
# unchanged: kernel -> (source files, sha256 prefix of their code without
# comments and blank lines at capture, workload, bytes)
NCU_TRAFFIC = {
    ("gemm_tc_kernel", "2.9b"): (("recurrent_decode_gb300/csrc/gemm.cu", "recurrent_decode_gb300/csrc/gemm_common.cuh"),
                                  "61ffbca0c231fdc5",
                                  "2.9B shape, B=64: DRAM read+write of the 7 GEMM launches of one step of "
                                  "a 2-layer cut (ncu), scaled to 32 layers + head, "
                                  "per launch", 59051560),
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and blank lines, so that a hash of it
    changes with the code and not with its documentation."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def _sha(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
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
        # the key and value projections as one launch (fused channel mix)
        "gemm_ffn": L * (F * d * f16 + B * d * f16 + B * F * f16) + L * (d * F * f16 + B * F * f16 + 2 * B * d * f32),
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


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline(weights, dm, wl, seconds=15.0, threads=None):
    """The oracle, as it stands, on a bounded sample of the workload: decode
    tokens of one slot (after a short prompt) until ~`seconds` have passed."""
    import oracle
    threads = threads or os.cpu_count() or 1
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
    return {"value": n / dt, "unit": "tok/s", "cores": threads, "kind": "oracle", "cpu_model": cpu_model(),
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


def run_trace_bench(args, wl, ctx=None, name=None):
    """The continuous-batching trace: every request to completion through the
    worker loop (recurrent_decode_gb300.trace); value = generated tokens per
    second of wall time, prefills included.  With ctx (a context of the trace's
    shape with enough slots) the trace runs on it and the line is returned
    instead of printed."""
    import torch
    import recurrent_decode_gb300 as rd
    from recurrent_decode_gb300.trace import Request, run_trace
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    from recurrent_decode_gb300.prefix_cache import PrefixStateCache
    dm = synth.Dims(wl["shape"])
    n_cache = wl.get("cache_slots", 0)
    own = ctx is None
    if own:
        weights = synth.make_weights(wl["shape"])
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
    if own:
        ctx.close()
    ttft = np.array(stats.ttft_s)
    total_in = stats.prefill_tokens + stats.decode_fed_tokens + stats.generated
    line = {"metric": METRIC, "value": world * stats.generated / stats.wall_s, "unit": "tok/s", "n_gpus": world,
            "steps": stats.rounds, "warmup": 0, "ms_per_step": stats.wall_s * 1e3 / max(1, stats.rounds),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": f"continuous-batching trace on the {dm.name} shape ({name or args.config})",
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
    if not own:
        return line
    if rank == 0:
        print(json.dumps(line))
    return 0


def in_graph_times(ctx, slots, tokens, with_sampling=True, reps=3):
    """Per-class time each kernel class adds to the graph-replayed step, from the
    in-graph timeline (rwkv7_step_timeline): launch k adds end_k - end_{k-1}.
    Returns ({class: (ms per step, launches)}, timeline step ms); the median of
    `reps` timeline steps per class."""
    runs = []
    for _ in range(reps):
        t, cls = ctx.step_timeline(slots, tokens, with_sampling=with_sampling)
        add = {}
        for k in range(len(cls)):
            prev = t[k - 1, 3] if k else t[0, 0]
            a = add.setdefault(cls[k], [0.0, 0])
            a[0] += (t[k, 3] - prev) / 1e6
            a[1] += 1
        runs.append((add, (t[-1, 3] - t[0, 0]) / 1e6))
    out = {}
    for c in runs[0][0]:
        out[c] = (statistics.median(r[0][c][0] for r in runs), runs[0][0][c][1])
    return out, statistics.median(r[1] for r in runs)


def union_sweep(dev, fractions=(1.0, 0.75, 0.5, 0.25, 0.1), n_layer=8, B=64, steps=16):
    """The sparse channel-mix value projection on weights whose key rows are
    zero for a chosen share of the 64-row hidden blocks (every layer, seeded):
    those hidden blocks are zero for every slot, so the value projection skips
    their 64 rows of the value matrix.  Per union fraction: the value
    projection's in-graph time per launch when it runs as its own launch (the
    RWKV7_FUSE_FFN=0 configuration), the roofline counting only the union's
    value rows, and the whole step both that way and with the fused channel mix
    the library runs by default (whose speculatively fetched first value stages
    are never skipped)."""
    import torch
    import recurrent_decode_gb300 as rd
    dm = synth.Dims("2.9b", n_layer)
    W = synth.make_weights("2.9b", n_layer=n_layer)
    nblk = dm.d_ffn // 64
    peak, peak_kind = _peaks()
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    tokens = torch.from_numpy(synth.prompt_tokens(dm.vocab, B, 1)[:, 0].copy()).to(dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    res = {}
    for fused in (False, True):
        old = os.environ.get("RWKV7_FUSE_FFN")
        os.environ["RWKV7_FUSE_FFN"] = "1" if fused else "0"  # read when the step graph is captured
        ctx = rd.Rwkv7(dm, B)
        ctx.set_weights(W)
        for s in range(B):
            ctx.set_sampling(s, greedy=True)
        rng = np.random.default_rng(5)
        for f in fractions:
            keep = np.zeros(nblk, bool)
            keep[rng.permutation(nblk)[:max(1, round(f * nblk))]] = True
            for l in range(n_layer):
                k = W[f"blocks.{l}.ffn.key"].copy()
                k.reshape(nblk, 64, dm.d_model)[~keep] = 0
                ctx.set_weight(f"blocks.{l}.ffn.key", k)
            for _ in range(3):
                ctx.decode_step(slots, tokens, None, nxt)
            ctx.synchronize()
            ctx.ffn_union_stats()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                ctx.decode_step(slots, tokens, None, nxt)
            e1.record()
            torch.cuda.synchronize()
            nz, tot = ctx.ffn_union_stats()
            ig, _ = in_graph_times(ctx, slots, tokens, with_sampling=False)
            res[(fused, f)] = (nz / max(1, tot), e0.elapsed_time(e1) / steps, ig)
        ctx.close()
        if old is None:
            os.environ.pop("RWKV7_FUSE_FFN", None)
        else:
            os.environ["RWKV7_FUSE_FFN"] = old
    rows = []
    for f in fractions:
        union, step_ms, ig = res[(False, f)]
        _, step_fused, igf = res[(True, f)]
        v_ms, v_n = ig["gemm_value"]
        vbytes = union * dm.d_model * dm.d_ffn * 2  # value rows of the union, per launch
        rows.append({"union_fraction": union, "value_us_per_launch": 1e3 * v_ms / v_n,
                     "key_us_per_launch": 1e3 * ig["gemm_key"][0] / ig["gemm_key"][1],
                     "step_ms": step_ms,
                     "union_roofline_GBps": vbytes / (v_ms / v_n / 1e3) / 1e9,
                     "union_roofline_frac": vbytes / (v_ms / v_n / 1e3) / 1e9 / peak,
                     "fused_ffn_us_per_launch": 1e3 * igf["gemm_ffn"][0] / igf["gemm_ffn"][1],
                     "fused_step_ms": step_fused})
    return {"shape": f"2.9b, {n_layer} layers, B={B}", "peak_kind": peak_kind, "points": rows,
            "note": "ffn.key rows zeroed for (1 - fraction) of the 64-row hidden blocks; times are in-graph per launch "
                    "(rwkv7_step_timeline); value_us: the value projection as its own launch; fused: key + value "
                    "as one launch; the roofline counts union rows only"}


def shrink_sweep(ctx, dm, dev, batches=(256, 128, 64, 32, 16, 8, 4, 2, 1), steps=20):
    """Batch shrink: the same context decoding B = 256 ... 1 slots.  Per B: the
    first step at that B timed on the host (it captures and instantiates the
    step's CUDA graph), then ms/step of the replayed graph and the whole-step
    roofline."""
    import torch
    peak, peak_kind = _peaks()
    rows = []
    for B in batches:
        slots = torch.arange(B, dtype=torch.int32, device=dev)
        tokens = torch.from_numpy(synth.prompt_tokens(dm.vocab, B, 1, seed=3)[:, 0].copy()).to(dev)
        nxt = torch.empty(B, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ctx.decode_step(slots, tokens, None, nxt)
        torch.cuda.synchronize()
        first_ms = (time.perf_counter() - t0) * 1e3
        for _ in range(3):
            ctx.decode_step(slots, tokens, None, nxt)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            ctx.decode_step(slots, tokens, None, nxt)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        gbs = step_bytes(dm, B) / (ms / 1e3) / 1e9
        rows.append({"B": B, "first_step_ms": first_ms, "ms_per_step": ms, "tok_s": B / (ms / 1e3),
                     "step_GBps": gbs, "frac_of_peak": gbs / peak, "frac_of_8TBps": gbs / NOMINAL_HBM_GBS})
    ctx.synchronize()
    return {"shape": dm.name, "peak_kind": peak_kind, "points": rows,
            "note": "greedy steps; first_step_ms includes capturing and instantiating the step graph for a B "
                    "not seen before"}


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
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run a model with this many layers of the shape's sizes")
    ap.add_argument("--prompt", type=int, default=0, help="profiling only: override the prompt length")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the 7.2B-shape measurement added to the 2.9B line")
    ap.add_argument("--mode", type=int, default=-1,
                    help="implementation: 0 CUDA-graph replay, 1 direct launches, 2 CUDA-core cross-check "
                         "(default: library default)")
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
    full = args.config == "2.9b" and world == 1 and not args.layers and not args.prompt and not args.no_secondary
    # the headline context keeps 256 slots so that the batch-shrink sweep and the
    # trace can run on it after the timed steps (slots beyond B are untouched then)
    ctx = rd.Rwkv7(dm, 256 if full else B)
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

    # time each kernel class adds to the graph-replayed step (in-graph timeline),
    # and the device time of each class in one directly launched step (events)
    ig, tl_ms = in_graph_times(ctx, slots, tokens, with_sampling=True)
    prof = ctx.profile_step(slots, tokens, with_sampling=True)
    cb = class_bytes(dm, B)
    peak, peak_kind = _peaks()

    def family(times):
        gemm_cls = [k for k in times if k.startswith("gemm") and k in cb]
        # the r, k, v launch carries the LoRA up projections too when they are
        # fused into it (no gemm_lora launches in the step)
        cbx = dict(cb)
        if "gemm_proj" in times and "gemm_lora" not in times:
            cbx["gemm_proj"] = cb["gemm_proj"] + cb["gemm_lora"]
        return {"gemm_tc_kernel": (sum(times[k][0] for k in gemm_cls), sum(times[k][1] for k in gemm_cls),
                                   sum(cbx[k] for k in gemm_cls)),
                "wkv_kernel": (times["wkv"][0], times["wkv"][1], cb["wkv"])}

    kern = family(ig)
    dom = max(kern, key=lambda k: kern[k][0])
    dms, dn, dbytes = kern[dom]
    achieved = (dbytes / dn) / ((dms / dn) / 1e3) / 1e9
    iso_ms, iso_n, _ = family(prof)[dom]
    iso_achieved = (dbytes / dn) / ((iso_ms / iso_n) / 1e3) / 1e9
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
                     "algorithmic_bytes_per_launch": dbytes / dn, "launches_per_step": dn,
                     "kernel_ms_per_step": dms,
                     "timing": "in-graph: the time this kernel's launches add to the replayed step "
                               "(rwkv7_step_timeline, GPU global timer)",
                     "isolated": {"achieved": iso_achieved, "frac": iso_achieved / peak, "ms_per_step": iso_ms,
                                  "timing": "directly launched step, CUDA events around each launch"}},
        "step_roofline": {"bytes_per_step": sb, "achieved_GBps": step_gbs,
                          "frac_of_8TBps": step_gbs / NOMINAL_HBM_GBS, "frac_of_peak": step_gbs / peak},
        "in_graph_ms_per_step": {k: round(v[0], 4) for k, v in ig.items()},
        "timeline_step_ms": tl_ms,
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
    if full:
        line["batch_shrink"] = shrink_sweep(ctx, dm, dev)
        # the continuous-batching trace at the pages' measured prefill mix, on the same context
        tr = run_trace_bench(args, synth.WORKLOADS["trace-3pct"], ctx=ctx, name="trace-3pct")
        line["trace_3pct"] = {"value": tr["value"], "unit": tr["unit"], "config": tr["config"],
                              "trace": tr["trace"], "clocks": tr["clocks"]}
    ctx.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb_all = cpu_baseline(weights, dm, wl, args.cpu_seconds)
        cb_one = cpu_baseline(weights, dm, wl, args.cpu_seconds / 2, threads=1)
        cb_all["single_thread"] = {"value": cb_one["value"], "cores": 1, "sample": cb_one["sample"]}
        line["cpu_baseline"] = cb_all
    if full:
        # the metric names both shapes: the 7.2B workload rides along on the same line
        line["secondary"] = secondary("7.2b", max(16, min(64, args.steps)), args, dev, world)
        # the int8 weight variant of the headline workload (a separate row, not the headline)
        line["int8"] = secondary("2.9b", max(16, min(256, args.steps)), args, dev, world, int8=True)
        line["ffn_union_sweep"] = union_sweep(dev)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
