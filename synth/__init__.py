"""Seeded synthetic inputs for the RWKV-7 decode path: model shapes, random-init
weights, prompt token ids and the raw weight-file container.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It holds no step of the model's arithmetic: only shapes, seeded
random draws (numpy PCG64) and a byte container.

Shapes follow the workloads the source pages measure on ("RWKV 批量推理中 Prefill
的正确打开方式", §二 measured-throughput table: 2.9B and 7.2B RWKV-7 models); the
pages publish no weights, so every tensor is drawn at random:
  * matrices ~ N(0, 0.02) rounded to fp16; w0 ~ U(-6, -1);
  * token-shift mixes mu ~ U(0, 1); k_k, k_a ~ U(0.5, 1.5); r_k ~ N(0, 0.1);
    a0, v0 ~ U(-1, 1); LayerNorm / GroupNorm scales ~ U(0.8, 1.2) and shifts
    ~ U(-0.1, 0.1) (non-trivial so that a dropped affine term shows up).
All parameters are stored as fp16 (the pages' models are "CUDA fp16" .pth
checkpoints: RWKV-Runner Albatross article, "Albatross 是什么").
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HEAD_SIZE = 64

# name -> (n_layer, d_model, d_ffn, vocab, (lora_w, lora_a, lora_v, lora_g))
SHAPES = {
    "tiny": (2, 128, 512, 1024, (16, 16, 16, 32)),
    "0.1b": (12, 768, 3072, 65536, (64, 64, 32, 128)),
    "2.9b": (32, 2560, 10240, 65536, (96, 96, 64, 320)),
    "7.2b": (32, 4096, 16384, 65536, (128, 128, 96, 480)),
}

# Decode workloads: shape, slots in the step B, prompt length, decode steps, sampling.
# Sampling defaults (temperature 1.0, top_p 0.3, top_k 0, frequency 1, decay 0.996,
# presence 0) are the Albatross adapter's defaults (RWKV-Runner Albatross article,
# "适配器Runner 与异步引擎之间的桥").
WORKLOADS = {
    "tiny": dict(shape="tiny", B=1, prompt=8, steps=16, greedy=True),
    "0.1b": dict(shape="0.1b", B=32, prompt=64, steps=256, greedy=False,
                 temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0,
                 penalty_decay=0.996),
    "2.9b": dict(shape="2.9b", B=64, prompt=128, steps=512, greedy=True),
    "7.2b": dict(shape="7.2b", B=256, prompt=64, steps=256, greedy=False,
                 temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0,
                 penalty_decay=0.996),
    # continuous-batching traces: 256 requests through 128 slots, one prefill phase
    # per 5 decode rounds; prompts as written (U[20, 2000]) or as the pages'
    # measured mix (~3 % prefill tokens: U[20, 138])
    "trace": dict(shape="2.9b", n_slots=128, n_req=256, prompt_range=(20, 2000), out_range=(1000, 3000),
                  decode_prefill_ratio=5, min_forward_seq_len=10, temperature=1.0, top_p=0.3, top_k=0,
                  presence=0.0, frequency=1.0, penalty_decay=0.996),
    "trace-3pct": dict(shape="2.9b", n_slots=128, n_req=256, prompt_range=(20, 138), out_range=(1000, 3000),
                       decode_prefill_ratio=5, min_forward_seq_len=10, temperature=1.0, top_p=0.3, top_k=0,
                       presence=0.0, frequency=1.0, penalty_decay=0.996),
    # every prompt = one shared 1024-token prefix (a system prompt) + its own
    # tail; run with and without the prefix-state cache (8 cache slots)
    "trace-prefix": dict(shape="2.9b", n_slots=64, n_req=128, prompt_range=(20, 138), out_range=(64, 128),
                         shared_prefix=1024, cache_slots=8, decode_prefill_ratio=5, min_forward_seq_len=10,
                         temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0,
                         penalty_decay=0.996),
}

WEIGHT_SEED = 0
PROMPT_SEED = 1
TRACE_SEED = 2
SAMPLING_SEED_BASE = 1000

_CHUNK = 1 << 22  # elements per independent RNG stream (fixed: results do not depend on threads)


class Dims:
    """Model dimensions of one named shape."""

    def __init__(self, name: str, n_layer: int | None = None):
        """n_layer, if given, replaces the shape's layer count (a shorter model
        with the same per-layer sizes, for small profiling cases)."""
        nl, d, f, v, lora = SHAPES[name]
        self.name = name
        self.n_layer = int(n_layer) if n_layer else nl
        self.d_model = d
        self.head_size = HEAD_SIZE
        self.n_head = d // HEAD_SIZE
        self.d_ffn = f
        self.vocab = v
        self.lora_w, self.lora_a, self.lora_v, self.lora_g = lora

    def as_tuple(self):
        return (self.n_layer, self.d_model, self.head_size, self.d_ffn, self.vocab,
                self.lora_w, self.lora_a, self.lora_v, self.lora_g)


def tensor_specs(dims: Dims):
    """Ordered list of (name, shape, init) for every parameter.

    Matrices are [out, in] (a row per output feature).  init is one of
    ("normal", std) or ("uniform", lo, hi).
    """
    d, f, v = dims.d_model, dims.d_ffn, dims.vocab
    rw, ra, rv, rg = dims.lora_w, dims.lora_a, dims.lora_v, dims.lora_g
    mat = ("normal", 0.02)
    gam = ("uniform", 0.8, 1.2)
    bet = ("uniform", -0.1, 0.1)
    specs = [("emb", (v, d), mat), ("ln0.w", (d,), gam), ("ln0.b", (d,), bet)]
    for l in range(dims.n_layer):
        p = f"blocks.{l}."
        specs += [
            (p + "ln1.w", (d,), gam), (p + "ln1.b", (d,), bet),
            (p + "ln2.w", (d,), gam), (p + "ln2.b", (d,), bet),
            (p + "att.x_r", (d,), ("uniform", 0.0, 1.0)),
            (p + "att.x_w", (d,), ("uniform", 0.0, 1.0)),
            (p + "att.x_k", (d,), ("uniform", 0.0, 1.0)),
            (p + "att.x_v", (d,), ("uniform", 0.0, 1.0)),
            (p + "att.x_a", (d,), ("uniform", 0.0, 1.0)),
            (p + "att.x_g", (d,), ("uniform", 0.0, 1.0)),
            (p + "att.w0", (d,), ("uniform", -6.0, -1.0)),
            (p + "att.w1", (rw, d), mat), (p + "att.w2", (d, rw), mat),
            (p + "att.a0", (d,), ("uniform", -1.0, 1.0)),
            (p + "att.a1", (ra, d), mat), (p + "att.a2", (d, ra), mat),
            (p + "att.v0", (d,), ("uniform", -1.0, 1.0)),
            (p + "att.v1", (rv, d), mat), (p + "att.v2", (d, rv), mat),
            (p + "att.g1", (rg, d), mat), (p + "att.g2", (d, rg), mat),
            (p + "att.k_k", (d,), ("uniform", 0.5, 1.5)),
            (p + "att.k_a", (d,), ("uniform", 0.5, 1.5)),
            (p + "att.r_k", (d,), ("normal", 0.1)),
            (p + "att.receptance", (d, d), mat),
            (p + "att.key", (d, d), mat),
            (p + "att.value", (d, d), mat),
            (p + "att.output", (d, d), mat),
            (p + "att.ln_x.w", (d,), gam), (p + "att.ln_x.b", (d,), bet),
            (p + "ffn.x_k", (d,), ("uniform", 0.0, 1.0)),
            (p + "ffn.key", (f, d), mat),
            (p + "ffn.value", (d, f), mat),
        ]
    specs += [("ln_out.w", (d,), gam), ("ln_out.b", (d,), bet), ("head", (v, d), mat)]
    return specs


def n_params(dims: Dims) -> int:
    return sum(int(np.prod(s)) for _, s, _ in tensor_specs(dims))


def _fill(out16: np.ndarray, init, seed: int, tid: int, c0: int, c1: int):
    flat = out16.reshape(-1)
    for c in range(c0, c1):
        lo = c * _CHUNK
        hi = min(flat.size, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, c])))
        if init[0] == "normal":
            vals = g.standard_normal(hi - lo, dtype=np.float32) * np.float32(init[1])
        else:
            lo_v, hi_v = init[1], init[2]
            vals = g.random(hi - lo, dtype=np.float32) * np.float32(hi_v - lo_v) + np.float32(lo_v)
        flat[lo:hi] = vals.astype(np.float16)


def make_weights(shape: str, seed: int = WEIGHT_SEED, threads: int | None = None,
                 overrides: dict | None = None, n_layer: int | None = None):
    """Return {name: fp16 ndarray} for the named shape, drawn from `seed`.

    Every tensor (and every 4 Mi-element chunk of it) has its own PCG64 stream
    keyed by (seed, tensor index, chunk index), so the result is the same for any
    thread count.  `overrides` maps name -> callable(ndarray) that edits a tensor
    in place after drawing (used by tests that zero parts of the model).
    `n_layer` shortens the model as in Dims.
    """
    dims = Dims(shape, n_layer)
    specs = tensor_specs(dims)
    out = {name: np.empty(shp, dtype=np.float16) for name, shp, _ in specs}
    jobs = []
    for tid, (name, shp, init) in enumerate(specs):
        nchunks = (int(np.prod(shp)) + _CHUNK - 1) // _CHUNK
        for c0 in range(0, nchunks, 4):
            jobs.append((name, init, tid, c0, min(nchunks, c0 + 4)))
    nthr = threads or min(32, os.cpu_count() or 1)
    if nthr <= 1 or len(jobs) < 8:
        for name, init, tid, c0, c1 in jobs:
            _fill(out[name], init, seed, tid, c0, c1)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(lambda j: _fill(out[j[0]], j[1], seed, j[2], j[3], j[4]), jobs))
    if overrides:
        for name, fn in overrides.items():
            fn(out[name])
    return out


# The int8 weight variant: these matrices are given as int8 values with one
# fp16 scale per output row (W = q * scale); everything else stays fp16.
I8_LAYER_MATRICES = ("att.w1", "att.w2", "att.a1", "att.a2", "att.v1", "att.v2", "att.g1", "att.g2",
                     "att.receptance", "att.key", "att.value", "att.output", "ffn.key", "ffn.value")
I8_Q_STD = float(np.sqrt((255.0 ** 2 - 1.0) / 12.0))  # std of q uniform on [-127, 127]


def i8_matrix_names(dims: Dims):
    return [f"blocks.{l}.{m}" for l in range(dims.n_layer) for m in I8_LAYER_MATRICES] + ["head"]


def _fill_i8(q: np.ndarray, seed: int, tid: int, c0: int, c1: int):
    flat = q.reshape(-1)
    for c in range(c0, c1):
        lo = c * _CHUNK
        hi = min(flat.size, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, c, 8])))
        flat[lo:hi] = g.integers(-127, 128, size=hi - lo, dtype=np.int8)


def make_weights_i8(shape: str, seed: int = WEIGHT_SEED, threads: int | None = None,
                    n_layer: int | None = None, pow2_scales: bool = False):
    """Weights of the int8 variant for the named shape: ({name: fp16 ndarray} for
    every tensor that is not an int8 matrix -- the same values make_weights draws
    -- , {name: (int8 q [out, in], fp16 scale [out])}).  q is uniform on
    [-127, 127]; a row's scale is 0.02 / I8_Q_STD * U(0.75, 1.25), so the matrix
    has about the fp16 variant's N(0, 0.02) spread; with pow2_scales every scale
    is 2^-12 or 2^-13 instead (q * scale is then exact in fp16)."""
    dims = Dims(shape, n_layer)
    specs = tensor_specs(dims)
    i8set = set(i8_matrix_names(dims))
    out = {name: np.empty(shp, dtype=np.float16) for name, shp, _ in specs if name not in i8set}
    q8 = {name: np.empty(shp, dtype=np.int8) for name, shp, _ in specs if name in i8set}
    jobs = []
    for tid, (name, shp, init) in enumerate(specs):
        nchunks = (int(np.prod(shp)) + _CHUNK - 1) // _CHUNK
        for c0 in range(0, nchunks, 4):
            jobs.append((name, init, tid, c0, min(nchunks, c0 + 4)))

    def run(j):
        name, init, tid, c0, c1 = j
        if name in i8set:
            _fill_i8(q8[name], seed, tid, c0, c1)
        else:
            _fill(out[name], init, seed, tid, c0, c1)

    nthr = threads or min(32, os.cpu_count() or 1)
    if nthr <= 1 or len(jobs) < 8:
        for j in jobs:
            run(j)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(run, jobs))
    int8 = {}
    for tid, (name, shp, _) in enumerate(specs):
        if name not in i8set:
            continue
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid, 9])))
        if pow2_scales:
            sc = np.where(g.random(shp[0]) < 0.5, 2.0 ** -12, 2.0 ** -13)
        else:
            sc = 0.02 / I8_Q_STD * (0.75 + 0.5 * g.random(shp[0]))
        int8[name] = (q8[name], sc.astype(np.float16))
    return out, int8


def prompt_tokens(vocab: int, n_seq: int, length: int, seed: int = PROMPT_SEED):
    """Uniform random token ids, one independent stream per sequence: int32 [n_seq, length]."""
    rows = []
    for s in range(n_seq):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, s])))
        rows.append(g.integers(0, vocab, size=length, dtype=np.int64).astype(np.int32))
    return np.stack(rows) if rows else np.zeros((0, length), np.int32)


def random_logits(rows: int, vocab: int, seed: int, scale: float = 1.0):
    """fp32 logits ~ N(0, scale^2) for sampler tests."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 77])))
    return (g.standard_normal((rows, vocab), dtype=np.float32) * np.float32(scale)).astype(np.float32)


def trace_requests(n_req: int, prompt_lo: int, prompt_hi: int, out_lo: int, out_hi: int,
                   seed: int = TRACE_SEED):
    """Continuous-batching trace: per request (prompt_len, output_len), uniform."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed])))
    p = g.integers(prompt_lo, prompt_hi + 1, size=n_req)
    o = g.integers(out_lo, out_hi + 1, size=n_req)
    return [(int(a), int(b)) for a, b in zip(p, o)]


# ---------------------------------------------------------------------------
# Raw weight file: a text header then 256-byte-aligned little-endian tensors.
#   "RWKV7W01\n" "<n>\n" then n lines "name dtype d0xd1.. offset nbytes\n", "END\n",
#   zero padding to 4096 bytes; offsets are relative to the 4096-byte data start.
# ---------------------------------------------------------------------------
MAGIC = b"RWKV7W01\n"
DATA_START = 4096


def write_weight_file(path: str, weights: dict):
    lines, off = [], 0
    for name, arr in weights.items():
        assert arr.dtype == np.float16
        shape = "x".join(str(s) for s in arr.shape)
        lines.append(f"{name} f16 {shape} {off} {arr.nbytes}\n")
        off += (arr.nbytes + 255) // 256 * 256
    header = MAGIC + f"{len(lines)}\n".encode() + "".join(lines).encode() + b"END\n"
    if len(header) > DATA_START:
        raise ValueError("weight file header too long")
    with open(path, "wb") as fh:
        fh.write(header + b"\0" * (DATA_START - len(header)))
        pos = 0
        for arr in weights.values():
            fh.write(np.ascontiguousarray(arr).tobytes())
            pad = (arr.nbytes + 255) // 256 * 256 - arr.nbytes
            fh.write(b"\0" * pad)
            pos += arr.nbytes + pad


def read_weight_file(path: str):
    with open(path, "rb") as fh:
        head = fh.read(DATA_START)
        if not head.startswith(MAGIC):
            raise ValueError("not an RWKV7W01 weight file")
        text = head[len(MAGIC):].split(b"END\n")[0].decode().splitlines()
        n = int(text[0])
        out = {}
        for ln in text[1:1 + n]:
            name, dt, shape, off, nb = ln.split()
            shp = tuple(int(s) for s in shape.split("x"))
            fh.seek(DATA_START + int(off))
            out[name] = np.frombuffer(fh.read(int(nb)), dtype=np.float16).reshape(shp).copy()
        return out


__all__ = ["SHAPES", "WORKLOADS", "Dims", "tensor_specs", "n_params", "make_weights",
           "prompt_tokens", "random_logits", "trace_requests", "write_weight_file",
           "make_weights_i8", "i8_matrix_names", "I8_LAYER_MATRICES",
           "read_weight_file"]
