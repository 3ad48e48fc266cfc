"""CPU oracle of the RWKV-7 batched decode path (ctypes binding of rwkv7_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg use it; the library under recurrent_decode_gb300/ never imports
it, and it imports nothing from there.

Parity status of each function (what pins it) is written beside it; the tests
that hold the pins live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rwkv7_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")

HEAD_SIZE = 64
LN_EPS = 1e-5
GN_EPS = 64e-5

# Pointer-table order expected by orc_model_new (globals, then per layer).
GLOBAL_ORDER = ["emb", "ln0.w", "ln0.b", "ln_out.w", "ln_out.b", "head"]
LAYER_ORDER = ["ln1.w", "ln1.b", "ln2.w", "ln2.b",
               "att.x_r", "att.x_w", "att.x_k", "att.x_v", "att.x_a", "att.x_g",
               "att.w0", "att.w1", "att.w2", "att.a0", "att.a1", "att.a2",
               "att.v0", "att.v1", "att.v2", "att.g1", "att.g2",
               "att.k_k", "att.k_a", "att.r_k",
               "att.receptance", "att.key", "att.value", "att.output",
               "att.ln_x.w", "att.ln_x.b", "ffn.x_k", "ffn.key", "ffn.value"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP, no fp contraction)."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-std=gnu11", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _OUT)
    return _OUT


_lib = None
_dp = C.POINTER(C.c_double)


class Sampling(C.Structure):
    _fields_ = [("temperature", C.c_float), ("top_p", C.c_float), ("top_k", C.c_int32),
                ("presence", C.c_float), ("frequency", C.c_float),
                ("penalty_decay", C.c_float), ("seed", C.c_uint64), ("greedy", C.c_int32)]


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        L.orc_model_new.restype = C.c_void_p
        L.orc_model_new.argtypes = [C.POINTER(C.c_int32), C.POINTER(C.c_void_p)]
        L.orc_model_free.argtypes = [C.c_void_p]
        L.orc_state_new.restype = C.c_void_p
        L.orc_state_new.argtypes = [C.c_void_p]
        L.orc_state_free.argtypes = [C.c_void_p]
        L.orc_state_doubles.restype = C.c_size_t
        L.orc_state_doubles.argtypes = [C.c_void_p]
        L.orc_state_get.argtypes = [C.c_void_p, C.c_void_p, _dp]
        L.orc_state_set.argtypes = [C.c_void_p, C.c_void_p, _dp]
        L.orc_step.restype = C.c_int
        L.orc_step.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, _dp]
        L.orc_prefill_chunked.restype = C.c_int
        L.orc_prefill_chunked.argtypes = [C.c_void_p, C.c_void_p, C.POINTER(C.c_int32),
                                          C.c_int, C.c_int, _dp]
        L.orc_wkv_step.argtypes = [C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
        L.orc_wkv_chunk.argtypes = [C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
        L.orc_layernorm.argtypes = [C.c_int, _dp, _dp, _dp, C.c_double, _dp]
        L.orc_groupnorm.argtypes = [C.c_int, C.c_int, _dp, _dp, _dp, C.c_double, _dp]
        L.orc_gemv.argtypes = [C.c_int, C.c_int, C.c_void_p, _dp, _dp]
        L.orc_gemv_i8.argtypes = [C.c_int, C.c_int, C.c_void_p, C.c_void_p, _dp, _dp]
        L.orc_model_set_i8.restype = C.c_int
        L.orc_model_set_i8.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
        L.orc_f16_to_f64.restype = C.c_double
        L.orc_f16_to_f64.argtypes = [C.c_uint16]
        L.orc_f64_to_f16.restype = C.c_uint16
        L.orc_f64_to_f16.argtypes = [C.c_double]
        L.orc_philox4x32_10.argtypes = [C.POINTER(C.c_uint32), C.POINTER(C.c_uint32),
                                        C.POINTER(C.c_uint32)]
        L.orc_draw_u64.restype = C.c_uint64
        L.orc_draw_u64.argtypes = [C.c_uint64, C.c_uint64]
        L.orc_exp2.restype = C.c_float
        L.orc_exp2.argtypes = [C.c_float]
        L.orc_sample.restype = C.c_int32
        L.orc_sample.argtypes = [C.c_int, C.c_void_p, C.c_void_p, C.POINTER(Sampling),
                                 C.c_uint64, C.c_void_p, C.c_void_p]
        L.orc_sample_weights.argtypes = [C.c_int, C.c_void_p, C.c_void_p, C.POINTER(Sampling),
                                         C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
        L.orc_pick.restype = C.c_int32
        L.orc_pick.argtypes = [C.c_int, C.c_void_p, C.c_uint64]
        L.orc_set_threads.argtypes = [C.c_int]
        L.orc_get_threads.restype = C.c_int
        _lib = L
    return _lib


def set_threads(n: int):
    lib().orc_set_threads(int(n))


def _d(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_dp)


# ---------------------------------------------------------------- primitives
def f16_to_f64(bits: int) -> float:
    return lib().orc_f16_to_f64(int(bits))


def f64_to_f16(x: float) -> int:
    return lib().orc_f64_to_f16(float(x))


def gemv(W16: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = W x for fp16 W [rows, cols] (fp64 accumulation).  Pinned: numpy matmul."""
    W16 = np.ascontiguousarray(W16, dtype=np.float16)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros(W16.shape[0], np.float64)
    lib().orc_gemv(W16.shape[0], W16.shape[1], W16.ctypes.data, _d(x), _d(y))
    return y


def gemv_i8(q: np.ndarray, scale16: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = W x for the int8 form W[o][i] = q[o][i] * scale[o] (int8 q [rows, cols],
    fp16 scale [rows]).  Pinned: with power-of-two scales W is exact in fp16 and
    the result equals gemv on that fp16 matrix bit for bit."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    scale16 = np.ascontiguousarray(scale16, dtype=np.float16)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros(q.shape[0], np.float64)
    lib().orc_gemv_i8(q.shape[0], q.shape[1], q.ctypes.data, scale16.ctypes.data, _d(x), _d(y))
    return y


def layernorm(x, g, b, eps=LN_EPS):
    """Pinned: torch.nn.functional.layer_norm in fp64; zero mean / unit variance."""
    x = np.ascontiguousarray(x, np.float64); g = np.ascontiguousarray(g, np.float64)
    b = np.ascontiguousarray(b, np.float64); y = np.zeros_like(x)
    lib().orc_layernorm(x.size, _d(x), _d(g), _d(b), eps, _d(y))
    return y


def groupnorm(x, g, b, group, eps=GN_EPS):
    """Pinned: torch.nn.functional.group_norm in fp64."""
    x = np.ascontiguousarray(x, np.float64); g = np.ascontiguousarray(g, np.float64)
    b = np.ascontiguousarray(b, np.float64); y = np.zeros_like(x)
    lib().orc_groupnorm(x.size, group, _d(x), _d(g), _d(b), eps, _d(y))
    return y


def wkv_step(S, r, decay, kh, a, kp, vp):
    """One rank-1 state update of one head; returns (S_new, y).
    Pinned: dense transition-matrix recurrence, closed-form invariants."""
    N = S.shape[0]
    S = np.ascontiguousarray(S, np.float64).copy()
    y = np.zeros(N, np.float64)
    args = [np.ascontiguousarray(v, np.float64) for v in (r, decay, kh, a, kp, vp)]
    lib().orc_wkv_step(N, _d(S), *[_d(v) for v in args], _d(y))
    return S, y


def wkv_chunk(S, r, decay, kh, a, kp, vp):
    """T state updates of one head via chained transition products; inputs [T, N].
    Pinned: equals T calls of wkv_step (chunked-vs-stepwise identity)."""
    N = S.shape[0]
    T = r.shape[0]
    S = np.ascontiguousarray(S, np.float64).copy()
    y = np.zeros((T, N), np.float64)
    args = [np.ascontiguousarray(v, np.float64) for v in (r, decay, kh, a, kp, vp)]
    lib().orc_wkv_chunk(N, T, _d(S), *[_d(v) for v in args], _d(y))
    return S, y


def philox4x32_10(ctr, key):
    """Pinned: the published known-answer vectors of Philox4x32-10."""
    c = (C.c_uint32 * 4)(*ctr)
    k = (C.c_uint32 * 2)(*key)
    o = (C.c_uint32 * 4)()
    lib().orc_philox4x32_10(c, k, o)
    return [int(v) for v in o]


def draw_u64(seed: int, n: int) -> int:
    return int(lib().orc_draw_u64(seed, n))


def exp2(e: float) -> float:
    """Pinned: within 2 ulp of the C library's exp2 over (-126, 0]."""
    return float(lib().orc_exp2(float(e)))


# ---------------------------------------------------------------- model
class Model:
    """RWKV-7 model over fp16 weight arrays (dict name -> ndarray, [out, in]).
    `int8` (optional) maps matrix names to (int8 q [out, in], fp16 scale [out]):
    those matrices are W = q * scale per row (the int8 weight variant) and need
    no entry in `weights`."""

    def __init__(self, weights: dict, dims, int8: dict | None = None):
        self.dims = dims
        self._keep = []
        int8 = int8 or {}
        ptrs = []
        names = list(GLOBAL_ORDER)
        for l in range(dims.n_layer):
            names += [f"blocks.{l}.{n}" for n in LAYER_ORDER]
        i8 = {}
        for n in names:
            if n in int8:
                q = np.ascontiguousarray(int8[n][0], dtype=np.int8)
                sc = np.ascontiguousarray(int8[n][1], dtype=np.float16)
                if sc.shape != (q.shape[0],):
                    raise ValueError(f"{n}: one fp16 scale per row expected")
                i8[n] = (q, sc)
                self._keep += [q, sc]
                ptrs.append(q.ctypes.data)  # the fp16 slot is not read for an int8 matrix
            else:
                a = np.ascontiguousarray(weights[n], dtype=np.float16)
                self._keep.append(a)
                ptrs.append(a.ctypes.data)
        dd = (C.c_int32 * 9)(*dims.as_tuple())
        pp = (C.c_void_p * len(ptrs))(*ptrs)
        self.h = lib().orc_model_new(dd, pp)
        if not self.h:
            raise ValueError("oracle rejected the model dimensions")
        for idx, n in enumerate(names):
            if n in i8:
                q, sc = i8[n]
                if lib().orc_model_set_i8(self.h, idx, q.ctypes.data, sc.ctypes.data) != 0:
                    raise ValueError(f"oracle rejected the int8 tensor {n}")

    def __del__(self):
        if getattr(self, "h", None) and _lib is not None:
            _lib.orc_model_free(self.h)
            self.h = None

    def new_state(self):
        return State(self)


class State:
    """One sequence's recurrent state: wkv [L,H,N,N], shift_att [L,d], shift_ffn [L,d] (fp64)."""

    def __init__(self, model: Model):
        self.m = model
        self.h = lib().orc_state_new(model.h)

    def __del__(self):
        if getattr(self, "h", None) and _lib is not None:
            _lib.orc_state_free(self.h)
            self.h = None

    def get(self):
        dm = self.m.dims
        n = lib().orc_state_doubles(self.m.h)
        out = np.zeros(n, np.float64)
        lib().orc_state_get(self.m.h, self.h, _d(out))
        nw = dm.n_layer * dm.n_head * 64 * 64
        ns = dm.n_layer * dm.d_model
        return (out[:nw].reshape(dm.n_layer, dm.n_head, 64, 64),
                out[nw:nw + ns].reshape(dm.n_layer, dm.d_model),
                out[nw + ns:].reshape(dm.n_layer, dm.d_model))

    def set(self, wkv, shift_att, shift_ffn):
        flat = np.concatenate([np.ravel(wkv), np.ravel(shift_att), np.ravel(shift_ffn)]).astype(np.float64)
        lib().orc_state_set(self.m.h, self.h, _d(flat))

    def copy(self):
        s = State(self.m)
        s.set(*self.get())
        return s

    def step(self, token: int, want_logits: bool = True):
        """Consume one token; return fp64 logits [V] (or None)."""
        lg = np.zeros(self.m.dims.vocab, np.float64) if want_logits else None
        rc = lib().orc_step(self.m.h, self.h, int(token), _d(lg) if lg is not None else None)
        if rc != 0:
            raise ValueError("oracle step rejected its input")
        return lg

    def prefill_chunked(self, tokens, chunk: int = 64, want_logits: bool = True):
        """Consume tokens[T] layer-major with the chunked state update; logits [T, V]."""
        t = np.ascontiguousarray(tokens, np.int32)
        lg = np.zeros((t.size, self.m.dims.vocab), np.float64) if want_logits else None
        rc = lib().orc_prefill_chunked(self.m.h, self.h, t.ctypes.data_as(C.POINTER(C.c_int32)),
                                       t.size, chunk, _d(lg) if lg is not None else None)
        if rc != 0:
            raise ValueError("oracle prefill rejected its input")
        return lg


# ---------------------------------------------------------------- sampler
def _sp(params: dict) -> Sampling:
    return Sampling(float(params.get("temperature", 1.0)), float(params.get("top_p", 1.0)),
                    int(params.get("top_k", 0)), float(params.get("presence", 0.0)),
                    float(params.get("frequency", 0.0)), float(params.get("penalty_decay", 1.0)),
                    int(params.get("seed", 0)), int(bool(params.get("greedy", False))))


def sample_weights(logits32: np.ndarray, occ: np.ndarray, params: dict):
    """(q1, qT, kept) for one row: integer weights before/after temperature and
    the kept set.  Pinned: closed-form weights within one unit, and the top-p
    set is the smallest upward-closed set reaching the mass."""
    V = logits32.size
    lg = np.ascontiguousarray(logits32, np.float32)
    oc = np.ascontiguousarray(occ, np.float32)
    q1 = np.zeros(V, np.uint32); qT = np.zeros(V, np.uint32); kept = np.zeros(V, np.uint32)
    scratch = np.zeros(2 * V, np.uint32)
    sp = _sp(params)
    lib().orc_sample_weights(V, lg.ctypes.data, oc.ctypes.data, C.byref(sp), q1.ctypes.data,
                             qT.ctypes.data, kept.ctypes.data, scratch.ctypes.data)
    return q1, qT, kept.astype(bool)


def pick(weights: np.ndarray, r: int) -> int:
    """First index whose running sum of integer weights exceeds r.
    Pinned: enumerating every r gives the weights as the histogram."""
    w = np.ascontiguousarray(weights, np.uint32)
    return int(lib().orc_pick(w.size, w.ctypes.data, int(r)))


def sample(logits32: np.ndarray, occ: np.ndarray, params: dict, draw_index: int):
    """Sample one token from fp32 logits [V]; updates occ (fp32 [V]) in place
    unless greedy.  Returns (token, kept_mask).  Pinned: greedy / top-k=1 /
    top-p->0 reductions, the penalty under top-k=1, closed-form decayed counts,
    and the empirical histogram on a tiny vocabulary."""
    V = logits32.size
    lg = np.ascontiguousarray(logits32, np.float32)
    assert occ.dtype == np.float32 and occ.flags.c_contiguous
    sp = _sp(params)
    scratch = np.zeros(5 * V, np.uint32)
    kept = np.zeros(V, np.uint32)
    tok = lib().orc_sample(V, lg.ctypes.data, occ.ctypes.data, C.byref(sp), int(draw_index),
                           scratch.ctypes.data, kept.ctypes.data)
    return int(tok), kept.astype(bool)
