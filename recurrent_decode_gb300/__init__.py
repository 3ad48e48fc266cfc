"""Python binding of librwkv7 (include/rwkv7.h): the GB300 RWKV-7 batched decode path.

Argument marshalling only -- every step of the path runs in the library's
sm_103a kernels.  torch is used for device memory and streams: device arguments
are torch CUDA tensors, passed to the C ABI as raw pointers on the current
stream.  Importing this package fails loudly if the library has not been built
(python -m recurrent_decode_gb300.build); there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import LIB as LIB_PATH
from .build import build

OK, EINVAL, ESHAPE, ENOMEM, ECUDA, ETIMEOUT, ESTATE = 0, -1, -2, -3, -4, -5, -6
MAX_STEP_BATCH = 256


class RWKV7Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"rwkv7 error {code}: {msg}")
        self.code = code


class Config(C.Structure):
    _fields_ = [("n_layer", C.c_int32), ("d_model", C.c_int32), ("head_size", C.c_int32),
                ("d_ffn", C.c_int32), ("vocab", C.c_int32), ("lora_w", C.c_int32),
                ("lora_a", C.c_int32), ("lora_v", C.c_int32), ("lora_g", C.c_int32),
                ("n_slots", C.c_int32)]


class Sampling(C.Structure):
    _fields_ = [("temperature", C.c_float), ("top_p", C.c_float), ("top_k", C.c_int32),
                ("presence", C.c_float), ("frequency", C.c_float), ("penalty_decay", C.c_float),
                ("seed", C.c_uint64), ("greedy", C.c_int32)]


# name -> (restype, argtypes): the whole exported ABI
_VP, _I32P, _FP = C.c_void_p, C.POINTER(C.c_int32), C.c_void_p
ALLOC_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_size_t, C.POINTER(C.c_void_p))
FREE_FN = C.CFUNCTYPE(None, C.c_void_p, C.c_void_p)
SIGNATURES = {
    "rwkv7_create": (C.c_int, [C.POINTER(Config), C.c_void_p, C.POINTER(C.c_void_p)]),
    "rwkv7_create_ex": (C.c_int, [C.POINTER(Config), C.c_int32, C.c_void_p, C.POINTER(C.c_void_p)]),
    "rwkv7_weight_bits": (C.c_int32, [_VP]),
    "rwkv7_set_weight_i8": (C.c_int, [_VP, C.c_char_p, C.c_void_p, C.c_size_t, C.c_void_p, C.c_size_t]),
    "rwkv7_destroy": (None, [_VP]),
    "rwkv7_last_error": (C.c_char_p, [_VP]),
    "rwkv7_set_weight": (C.c_int, [_VP, C.c_char_p, C.c_void_p, C.c_size_t]),
    "rwkv7_load_weights": (C.c_int, [_VP, C.c_char_p]),
    "rwkv7_slot_reset": (C.c_int, [_VP, C.c_int32]),
    "rwkv7_slot_swap": (C.c_int, [_VP, C.c_int32, C.c_int32]),
    "rwkv7_slot_copy": (C.c_int, [_VP, C.c_int32, C.c_int32]),
    "rwkv7_slot_set_sampling": (C.c_int, [_VP, C.c_int32, C.POINTER(Sampling)]),
    "rwkv7_slot_state_bytes": (C.c_size_t, [_VP]),
    "rwkv7_slot_get_state": (C.c_int, [_VP, C.c_int32, C.c_void_p, C.c_size_t]),
    "rwkv7_slot_set_state": (C.c_int, [_VP, C.c_int32, C.c_void_p, C.c_size_t]),
    "rwkv7_prefill_seq": (C.c_int, [_VP, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p]),
    "rwkv7_decode_step": (C.c_int, [_VP, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "rwkv7_decode_step_host": (C.c_int, [_VP, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "rwkv7_sample_batch": (C.c_int, [_VP, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p]),
    "rwkv7_sample_rows_static": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                           C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                           C.POINTER(C.c_char_p)]),
    "rwkv7_ffn_union_stats": (C.c_int, [_VP, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]),
    "rwkv7_synchronize": (C.c_int, [_VP]),
    "rwkv7_set_mode": (C.c_int, [_VP, C.c_int32]),
    "rwkv7_get_io_buffers": (C.c_int, [_VP, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                       C.POINTER(C.c_void_p), C.POINTER(C.c_void_p)]),
    "rwkv7_step_kernel_count": (C.c_int32, [_VP, C.c_int32, C.c_int32]),
    "rwkv7_profile_step": (C.c_int, [_VP, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p,
                                     C.c_void_p, C.c_int32]),
    "rwkv7_set_device_allocator": (C.c_int, [ALLOC_FN, FREE_FN, C.c_void_p]),
    "rwkv7_debug_latch_error": (C.c_int, [_VP, C.c_uint32]),
    "rwkv7_step_timeline": (C.c_int, [_VP, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p,
                                      C.c_void_p, C.c_int32, C.POINTER(C.c_int32)]),
}

SAMPLE_STATIC_MAX_ELEMS = 1 << 22

PROF_CLASSES = ["embed", "ln_mix", "gemm_proj", "gemm_lora", "wkv", "gemm_out", "gemm_key", "gemm_value",
                "ln_out", "gemm_head", "sampler", "lora_fin", "gemm_ffn"]

_lib = None


def load_library(path: str = LIB_PATH):
    """Load librwkv7.so (ctypes).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"librwkv7.so not built at {path}; run python -m recurrent_decode_gb300.build")
        L = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t, dtype, what):
    """Device pointer of a contiguous torch CUDA tensor of the given dtype (or None)."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{what} must be a contiguous {dtype} tensor")
    return C.c_void_p(t.data_ptr())


def sampling_table(params) -> np.ndarray:
    """Pack a list of sampling-parameter dicts (keys of Rwkv7.set_sampling) into
    the byte image of an rwkv7_sampling array, ready to copy to the device for
    sample_rows_static."""
    arr = (Sampling * len(params))()
    for i, p in enumerate(params):
        q = dict(temperature=1.0, top_p=0.3, top_k=0, presence=0.0, frequency=1.0, penalty_decay=0.996,
                 seed=0, greedy=False)
        q.update(p)
        arr[i] = Sampling(q["temperature"], q["top_p"], q["top_k"], q["presence"], q["frequency"],
                          q["penalty_decay"], q["seed"], int(bool(q["greedy"])))
    return np.frombuffer(bytes(arr), dtype=np.uint8).copy()


def sample_rows_static(logits, rows, occ, params, ndraw, next_out, err, stream=None):
    """rwkv7_sample_rows_static: sample one token per row of logits [B][V] with
    the per-sequence entries rows[b] of occ [n_rows][V] fp32, params (uint8
    device image of an rwkv7_sampling array, see sampling_table) and ndraw
    [n_rows] int64 (the uint64 draw counters), writing next_out [B] int32 and
    OR-ing error flags into err [1] int32.  The library allocates nothing for
    this call; its scratch is a fixed 16 MiB device array, so B * V must not
    exceed SAMPLE_STATIC_MAX_ELEMS.  Every buffer must be on one device; the
    call runs with that device current.  stream: a torch.cuda.Stream of that
    device, or None (its current stream)."""
    import torch
    lib = load_library()
    B, V = int(logits.shape[0]), int(logits.shape[1])
    n_rows = int(occ.shape[0])
    if params.dtype != torch.uint8 or params.numel() != n_rows * C.sizeof(Sampling):
        raise TypeError("params must be a uint8 tensor holding n_rows rwkv7_sampling records")
    if logits.dim() != 2 or occ.dim() != 2 or occ.shape[1] != V or rows.numel() != B \
            or next_out.numel() != B or ndraw.numel() != n_rows or err.numel() != 1:
        raise ValueError("shapes: logits [B][V], rows [B], occ [n_rows][V], ndraw [n_rows], next_out [B], err [1]")
    dev = logits.device
    for name, t in (("rows", rows), ("occ", occ), ("params", params), ("ndraw", ndraw), ("next_out", next_out),
                    ("err", err)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, logits on {dev}: every buffer must be on one device")
    if stream is not None and stream.device != dev:
        raise ValueError(f"the stream belongs to {stream.device}, the buffers to {dev}")
    msg = C.c_char_p()
    with torch.cuda.device(dev):  # the library resolves its scratch and launches on the current device
        st = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = lib.rwkv7_sample_rows_static(_ptr(logits, torch.float32, "logits"), _ptr(rows, torch.int32, "rows"),
                                          B, V, n_rows, _ptr(occ, torch.float32, "occ"),
                                          _ptr(params, torch.uint8, "params"), _ptr(ndraw, torch.int64, "ndraw"),
                                          _ptr(next_out, torch.int32, "next_out"), _ptr(err, torch.int32, "err"),
                                          C.c_void_p(st.cuda_stream), C.byref(msg))
    if rc != OK:
        raise RWKV7Error(rc, (msg.value or b"").decode())


_allocator_refs = None  # keeps the installed ctypes callbacks alive


def set_device_allocator(alloc=None, free=None):
    """rwkv7_set_device_allocator: contexts created from now on take their device
    memory from alloc(nbytes) -> device address (int; 0 or an exception refuses)
    and return it through free(address).  No arguments restores cudaMalloc."""
    global _allocator_refs
    lib = load_library()
    if alloc is None and free is None:
        rc = lib.rwkv7_set_device_allocator(ALLOC_FN(), FREE_FN(), None)
        _allocator_refs = None
    else:
        def _a(_user, nbytes, out):
            try:
                p = int(alloc(int(nbytes)) or 0)
            except Exception:
                p = 0
            out[0] = p or None
            return 0 if p else 1

        def _f(_user, ptr):
            free(int(ptr or 0))
        refs = (ALLOC_FN(_a), FREE_FN(_f))
        rc = lib.rwkv7_set_device_allocator(refs[0], refs[1], None)
        if rc == OK:
            _allocator_refs = refs
    if rc != OK:
        raise RWKV7Error(rc, "alloc and free must both be given or both omitted")


class Rwkv7:
    """One library context: device weights + a pool of n_slots state slots."""

    def __init__(self, dims, n_slots: int, stream=None, weight_bits: int = 16):
        """dims: object with n_layer, d_model, head_size, d_ffn, vocab, lora_w/a/v/g
        (e.g. synth.Dims).  stream: torch.cuda.Stream or None (current stream).
        weight_bits: 16 (fp16 matrices) or 8 (int8 matrices with fp16 row scales,
        rwkv7_create_ex)."""
        import torch
        self.lib = load_library()
        self.dims = dims
        self.n_slots = int(n_slots)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        cfg = Config(dims.n_layer, dims.d_model, dims.head_size, dims.d_ffn, dims.vocab,
                     dims.lora_w, dims.lora_a, dims.lora_v, dims.lora_g, self.n_slots)
        h = C.c_void_p()
        self.weight_bits = int(weight_bits)
        rc = self.lib.rwkv7_create_ex(C.byref(cfg), self.weight_bits, C.c_void_p(self.stream.cuda_stream),
                                      C.byref(h))
        self.h = h
        if rc != OK:
            msg = self.lib.rwkv7_last_error(h).decode() if h.value else "invalid configuration"
            if h.value:
                self.lib.rwkv7_destroy(h)
            self.h = C.c_void_p()
            raise RWKV7Error(rc, msg)

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            self.lib.rwkv7_destroy(self.h)
            self.h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc):
        if rc != OK:
            raise RWKV7Error(rc, self.lib.rwkv7_last_error(self.h).decode())

    # ------------------------------------------------------------ weights
    def set_weight(self, name: str, arr: np.ndarray):
        a = np.ascontiguousarray(arr, dtype=np.float16)
        self._check(self.lib.rwkv7_set_weight(self.h, name.encode(), a.ctypes.data, a.nbytes))

    def set_weights(self, weights: dict, int8: dict | None = None):
        """weights: {name: fp16 array}; int8 (int8 context): {name: (int8 q [out, in],
        fp16 scale [out])} for the int8 matrices."""
        for n, a in weights.items():
            self.set_weight(n, a)
        for n, (q, sc) in (int8 or {}).items():
            self.set_weight_i8(n, q, sc)

    def set_weight_i8(self, name: str, q: np.ndarray, scale: np.ndarray):
        q = np.ascontiguousarray(q, dtype=np.int8)
        sc = np.ascontiguousarray(scale, dtype=np.float16)
        self._check(self.lib.rwkv7_set_weight_i8(self.h, name.encode(), q.ctypes.data, q.nbytes,
                                                  sc.ctypes.data, sc.nbytes))

    def load_weights(self, path: str):
        self._check(self.lib.rwkv7_load_weights(self.h, os.fsencode(path)))

    # ------------------------------------------------------------ slots
    def slot_reset(self, slot: int):
        self._check(self.lib.rwkv7_slot_reset(self.h, slot))

    def slot_swap(self, a: int, b: int):
        self._check(self.lib.rwkv7_slot_swap(self.h, a, b))

    def slot_copy(self, src: int, dst: int):
        self._check(self.lib.rwkv7_slot_copy(self.h, src, dst))

    def set_sampling(self, slot: int, temperature=1.0, top_p=0.3, top_k=0, presence=0.0,
                     frequency=1.0, penalty_decay=0.996, seed=0, greedy=False):
        sp = Sampling(temperature, top_p, top_k, presence, frequency, penalty_decay, seed, int(bool(greedy)))
        self._check(self.lib.rwkv7_slot_set_sampling(self.h, slot, C.byref(sp)))

    def state_bytes(self) -> int:
        return int(self.lib.rwkv7_slot_state_bytes(self.h))

    def get_state(self, slot: int):
        """(wkv [L,H,64,64], shift_att [L,d], shift_ffn [L,d]) as fp32 numpy."""
        buf = np.zeros(self.state_bytes() // 4, np.float32)
        self._check(self.lib.rwkv7_slot_get_state(self.h, slot, buf.ctypes.data, buf.nbytes))
        dm = self.dims
        nw = dm.n_layer * dm.n_head * 64 * 64
        ns = dm.n_layer * dm.d_model
        return (buf[:nw].reshape(dm.n_layer, dm.n_head, 64, 64), buf[nw:nw + ns].reshape(dm.n_layer, dm.d_model),
                buf[nw + ns:].reshape(dm.n_layer, dm.d_model))

    def set_state(self, slot: int, wkv, shift_att, shift_ffn):
        flat = np.concatenate([np.ravel(wkv), np.ravel(shift_att), np.ravel(shift_ffn)]).astype(np.float32)
        self._check(self.lib.rwkv7_slot_set_state(self.h, slot, flat.ctypes.data, flat.nbytes))

    # ------------------------------------------------------------ compute
    def prefill_seq(self, slot: int, tokens, logits_out=None):
        import torch
        self._check(self.lib.rwkv7_prefill_seq(self.h, slot, _ptr(tokens, torch.int32, "tokens"),
                                               tokens.numel(), _ptr(logits_out, torch.float32, "logits_out")))

    def decode_step(self, slots, tokens, logits_out=None, next_out=None):
        import torch
        B = slots.numel()
        if tokens.numel() != B:
            raise ValueError("slots and tokens differ in length")
        self._check(self.lib.rwkv7_decode_step(self.h, _ptr(slots, torch.int32, "slots"),
                                               _ptr(tokens, torch.int32, "tokens"), B,
                                               _ptr(logits_out, torch.float32, "logits_out"),
                                               _ptr(next_out, torch.int32, "next_out")))

    def decode_step_host(self, slots: np.ndarray, tokens: np.ndarray, logits_out=None, next_out=None):
        """Host-buffer step (numpy arrays or pinned CPU tensors); synchronous."""
        def hp(a, dt):
            if a is None:
                return None
            if isinstance(a, np.ndarray):
                assert a.dtype == dt and a.flags.c_contiguous
                return C.c_void_p(a.ctypes.data)
            assert not a.is_cuda and a.is_contiguous()
            return C.c_void_p(a.data_ptr())
        B = len(slots)
        self._check(self.lib.rwkv7_decode_step_host(self.h, hp(slots, np.int32), hp(tokens, np.int32), B,
                                                    hp(logits_out, np.float32), hp(next_out, np.int32)))

    def sample_batch(self, slots, logits, next_out):
        import torch
        self._check(self.lib.rwkv7_sample_batch(self.h, _ptr(slots, torch.int32, "slots"),
                                                _ptr(logits, torch.float32, "logits"), slots.numel(),
                                                _ptr(next_out, torch.int32, "next_out")))

    def ffn_union_stats(self):
        """(nonzero value-row blocks, blocks considered) since the last call; see
        rwkv7_ffn_union_stats."""
        nz, tot = C.c_uint64(), C.c_uint64()
        self._check(self.lib.rwkv7_ffn_union_stats(self.h, C.byref(nz), C.byref(tot)))
        return int(nz.value), int(tot.value)

    def synchronize(self):
        self._check(self.lib.rwkv7_synchronize(self.h))

    def debug_latch_error(self, flags: int):
        """Test hook: OR flags into the device error word (rwkv7_debug_latch_error)."""
        self._check(self.lib.rwkv7_debug_latch_error(self.h, int(flags)))

    def set_mode(self, mode: int):
        self._check(self.lib.rwkv7_set_mode(self.h, mode))

    def step_kernel_count(self, B: int, with_sampling: bool) -> int:
        return int(self.lib.rwkv7_step_kernel_count(self.h, B, int(bool(with_sampling))))

    def profile_step(self, slots, tokens, with_sampling: bool = False):
        """One directly-launched, event-bracketed step: {class: (ms, launches)}."""
        import torch
        n = len(PROF_CLASSES)
        ms = np.zeros(n, np.float32)
        cnt = np.zeros(n, np.int32)
        self._check(self.lib.rwkv7_profile_step(self.h, _ptr(slots, torch.int32, "slots"),
                                                _ptr(tokens, torch.int32, "tokens"), slots.numel(),
                                                int(bool(with_sampling)), ms.ctypes.data, cnt.ctypes.data, n))
        return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(PROF_CLASSES)}

    def step_timeline(self, slots, tokens, with_sampling: bool = False, max_launches: int = 4096):
        """rwkv7_step_timeline: one graph-replayed step with every kernel stamping
        the GPU timer.  Returns (times [n, 4] int64 ns -- earliest start, earliest
        and latest dependency release, latest end of each launch -- and the
        class name of each launch)."""
        import torch
        t = np.zeros((max_launches, 4), np.uint64)
        cls = np.zeros(max_launches, np.int32)
        n = C.c_int32()
        self._check(self.lib.rwkv7_step_timeline(self.h, _ptr(slots, torch.int32, "slots"),
                                                 _ptr(tokens, torch.int32, "tokens"), slots.numel(),
                                                 int(bool(with_sampling)), t.ctypes.data, cls.ctypes.data,
                                                 max_launches, C.byref(n)))
        k = int(n.value)
        return t[:k].astype(np.int64), [PROF_CLASSES[c] for c in cls[:k]]

    def io_buffers(self):
        """(slots, tokens, logits, next) device pointers owned by the context."""
        p = [C.c_void_p() for _ in range(4)]
        self._check(self.lib.rwkv7_get_io_buffers(self.h, *[C.byref(x) for x in p]))
        return tuple(x.value for x in p)


__all__ = ["Rwkv7", "RWKV7Error", "Config", "Sampling", "load_library", "build", "LIB_PATH",
           "SIGNATURES", "MAX_STEP_BATCH", "PROF_CLASSES", "set_device_allocator"]
