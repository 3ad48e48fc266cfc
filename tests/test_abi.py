"""CPU-side checks of the C ABI: the library builds, loads and exports exactly
the entry points include/rwkv7.h declares, and the binding declares a
signature for each.  No compute calls (no GPU here)."""
import ctypes as C
import os
import re

import pytest

import recurrent_decode_gb300 as rd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"RWKV7_API[^;(]*?\b(rwkv7_\w+)\s*\(", txt)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    rd.build()
    return rd.load_library()


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("rwkv7_load_weights", "rwkv7_prefill_seq", "rwkv7_decode_step", "rwkv7_sample_batch",
                 "rwkv7_slot_reset", "rwkv7_slot_swap"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol():
    assert sorted(rd.SIGNATURES) == _declared()


def test_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", rd.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if " T " in ln and ln.split()[-1].startswith("rwkv7_")})
    assert exported == _declared()


def test_null_arguments_rejected_without_a_device(lib):
    out = C.c_void_p(123)
    assert lib.rwkv7_create(None, None, C.byref(out)) == rd.EINVAL
    assert lib.rwkv7_decode_step(None, None, None, 1, None, None) == rd.EINVAL
    assert lib.rwkv7_sample_batch(None, None, None, 1, None) == rd.EINVAL
    assert lib.rwkv7_last_error(None) == b"null context"
    assert lib.rwkv7_slot_state_bytes(None) == 0
    bad = rd.Config(2, 100, 64, 512, 1024, 16, 16, 16, 32, 4)  # d not a multiple of 64
    assert lib.rwkv7_create(C.byref(bad), None, C.byref(out)) == rd.EINVAL
