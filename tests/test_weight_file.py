"""The RWKV7W01 weight file written by synth (text header, 256-byte aligned fp16
tensors after a 4096-byte header block) read back on the host: every tensor's
name, shape and bytes survive, offsets are aligned, and a file that is not an
RWKV7W01 file is refused."""
import numpy as np
import pytest

import synth


def test_roundtrip_tiny(tmp_path):
    w = synth.make_weights("tiny")
    p = tmp_path / "tiny.rwkv7w"
    synth.write_weight_file(str(p), w)
    back = synth.read_weight_file(str(p))
    assert list(back.keys()) == list(w.keys())
    for k in w:
        assert back[k].dtype == np.float16 and back[k].shape == w[k].shape
        assert np.array_equal(back[k].view(np.uint16), w[k].view(np.uint16))
    raw = p.read_bytes()
    assert raw.startswith(b"RWKV7W01\n")
    header = raw[:4096].split(b"END\n")[0].decode().splitlines()[2:]
    for line in header:
        name, dt, shape, off, nb = line.split()
        assert dt == "f16" and int(off) % 256 == 0 and int(nb) == int(np.prod([int(x) for x in shape.split("x")])) * 2


def test_not_a_weight_file(tmp_path):
    p = tmp_path / "junk"
    p.write_bytes(b"\0" * 5000)
    with pytest.raises(ValueError):
        synth.read_weight_file(str(p))
