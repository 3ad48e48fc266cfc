"""The benchmark's roofline numerators against an independent count.

bench.step_bytes / step_bytes_i8 are closed forms of the bytes one decode step
must move (every streamed matrix once, the recurrent and token-shift states
read and written once per slot); here the same totals are summed tensor by
tensor from synth.tensor_specs, the list the weight generator and both
implementations are built from, so a dropped matrix or a wrong factor in either
closed form fails."""
import numpy as np
import pytest

import bench
import synth


def _counted(dims, B, int8):
    i8 = set(synth.i8_matrix_names(dims))
    total = 0
    for name, shape, _ in synth.tensor_specs(dims):
        if len(shape) != 2 or name == "emb":
            continue  # vectors are not streamed per step; the embedding is gathered
        rows, cols = shape
        if int8:
            assert name in i8
            total += rows * cols + 2 * rows  # int8 values + one fp16 scale per row
        else:
            total += 2 * rows * cols
    state = dims.n_layer * (dims.n_head * 64 * 64 + 2 * dims.d_model) * 4  # wkv + two shift rows, fp32
    return total + 2 * B * state  # read and written


@pytest.mark.parametrize("shape,B", [("tiny", 1), ("0.1b", 32), ("2.9b", 64), ("7.2b", 256)])
def test_step_bytes_match_tensor_count(shape, B):
    dims = synth.Dims(shape)
    assert bench.step_bytes(dims, B) == _counted(dims, B, int8=False)
    assert bench.step_bytes_i8(dims, B) == _counted(dims, B, int8=True)


def test_headline_bytes_per_step():
    # weights + states per step of the 2.9B (B = 64) and 7.2B (B = 256) decode workloads
    assert round(bench.step_bytes(synth.Dims("2.9b"), 64) / 1e9, 3) == 8.326
    assert round(bench.step_bytes(synth.Dims("7.2b"), 256) / 1e9, 3) == 31.575


def test_traffic_hash_follows_code_not_comments(tmp_path):
    """The ncu traffic record stays valid across comment edits of the kernel
    source and is dropped on any code edit."""
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int *p) {\n    p[0] = 1;  // store\n}\n")
    h0 = bench._sha([str(src)])
    src.write_text("// header, reworded\n/* a block\n   comment */\n__global__ void k(int *p) {\n\n    p[0] = 1;\n}\n")
    assert bench._sha([str(src)]) == h0
    src.write_text("// header\n__global__ void k(int *p) {\n    p[0] = 2;  // store\n}\n")
    assert bench._sha([str(src)]) != h0

