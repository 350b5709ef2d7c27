"""The benchmark's byte model (host logic, no GPU): algorithmic bytes per element of each
pass, written out term by term here, for the workloads the benchmark reports.

Compressed step, per element: W rows of gradients read (s_g each), the worker buffer read
and written (8), one sign bit per worker written and read back by the server (1/8 + 1/8),
the server buffer read and written (8), the server's sign bit written and read (1/8 +
1/8), m read by the worker and written by the update (8), x read and written (8), v read
(4); plus the mask bit when a mask is set.
"""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def compressed_terms(W, s_g, masked):
    worker = W * s_g + W * 8 + W / 8
    server = W / 8 + 8 + 1 / 8
    update = 1 / 8 + 8 + 8 + 4
    return worker + server + update + (1 / 8 if masked else 0)


@pytest.mark.parametrize("W,s_g,masked,expected", [
    (8, 2, False, 110.25),          # BERT-Large-sized, float16 gradients
    (8, 4, True, 126.375),          # BERT-Base-sized, float32, mask
    (2, 4, False, 52.75),           # sweep
    (4, 4, False, 77.25),
    (8, 4, False, 126.25),
    (16, 4, False, 224.25),
    (4, 2, False, 69.25),           # GPT-like buffer, bfloat16, 1-bit step
])
def test_compressed_bytes(bench, W, s_g, masked, expected):
    assert compressed_terms(W, s_g, masked) == expected
    assert bench.bytes_per_elem("compressed", W, s_g, masked) == expected


@pytest.mark.parametrize("W,s_g,expected", [(2, 4, 32), (4, 4, 40), (8, 4, 56), (16, 4, 88), (8, 2, 40)])
def test_warmup_bytes(bench, W, s_g, expected):
    # W gradient rows read; m and v read and written; x read and written
    assert W * s_g + 8 + 8 + 8 == expected
    assert bench.bytes_per_elem("warmup", W, s_g) == expected


def test_loco_bytes(bench):
    # per worker: gradient read, moving-average error read and written, 4-bit code written;
    # server: W codes read, x, m, v read and written
    W, s_g = 4, 2
    expected = W * (s_g + 8 + 0.5) + W * 0.5 + 24
    assert expected == 68
    assert bench.bytes_per_elem("loco", W, s_g) == expected


def test_worker_bytes_and_bertl_launch(bench):
    # worker pass alone: gradients, z read and written, sign bits, m read
    assert bench.worker_bytes_per_elem(8, 2) == 8 * (2 + 8 + 0.125) + 4 == 85.0
    n = 333_496_320
    assert n * bench.worker_bytes_per_elem(8, 2) == 28_347_187_200


def test_dominant_kernel_bytes(bench):
    # the roofline's kernel per phase: worker pass; the warm-up kernel (the whole warm-up
    # step); LoCo quantize (gradient and error read, error and 4-bit code written per row)
    n = 1_315_723_264
    assert bench.dominant_kernel_bytes("compressed", n, 4, 2) == n * (4 * (2 + 8.125) + 4)
    assert bench.dominant_kernel_bytes("warmup", n, 4, 2) == n * (4 * 2 + 24)
    assert bench.dominant_kernel_bytes("loco", n, 4, 2) == n * 4 * (2 + 4 + 4 + 0.5)
    assert bench.dominant_kernel_bytes("loco", n, 4, 2, 256) == n * 4 * (2 + 4 + 4 + 0.5)
    # long chunks: one pass quantizes every row and takes the Adam step (x, m, v)
    assert bench.dominant_kernel_bytes("loco", n, 4, 2, n // 4) == n * (4 * (2 + 4 + 4) + 24)


def test_extra_workloads_cover_every_recipe(bench):
    keys = {tuple(e[:3]) for e in bench.EXTRA_WORKLOADS}
    assert ("bertB", "compressed", None) in keys
    for W in (2, 4, 8, 16):
        assert ("sweep", "compressed", W) in keys and ("sweep", "warmup", W) in keys
    assert ("loco", "loco", None) in keys and ("loco", "compressed", None) in keys
    assert ("tiny", "compressed", None) in keys
