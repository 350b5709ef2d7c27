"""Failure detection on the GPU, without a fault: every wait in the library's kernels is
bounded, and a wait that runs out leaves status 1 in the workspace instead of hanging.

ob_selftest_wait enqueues exactly that situation (a barrier nothing completes, a 5 ms
limit). The test checks that the status is reported, that the step's normal path
reports 0, and that the context and workspace are usable again after
ob_workspace_init: the next steps match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import CudaPath, Tracker, random_state

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_recoverable(ora):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from error_compensated_bit_gb300 import build
    build.build()
    rng = np.random.default_rng(77)
    W, n, C = 4, 4 * 256 * 64, 256 * 32
    st = random_state(rng, n, W, C)
    gpu = CudaPath(st)
    tr = Tracker(n, W, C)
    g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)

    out = ora.compressed_step(st, g)
    gpu.compressed_step(g)
    tr.compare(0, gpu.snapshot(), out, st)
    assert gpu.ctx.read_status(gpu.ws) == 0

    launches = gpu.ctx.launch_count()
    gpu.ctx.selftest_wait(gpu.ws, 5_000_000)
    assert gpu.ctx.read_status(gpu.ws) == 1, "the bounded wait ran out and said so"
    assert gpu.ctx.launch_count() == launches + 1

    # recover: a fresh workspace and zero errors are the documented restart state
    gpu.ctx.workspace_init(gpu.ws)
    gpu.ew.zero_()
    gpu.es.zero_()
    st.ew[:] = 0.0
    st.es[:] = 0.0
    assert gpu.ctx.read_status(gpu.ws) == 0
    tr = Tracker(n, W, C)
    for t in range(2):
        g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
        out = ora.compressed_step(st, g)
        gpu.compressed_step(g)
        tr.compare(t, gpu.snapshot(), out, st)
    assert tr.flips == 0
    assert gpu.ctx.read_status(gpu.ws) == 0
