"""The user-facing OneBitAdam object on the GPU: phases, checkpoints and the mask.

Follows the DeepSpeed 1-bit Adam training guide: full-precision Adam while the step
count is below freeze_step, the compression stage after it (§3.1, §4); loading a
checkpoint resets the worker and server errors while the rest of the state is restored
(§7); the momentum mask is not part of the saved state and is supplied again (§3.5).
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import assert_close

pytestmark = pytest.mark.gpu


def _grads(rng, W, n):
    return torch.from_numpy((rng.standard_normal((W, n)) * 1e-3).astype(np.float32)).cuda()


def test_phases_follow_freeze_step(ora):
    from error_compensated_bit_gb300.optimizer import OneBitAdam
    rng = np.random.default_rng(70)
    W, n, freeze = 4, 4 * 256 * 100, 3
    x0 = rng.standard_normal(n).astype(np.float32) * 0.02
    opt = OneBitAdam(n, W, lr=1e-3, freeze_step=freeze, x=torch.from_numpy(x0).cuda())
    st = O.OracleState(n, W, n // W, x=x0, m=np.zeros(n), v=np.zeros(n), lr=1e-3)
    for t in range(6):
        g = _grads(rng, W, n)
        assert opt.compressed == (t >= freeze)
        opt.step(g)
        if t < freeze:
            ora.warmup_step(st, g.cpu().numpy())
        else:
            ora.compressed_step(st, g.cpu().numpy())
        torch.cuda.synchronize()
        assert_close("step %d x" % t, opt.x.cpu().numpy(), st.x)
        assert_close("step %d m" % t, opt.m.cpu().numpy(), st.m)
    assert opt.step_count == 6
    ew, es = opt.errors()
    assert_close("worker errors", ew.cpu().numpy(), st.ew, atol=1e-7 + 1e-5 * np.abs(st.ew).max())


def test_checkpoint_resets_errors_and_drops_mask(ora):
    from error_compensated_bit_gb300.optimizer import OneBitAdam
    rng = np.random.default_rng(71)
    W, n = 4, 4 * 256 * 80
    mask = torch.from_numpy((rng.random(n) > 0.1).astype(np.float32)).cuda()
    a = OneBitAdam(n, W, lr=1e-3, freeze_step=1)
    a.set_mask(mask)
    for t in range(4):
        a.step(_grads(rng, W, n))
    ew, es = a.errors()
    assert ew.abs().sum() > 0 and es.abs().sum() > 0
    sd = a.state_dict()
    assert set(sd) == {"x", "m", "v", "step", "freeze_step"}, "errors and mask are not saved"
    b = OneBitAdam(n, W, lr=1e-3, freeze_step=100)
    b.load_state_dict(sd)
    assert b.step_count == 4 and b.freeze_step == 1 and b.compressed
    ew, es = b.errors()
    assert ew.abs().sum() == 0 and es.abs().sum() == 0, "errors restart from zero on load"
    assert torch.equal(b.x, a.x) and torch.equal(b.m, a.m) and torch.equal(b.v, a.v)
    # the restored optimizer continues like one whose errors were reset: compare with the
    # oracle started from the restored state and zero errors, mask supplied again
    st = O.OracleState(n, W, n // W, x=sd["x"].cpu().numpy(), m=sd["m"].cpu().numpy(),
                       v=sd["v"].cpu().numpy(), lr=1e-3, mask=mask.cpu().numpy())
    b.set_mask(mask)
    g = _grads(rng, W, n)
    b.step(g)
    ora.compressed_step(st, g.cpu().numpy())
    torch.cuda.synchronize()
    assert_close("x after load", b.x.cpu().numpy(), st.x)
    assert_close("m after load", b.m.cpu().numpy(), st.m)
    assert torch.all(b.m[mask == 0] == 0)


def test_loco_adam_matches_oracle_and_resumes(ora):
    """LocoAdam: 8-bit codes, ratio 1/2, several steps equal to the oracle's LoCo step;
    a saved state loaded into a fresh object continues identically."""
    from error_compensated_bit_gb300.optimizer import LocoAdam
    rng = np.random.default_rng(71)
    W, n = 3, 3 * 256 * 64
    C = 256 * 4
    x0 = rng.standard_normal(n).astype(np.float32) * 0.02
    opt = LocoAdam(n, W, chunk=C, lr=1e-3, bits=8, beta=0.8, ratio=0.5, x=torch.from_numpy(x0).cuda())
    st = O.OracleState(n, W, C, x=x0, m=np.zeros(n), v=np.zeros(n), lr=1e-3)
    err = np.zeros((W, n), np.float32)
    gs = [_grads(rng, W, n) for _ in range(5)]
    for t in range(3):
        opt.step(gs[t])
        out = ora.loco_step(st, gs[t].cpu().numpy(), err, beta=0.8, bits=8, ratio=0.5)
        torch.cuda.synchronize()
        codes, scales = opt.messages()
        assert np.array_equal(codes.cpu().numpy(), out["codes"])
        assert np.array_equal(scales.cpu().numpy(), out["scales"])
        assert np.array_equal(opt.err.cpu().numpy(), err)
        assert np.array_equal(opt.x.cpu().numpy(), st.x)
    sd = opt.state_dict()
    resumed = LocoAdam(n, W, chunk=C, lr=1e-3, bits=8, beta=0.8, ratio=0.5)
    resumed.load_state_dict(sd)
    assert resumed.step_count == 3
    for t in range(3, 5):
        opt.step(gs[t])
        resumed.step(gs[t])
    torch.cuda.synchronize()
    for name in ("x", "m", "v", "err"):
        assert torch.equal(getattr(opt, name), getattr(resumed, name)), name
