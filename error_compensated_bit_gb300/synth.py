"""Seeded synthetic workloads for the compression-stage step.

This module only draws inputs (gradients, parameters, frozen variances, masks) with
the shapes and distributions of the workloads below; it holds none of the method's
arithmetic. The same draws feed the CUDA path and the CPU oracle. Every draw comes
from a torch generator seeded by (seed, tensor kind, step, worker), so a tensor can be
regenerated on its own, on the host or on a device; values drawn on the host and on a
device with the same seed are NOT equal, so a test that compares the two sides draws
once and copies.

Workloads (element counts are padded to a multiple of W*256; pad elements carry
g = 0, x = 0, m = 0, v = 1 and mask = 1):

  tiny   n = 2^20, W = 4, chunk = n/W, float32 grads ~ N(0, 1e-3); x ~ N(0, 0.02);
         v ~ U(1e-8, 1e-4); m and errors zero; 10 compressed steps; seed 1.
  bertB  n = 110,000,000 -> 110,000,128, W = 8, chunk = n/W, float32 grads ~ N(0, 1e-3)
         with a fixed 2% of positions exactly zero (the momentum mask is zero there);
         v0 ~ lognormal(-12, 2); 5 warm-up Adam steps then 20 compressed; seed 2.
  bertL  BERT-Large's 390 parameter tensors fused into one buffer (333,495,296 ->
         333,496,320), W = 8, chunk = n/W, float16 grads ~ N(0, 1e-3);
         v ~ U(1e-8, 1e-4); 20 compressed steps; seed 3.
  sweep  n = 2^28, W in {2, 4, 8, 16}, float32 grads 1e-3 * Student-t(3); seed 4.
  loco   GPT-like 1.3B buffer (24 layers, d = 2048, 4x MLP, vocab 50257, 2048
         positions) = 1,315,723,264, W = 4, bfloat16 grads ~ N(0, 1e-3); seed 5.
"""
from dataclasses import dataclass, field

import torch

B1, B2, EPS, LR = 0.9, 0.999, 1e-8, 1e-4

_KIND = {"grad": 1, "x": 2, "v": 3, "zero_pos": 4}


def bert_large_sizes():
    """Element counts of BERT-Large's 390 parameter tensors, in model order.

    Word embedding 30522x1024; 24 encoder layers each with Q, K, V, O (1024x1024), the
    MLP (1024x4096 and 4096x1024) and ten 1024-vectors (4 attention biases, 2 LayerNorms
    x 2, the MLP output bias ... counted as in the workload recipe); five trailing
    1024-vectors. 145 matrices + 245 vectors.
    """
    sizes = [30522 * 1024]
    for _ in range(24):
        sizes += [1024 * 1024] * 4 + [1024 * 4096, 4096 * 1024] + [1024] * 10
    sizes += [1024] * 5
    return sizes


def gpt_like_size(layers=24, d=2048, vocab=50257, positions=2048):
    """Parameter count of the GPT-like buffer: 12d^2 + 13d per layer, embeddings, final LN."""
    return layers * (12 * d * d + 13 * d) + vocab * d + positions * d + 2 * d


def pad_to(n, multiple):
    return (n + multiple - 1) // multiple * multiple


@dataclass
class Workload:
    name: str
    n_real: int
    W: int
    grad_dtype: torch.dtype
    seed: int
    grad_dist: str = "normal"          # "normal" or "student_t3"
    v_dist: str = "uniform"            # "uniform" or "lognormal"
    zero_frac: float = 0.0             # fixed fraction of exactly-zero gradient positions
    warmup_steps: int = 0
    steps: int = 10
    chunk: int = 0                     # 0 -> n / W
    b1: float = B1
    b2: float = B2
    eps: float = EPS
    lr: float = LR
    extra: dict = field(default_factory=dict)

    @property
    def n(self):
        return pad_to(self.n_real, self.W * 256)

    @property
    def C(self):
        return self.chunk or self.n // self.W

    @property
    def grad_bytes(self):
        return torch.empty((), dtype=self.grad_dtype).element_size()


def workload(name, W=None, n=None, chunk=None, seed=None):
    """The named workload, optionally resized (tests use smaller n with the same recipe)."""
    if name == "tiny":
        wl = Workload("tiny", 1 << 20, 4, torch.float32, 1, steps=10)
    elif name == "bertB":
        wl = Workload("bertB", 110_000_000, 8, torch.float32, 2, v_dist="lognormal",
                      zero_frac=0.02, warmup_steps=5, steps=20)
    elif name == "bertL":
        wl = Workload("bertL", sum(bert_large_sizes()), 8, torch.float16, 3, steps=20)
    elif name == "sweep":
        wl = Workload("sweep", 1 << 28, W or 8, torch.float32, 4, grad_dist="student_t3",
                      warmup_steps=5, steps=20)
    elif name == "loco":
        wl = Workload("loco", gpt_like_size(), 4, torch.bfloat16, 5, steps=20)
    else:
        raise KeyError(name)
    if W is not None:
        wl.W = W
    if n is not None:
        wl.n_real = n
    if chunk is not None:
        wl.chunk = chunk
    if seed is not None:
        wl.seed = seed
    return wl


def _gen(device, seed, kind, step=0, worker=0):
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + _KIND[kind] * 10_007 + step * 101 + worker) % (1 << 62))
    return g


def zero_positions(wl, device="cpu"):
    """Boolean [n] of the fixed exactly-zero gradient positions (False on pad elements)."""
    n, nr = wl.n, wl.n_real
    out = torch.zeros(n, dtype=torch.bool, device=device)
    if wl.zero_frac > 0:
        r = torch.rand(nr, generator=_gen(device, wl.seed, "zero_pos"), device=device)
        out[:nr] = r < wl.zero_frac
    return out


def grads(wl, step, device="cpu", out=None):
    """Gradients of all W workers for one step: [W, n] in the workload's grad dtype."""
    n, nr = wl.n, wl.n_real
    if out is None:
        out = torch.empty(wl.W, n, dtype=wl.grad_dtype, device=device)
    zpos = zero_positions(wl, device) if wl.zero_frac > 0 else None
    for w in range(wl.W):
        gen = _gen(device, wl.seed, "grad", step, w)
        row = torch.randn(nr, generator=gen, device=device, dtype=torch.float32)
        if wl.grad_dist == "student_t3":
            chi = torch.randn(3, nr, generator=gen, device=device, dtype=torch.float32)
            chi = chi.square_().sum(0).div_(3.0).sqrt_()
            row.div_(chi)
            del chi
        row.mul_(1e-3)
        if zpos is not None:
            row.masked_fill_(zpos[:nr], 0.0)
        out[w, :nr].copy_(row)
        out[w, nr:].zero_()
        del row
    return out


def params(wl, device="cpu"):
    """Initial x ~ N(0, 0.02) (pad 0)."""
    x = torch.zeros(wl.n, dtype=torch.float32, device=device)
    x[:wl.n_real] = torch.randn(wl.n_real, generator=_gen(device, wl.seed, "x"),
                                device=device).mul_(0.02)
    return x


def variance(wl, device="cpu"):
    """Frozen (or initial) second moment: U(1e-8, 1e-4) or lognormal(-12, 2) (pad 1)."""
    v = torch.ones(wl.n, dtype=torch.float32, device=device)
    gen = _gen(device, wl.seed, "v")
    if wl.v_dist == "lognormal":
        v[:wl.n_real] = torch.randn(wl.n_real, generator=gen, device=device).mul_(2.0).add_(-12.0).exp_()
    else:
        v[:wl.n_real] = torch.rand(wl.n_real, generator=gen, device=device).mul_(1e-4 - 1e-8).add_(1e-8)
    return v


def mask(wl, device="cpu"):
    """Momentum mask as float 0/1 [n]: zero at the fixed zero-gradient positions, else one."""
    return (~zero_positions(wl, device)).to(torch.float32)


def to_numpy_grads(g):
    """Host copy of a gradient tensor in the oracle's storage formats.

    float32 -> float32, float16 -> float16, bfloat16 -> raw uint16 bits.
    """
    g = g.detach().cpu().contiguous()
    if g.dtype == torch.bfloat16:
        return g.view(torch.int16).numpy().view("uint16")
    return g.numpy()
