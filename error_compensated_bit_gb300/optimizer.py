"""A user-facing optimizer object over the C ABI: state tensors in torch device memory,
phases switched by step count, checkpoints that reset the compression errors.

Phases follow the DeepSpeed 1-bit Adam training guide, §3.1 and §4: full-precision Adam
while the step count is below ``freeze_step``, then the compression stage with the
variance frozen. Checkpoints follow §7: the error buffers are not saved and are reset
when a state is loaded; the momentum mask (§3.5) is not part of the state and must be
set again on every run.
"""
import torch

from . import ob


def _bytes_view(ws, ptr, count, dtype):
    off = ptr - ws.data_ptr()
    size = torch.empty((), dtype=dtype).element_size()
    return ws[off:off + count * size].view(dtype)


class OneBitAdam:
    """1-bit Adam over one flat float32 parameter buffer and W simulated workers.

    ``x`` (optional) initialises the parameters; gradients are passed per step as a
    [W, n] tensor of float32, float16 or bfloat16 on the same device.
    """

    def __init__(self, n, W, chunk=None, lr=1e-4, betas=(0.9, 0.999), eps=1e-8,
                 weight_decay=0.0, bias_correction=False, freeze_step=100000, x=None,
                 device="cuda"):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.device(self.device):
            self.ctx = ob.Context(n, W, chunk or n // W, betas[0], betas[1], eps, lr)
            self.ctx.set_options(weight_decay, bias_correction)
            self.n, self.W, self.chunk = n, W, chunk or n // W
            self.freeze_step = freeze_step
            f32 = dict(dtype=torch.float32, device=self.device)
            self.x = torch.zeros(n, **f32) if x is None else x.to(**f32).contiguous().clone()
            self.m = torch.zeros(n, **f32)
            self.v = torch.zeros(n, **f32)
            self.worker_err = torch.zeros(W, n, **f32)
            self.server_err = torch.zeros(n, **f32)
            self.ws = torch.empty(self.ctx.workspace_bytes(), dtype=torch.uint8, device=self.device)
            self.ctx.workspace_init(self.ws)
            self._mask = None

    @property
    def step_count(self):
        return self.ctx.get_step()

    @property
    def compressed(self):
        return self.step_count >= self.freeze_step

    def set_lr(self, lr):
        self.ctx.set_lr(lr)

    def set_mask(self, mask01):
        """0/1 float mask [n] (None clears); keep the tensor alive while it is in use."""
        self._mask = None if mask01 is None else mask01.to(torch.float32).contiguous()
        self.ctx.set_mask(self._mask, self.ws)

    def step(self, grads):
        """One optimizer step with the [W, n] gradients of the W workers."""
        with torch.cuda.device(self.device):
            if self.compressed:
                self.ctx.compressed_step(grads, self.x, self.m, self.v, self.worker_err,
                                         self.server_err, self.ws)
            else:
                self.ctx.warmup_step(grads, self.x, self.m, self.v, self.ws)

    def reset_errors(self):
        with torch.cuda.device(self.device):
            self.ctx.reset_errors(self.worker_err, self.server_err, self.ws)

    def errors(self):
        """The true worker and server residuals, (e_w [W, n], e_s [n])."""
        ew = torch.empty_like(self.worker_err)
        es = torch.empty_like(self.server_err)
        with torch.cuda.device(self.device):
            self.ctx.export_state(self.worker_err, self.server_err, self.ws, ew, es)
        return ew, es

    def messages(self):
        """This step's compressed messages as tensors viewing the workspace:
        worker signs [W, n/32] int32, worker scales [W, nchunks], server signs [n/32],
        server scales [nchunks]."""
        wb, wsc, sb, ssc = self.ctx.debug_views(self.ws)
        nch = self.n // self.chunk
        return (_bytes_view(self.ws, wb, self.W * self.n // 32, torch.int32).view(self.W, -1),
                _bytes_view(self.ws, wsc, self.W * nch, torch.float32).view(self.W, -1),
                _bytes_view(self.ws, sb, self.n // 32, torch.int32),
                _bytes_view(self.ws, ssc, nch, torch.float32))

    def state_dict(self):
        """Parameters, momentum, variance and step; the errors are not saved."""
        return {"x": self.x.clone(), "m": self.m.clone(), "v": self.v.clone(),
                "step": self.step_count, "freeze_step": self.freeze_step}

    def load_state_dict(self, sd):
        """Restore a state; compression errors restart from zero."""
        self.x.copy_(sd["x"])
        self.m.copy_(sd["m"])
        self.v.copy_(sd["v"])
        self.ctx.set_step(int(sd["step"]))
        self.freeze_step = int(sd.get("freeze_step", self.freeze_step))
        self.reset_errors()


class LocoAdam:
    """Adam on LoCo-compressed gradients over one flat float32 buffer and W simulated
    workers ("LoCo: Low-Bit Communication Adaptor for Large-scale Model Training",
    "Method"): every step each worker compensates its gradient with ``ratio`` times the
    moving average of its past compression errors (weight ``beta``), quantizes it per
    chunk to ``bits``-bit codes with an absmax scale, and the mean of the dequantized
    gradients drives a plain Adam step.

    The pages say nothing about checkpoints for LoCo; the moving average is part of the
    compressor's state, so it is saved and restored with the parameters here.
    """

    def __init__(self, n, W, chunk=None, lr=1e-4, betas=(0.9, 0.999), eps=1e-8,
                 weight_decay=0.0, bits=4, beta=0.9, ratio=1.0, x=None, device="cuda",
                 keep_codes=False):
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.device(self.device):
            self.ctx = ob.Context(n, W, chunk or n // W, betas[0], betas[1], eps, lr)
            self.ctx.set_options(weight_decay, False)
            self.ctx.set_loco_ratio(ratio)
            self.ctx.set_loco_codes(keep_codes)
            self.n, self.W, self.chunk = n, W, chunk or n // W
            self.bits, self.beta, self.ratio = bits, beta, ratio
            f32 = dict(dtype=torch.float32, device=self.device)
            self.x = torch.zeros(n, **f32) if x is None else x.to(**f32).contiguous().clone()
            self.m = torch.zeros(n, **f32)
            self.v = torch.zeros(n, **f32)
            self.err = torch.zeros(W, n, **f32)
            self.ws = torch.zeros(self.ctx.loco_workspace_bytes(bits), dtype=torch.uint8,
                                  device=self.device)

    @property
    def step_count(self):
        return self.ctx.get_step()

    def set_lr(self, lr):
        self.ctx.set_lr(lr)

    def step(self, grads):
        """One optimizer step with the [W, n] gradients of the W workers."""
        with torch.cuda.device(self.device):
            self.ctx.loco_step(grads, self.x, self.m, self.v, self.err, self.ws, self.beta, self.bits)

    def messages(self):
        """This step's low-bit messages viewing the workspace: codes [W, n*bits/8] uint8
        and scales [W, nchunks] float32. The codes are stored for chunks of up to 4096
        elements, or when the object was made with ``keep_codes=True`` (longer chunks
        otherwise keep them in registers)."""
        code_bytes = self.W * self.n * self.bits // 8
        off = (code_bytes + 255) // 256 * 256
        nch = self.n // self.chunk
        return (self.ws[:code_bytes].view(self.W, -1),
                self.ws[off:off + self.W * nch * 4].view(torch.float32).view(self.W, -1))

    def state_dict(self):
        return {"x": self.x.clone(), "m": self.m.clone(), "v": self.v.clone(),
                "err": self.err.clone(), "step": self.step_count}

    def load_state_dict(self, sd):
        self.x.copy_(sd["x"])
        self.m.copy_(sd["m"])
        self.v.copy_(sd["v"])
        self.err.copy_(sd["err"])
        self.ctx.set_step(int(sd["step"]))
