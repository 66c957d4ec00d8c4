"""Python-side plumbing around libmoe: device copies of stored inputs and a
layer object with the interface the pages use.

"Mixture of Experts: Scaling Parameters Without Scaling Compute", section
"The MoE layer": a layer is built from (d, d_ff, n_experts, k) and its
forward maps a token batch x of shape (tokens, d) to (output, auxiliary loss).
Here the weights are caller-provided device tensors and the whole forward
pass is one ``moe_forward`` call into libmoe; torch only allocates the
output, the scalars and the workspace.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .inputs import Inputs


def to_torch(a: np.ndarray, device="cuda") -> torch.Tensor:
    """A stored input array as a torch tensor (uint16 bit patterns -> bf16)."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def device_inputs(inp: Inputs, device="cuda") -> dict:
    """Every stored tensor of ``inp`` copied to ``device`` (weights included)."""
    out = {}
    for name in ("x", "W_r", "logit_bias", "W1", "b1", "W2", "b2"):
        a = getattr(inp, name)
        out[name] = None if a is None else to_torch(a, device)
    return out


class MoELayer:
    """Sparsely-gated MoE FFN layer whose forward pass runs in libmoe.

    W_r: (E - n_shared, d) fp32; W1: (E, d_ff, d); b1: (E, d_ff); W2: (E, d, d_ff);
    b2: (E, d), all on one CUDA device, W1..b2 of one dtype (fp32 or bf16).
    n_shared: experts 0 .. n_shared - 1 are always active with weight 1 (the
    router scores the other E - n_shared).
    routing: "token" (top-k experts per token) or "expert" (each expert takes
    its top-C tokens; k then sets C = ceil(T k / E) unless a capacity is given).
    overflow: "drop" (the capacity cap drops overflow) or "reroute" (a dropped
    slot is offered to the token's next-best expert).
    """

    def __init__(self, W_r, W1, b1, W2, b2, k: int, capacity: int | None = None,
                 renormalize: bool = True, logit_bias=None, routing: str = "token",
                 overflow: str = "drop", n_shared: int = 0):
        self.E, self.d_ff, self.d = W1.shape
        self.n_shared = n_shared
        self.k = k
        self.routing = routing
        self.overflow = overflow
        self.dtype = "bf16" if W1.dtype == torch.bfloat16 else "f32"
        self.capacity, self.renormalize = capacity, renormalize
        self.W_r, self.W1, self.b1, self.W2, self.b2 = W_r, W1, b1, W2, b2
        self.logit_bias = logit_bias
        self._ws = {}

    def config(self, T: int) -> B.MoeConfig:
        return B.config(T, self.d, self.d_ff, self.E, self.k, self.dtype, self.capacity,
                        self.renormalize, n_shared=self.n_shared, routing=self.routing,
                        overflow=self.overflow)

    def workspace(self, T: int) -> torch.Tensor:
        if T not in self._ws:
            self._ws[T] = B.workspace(self.config(T), device=self.W1.device)
        return self._ws[T]

    def forward(self, x, y=None, aux=None, expert_counts=None, logits_out=None, z_loss=None,
                logit_noise=None, stream=None):
        """(y, aux) for the token batch x (T, d); optional outputs (expert_counts,
        logits_out, z_loss: the router z-loss, one fp32) are filled in place;
        logit_noise (T, E fp32) is added to the router logits (noisy gating)."""
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        if aux is None:
            aux = torch.empty(1, dtype=torch.float32, device=x.device)
        B.forward(self.config(T), x, self.W_r, self.W1, self.b1, self.W2, self.b2, y,
                  self.workspace(T), logit_bias=self.logit_bias, aux_out=aux,
                  expert_counts=expert_counts, logits_out=logits_out, z_loss_out=z_loss,
                  logit_noise=logit_noise, stream=stream)
        return y, aux

    __call__ = forward

    def backward(self, x, dy, aux_grad: float = 0.0, z_grad: float = 0.0, stream=None) -> dict:
        """Gradients of <dy, y> + aux_grad * aux + z_grad * z_loss for the batch
        x (moe_backward; every layer this object can run):
        {"dx", "dW_r", "dW1", "db1", "dW2", "db2"}, dx in the layer dtype, the
        weight gradients fp32.  The routing decisions are held fixed."""
        T = x.shape[0]
        cfg = self.config(T)
        key = ("backward", T)
        if key not in self._ws:
            self._ws[key] = B.backward_workspace(cfg, device=self.W1.device)
        f32 = dict(dtype=torch.float32, device=self.W1.device)
        g = dict(dx=torch.empty_like(x), dW_r=torch.empty(tuple(self.W_r.shape), **f32),
                 dW1=torch.empty((self.E, self.d_ff, self.d), **f32),
                 db1=torch.empty((self.E, self.d_ff), **f32),
                 dW2=torch.empty((self.E, self.d, self.d_ff), **f32),
                 db2=torch.empty((self.E, self.d), **f32))
        B.backward(cfg, x, self.W_r, self.W1, self.b1, self.W2, self.b2, dy, g["dx"], g["dW_r"],
                   g["dW1"], g["db1"], g["dW2"], g["db2"], self._ws[key],
                   logit_bias=self.logit_bias, aux_grad=aux_grad, z_grad=z_grad, stream=stream)
        return g

    def host_pipeline(self, T: int, depth: int = 2, stream=None) -> B.Pipeline:
        """An executor for batches of T tokens in host memory (moe_pipeline_*):
        ``submit(x_host, y_host, aux_host)`` per batch, ``join()`` to make the
        stream wait for the outputs; the copies overlap the forward passes."""
        return B.Pipeline(self.config(T), self.W_r, self.W1, self.b1, self.W2, self.b2,
                          logit_bias=self.logit_bias, depth=depth, stream=stream,
                          device=self.W1.device)


def capture_graph(fn, stream=None, warmup: int = 2):
    """Record the libmoe calls made by ``fn(stream)`` into a CUDA graph.

    ``fn`` must enqueue its work on the stream it is given and use fixed
    buffers; ``graph.replay()`` then re-runs the recorded kernels with one
    launch.  Warm-up calls run first, outside the capture, so that one-time
    host work (kernel attributes, driver entry points) is done before it."""
    side = torch.cuda.Stream() if stream is None else stream
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            fn(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        fn(torch.cuda.current_stream())
    return g
