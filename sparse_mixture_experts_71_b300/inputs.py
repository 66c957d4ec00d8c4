"""Seeded synthetic inputs for the MoE-layer forward workloads.

This module only draws stored input values: the token batch ``x``, the router
weight ``W_r``, an optional per-expert router logit bias, and the expert bank
(``W1, b1, W2, b2``).  It holds none of the layer's arithmetic; both the CUDA
path and the CPU oracle consume exactly the arrays it returns.

Layouts follow ``nn.Linear`` (out, in), as in the PyTorch layer printed on
"Mixture of Experts: Scaling Parameters Without Scaling Compute", section
"The MoE layer":

* ``x``    (T, d)        token representations, row-major
* ``W_r``  (E - n_shared, d)  fp32  router weight (no bias; over the routed experts)
* ``W1``   (E, F, d)     first expert Linear, ``b1`` (E, F)
* ``W2``   (E, d, F)     second expert Linear, ``b2`` (E, d)

bf16 tensors are returned as ``uint16`` arrays holding the bf16 bit patterns
(round-to-nearest-even from an fp32 draw); ``bf16_bits_to_f32`` widens them
exactly.

Random streams: every tensor has its own stream id and is cut into fixed
chunks of ``_CHUNK`` elements; chunk ``c`` of stream ``s`` under seed ``seed``
is drawn from ``PCG64(SeedSequence([seed, s, c]))``.  Values therefore do not
depend on how many threads draw them.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

_CHUNK = 1 << 22

# stream ids, one per tensor
_S_X, _S_WR, _S_W1, _S_B1, _S_W2, _S_B2 = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class Workload:
    """One synthetic MoE-layer workload.

    ``capacity`` is the per-expert assignment cap (``None``: no cap);
    ``capacity_factor`` records the factor it was derived from.
    ``zipf_bias`` > 0 adds ``zipf_bias * ln(1 / (e + 1))`` to expert ``e``'s
    router logit, which skews the load towards low expert indices.
    ``init`` is ``"uniform"`` (every weight and bias ~ U(+-1/sqrt(fan_in)),
    router included) or ``"normal"`` (router N(0, 0.02); expert weights
    N(0, std = 1/sqrt(fan_in)); biases U(+-1/sqrt(fan_in))).
    """

    name: str
    T: int
    d: int
    F: int
    E: int
    k: int
    dtype: str = "bf16"  # "f32" or "bf16": storage type of x, W1, b1, W2, b2 and y
    renormalize: bool = True
    capacity: int | None = None
    capacity_factor: float | None = None
    zipf_bias: float = 0.0
    init: str = "normal"
    n_shared: int = 0  # experts 0 .. n_shared-1 always active (the router covers the rest)
    routing: str = "token"  # "token": top-k experts per token; "expert": top-C tokens per expert
    overflow: str = "drop"  # "drop" or "reroute" (capped slots offered to the next-best expert)
    note: str = field(default="", compare=False)

    def with_(self, **kw) -> "Workload":
        """A copy with some fields replaced (used for scaled-down test cases)."""
        return replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("tiny-f32-T64-d256-F1024-E8-top2", 64, 256, 1024, 8, 2, dtype="f32",
                 init="uniform", note="fp32 parity case"),
        Workload("bf16-T4096-d1024-F4096-E8-top2", 4096, 1024, 4096, 8, 2),
        Workload("bf16-T16384-d4096-F14336-E8-top2", 16384, 4096, 14336, 8, 2,
                 note="large-batch, compute-bound grouped GEMMs"),
        Workload("switch-bf16-T32768-d2048-F8192-E64-top1-cap640", 32768, 2048, 8192, 64, 1,
                 renormalize=False, capacity=640, capacity_factor=1.25, zipf_bias=1.5,
                 note="top-1, capacity drop in token order, Zipf-skewed load"),
        Workload("decode-bf16-T64-d4096-F14336-E8-top2", 64, 4096, 14336, 8, 2,
                 note="decode-sized batch, HBM weight streaming"),
        Workload("finegrained-bf16-T4096-d2048-F1024-E64-top6", 4096, 2048, 1024, 64, 6,
                 note="fine-grained experts: many small experts, larger k"),
        Workload("expertchoice-bf16-T4096-d1024-F4096-E8-C1024", 4096, 1024, 4096, 8, 2,
                 routing="expert", note="expert-choice routing: each expert takes its top "
                 "C = T k / E = 1024 tokens (the default workload's shape)"),
        Workload("switch-reroute-bf16-T32768-d2048-F8192-E64-top1-cap640", 32768, 2048, 8192, 64,
                 1, renormalize=False, capacity=640, capacity_factor=1.25, zipf_bias=1.5,
                 overflow="reroute", note="the Switch workload with overflow rerouted to each "
                 "token's next-best expert instead of dropped"),
    )
}

(TINY, MEDIUM, LARGE, SWITCH, DECODE, FINEGRAINED, EXPERTCHOICE,
 SWITCH_REROUTE) = WORKLOADS.values()


@dataclass
class Inputs:
    """Stored inputs of one workload (bf16 tensors as uint16 bit patterns)."""

    wl: Workload
    x: np.ndarray
    W_r: np.ndarray
    logit_bias: np.ndarray | None
    W1: np.ndarray
    b1: np.ndarray
    W2: np.ndarray
    b2: np.ndarray

    def as_f32(self, name: str) -> np.ndarray:
        """The stored tensor ``name`` widened exactly to fp32."""
        a = getattr(self, name)
        if a is None:
            return None
        return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a


def router_noise(T: int, E: int, sigma: float, seed: int) -> np.ndarray:
    """(T, E) fp32 Gaussian noise of standard deviation sigma for noisy
    gating, drawn from its own stream (the caller of the layer draws it)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7, 0])))
    return (g.standard_normal((T, E)) * sigma).astype(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly to fp32 (in chunks, on threads for
    large arrays, without full-size temporaries)."""
    u = np.ascontiguousarray(u, dtype=np.uint16)
    out = np.empty(u.shape, dtype=np.uint32)
    src, dst = u.reshape(-1), out.reshape(-1)

    def conv(c: int) -> None:
        lo, hi = c * _CHUNK, min(src.size, (c + 1) * _CHUNK)
        d = dst[lo:hi]
        d[...] = src[lo:hi]
        d <<= np.uint32(16)

    nchunks = (src.size + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            conv(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(conv, range(nchunks)))
    return out.view(np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _draw(seed: int, stream: int, n: int, kind: str, scale: float,
          dtype: str = "f32") -> np.ndarray:
    """n values: kind "normal" -> N(0, scale^2); "uniform" -> U(-scale, scale),
    drawn in fp32; dtype "bf16" returns them rounded to bf16 bit patterns
    (each chunk rounded in the thread that drew it)."""
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, c])))
        if kind == "normal":
            v = g.standard_normal(hi - lo, dtype=np.float32)
            v *= np.float32(scale)
        else:
            v = g.random(hi - lo, dtype=np.float32)
            v *= np.float32(2.0 * scale)
            v -= np.float32(scale)
        out[lo:hi] = f32_to_bf16_bits(v) if dtype == "bf16" else v

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def zipf_logit_bias(E: int, scale: float) -> np.ndarray:
    """Per-expert router logit bias ``scale * ln(1/rank)``, rank_e = e + 1 (fp32)."""
    rank = np.arange(1, E + 1, dtype=np.float64)
    return (scale * np.log(1.0 / rank)).astype(np.float32)


def make_inputs(wl: Workload, seed: int = 0) -> Inputs:
    """Draw every stored input of workload ``wl`` from ``seed``."""
    T, d, F, E = wl.T, wl.d, wl.F, wl.E
    Er = E - wl.n_shared  # experts the router covers
    dt = wl.dtype
    x = _draw(seed, _S_X, T * d, "normal", 1.0, dt).reshape(T, d)
    if wl.init == "uniform":
        W_r = _draw(seed, _S_WR, Er * d, "uniform", 1.0 / math.sqrt(d)).reshape(Er, d)
        W1 = _draw(seed, _S_W1, E * F * d, "uniform", 1.0 / math.sqrt(d), dt).reshape(E, F, d)
        W2 = _draw(seed, _S_W2, E * d * F, "uniform", 1.0 / math.sqrt(F), dt).reshape(E, d, F)
    else:
        W_r = _draw(seed, _S_WR, Er * d, "normal", 0.02).reshape(Er, d)
        W1 = _draw(seed, _S_W1, E * F * d, "normal", 1.0 / math.sqrt(d), dt).reshape(E, F, d)
        W2 = _draw(seed, _S_W2, E * d * F, "normal", 1.0 / math.sqrt(F), dt).reshape(E, d, F)
    b1 = _draw(seed, _S_B1, E * F, "uniform", 1.0 / math.sqrt(d), dt).reshape(E, F)
    b2 = _draw(seed, _S_B2, E * d, "uniform", 1.0 / math.sqrt(F), dt).reshape(E, d)
    bias = zipf_logit_bias(Er, wl.zipf_bias) if wl.zipf_bias else None
    return Inputs(wl, x, W_r, bias, W1, b1, W2, b2)
