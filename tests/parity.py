"""Helpers of the GPU parity tests: run libmoe through its C ABI on stored
inputs, run the oracle on the same inputs, compare.

Tolerances (end-to-end layer output y against the fp64 oracle):
  bf16 layers: max |dy| <= 2e-2 and ||dy||_F / ||y||_F <= 5e-3
  fp32 layers: max |dy| <= 1e-4
Routing indices, counts, offsets, drop decisions and the dispatch layout are
compared bit-exactly when both sides route from the same fp32 logits.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300.layer import device_inputs

BF16_MAX_ABS, BF16_REL_FRO, F32_MAX_ABS = 2e-2, 5e-3, 1e-4
NEAR_TIE = 1e-6


def cfg_of(wl):
    return B.config(wl.T, wl.d, wl.F, wl.E, wl.k, wl.dtype, wl.capacity, wl.renormalize,
                    wl.n_shared, routing=wl.routing, overflow=wl.overflow)


def y_error(y_gpu: np.ndarray, y_ref: np.ndarray):
    d = y_gpu.astype(np.float64) - y_ref
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    nrm = float(np.linalg.norm(y_ref))
    rel = float(np.linalg.norm(d)) / nrm if nrm > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_y_close(y_gpu, y_ref, dtype):
    max_abs, rel = y_error(y_gpu, y_ref)
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"max abs {max_abs:.3e}"
    else:
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_FRO, f"max abs {max_abs:.3e} rel {rel:.3e}"
    return max_abs, rel


def near_tie_tokens(probs: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest probabilities differ by < 1e-6."""
    E = probs.shape[1]
    if k >= E:
        return np.zeros(probs.shape[0], bool)
    s = -np.sort(-probs, axis=1)
    return (s[:, k - 1] - s[:, k]) < NEAR_TIE


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


class LibRun:
    """Every stage of one layer call through the C ABI, with its outputs."""

    def __init__(self, wl, inp, dev=None, stream=None):
        self.wl, self.inp = wl, inp
        self.dev = dev if dev is not None else device_inputs(inp)
        self.cfg = cfg_of(wl)
        self.ws = B.workspace(self.cfg)
        self.stream = stream

    def staged(self, logits_in=None, noise=None):
        wl, D, T, E = self.wl, self.dev, self.wl.T, self.wl.E
        k = wl.k + wl.n_shared  # columns per token (routed, then shared)
        kr = B.ranked_columns(self.cfg)  # router columns (rerouting: the next-best too)
        dt = D["x"].dtype
        cuda = D["x"].device
        n = T * k
        r = {}
        r["logits"] = torch.empty((T, E - wl.n_shared), dtype=torch.float32, device=cuda)
        r["idx"] = torch.empty((T, kr), dtype=torch.int32, device=cuda)
        r["w"] = torch.empty((T, kr), dtype=torch.float32, device=cuda)
        r["counts"] = torch.empty(E, dtype=torch.int32, device=cuda)
        r["aux"] = torch.empty(1, dtype=torch.float32, device=cuda)
        r["z"] = torch.full((1,), -1.0, dtype=torch.float32, device=cuda)
        B.route(self.cfg, D["x"], D["W_r"], r["idx"], r["w"], self.ws, logit_bias=D["logit_bias"],
                logits_in=logits_in, logits_out=r["logits"], expert_counts=r["counts"],
                aux_out=r["aux"], z_loss_out=r["z"], logit_noise=noise, stream=self.stream)
        r["offsets"] = torch.empty(E + 1, dtype=torch.int32, device=cuda)
        r["slot_of"] = torch.empty((T, k), dtype=torch.int32, device=cuda)
        r["perm_token"] = torch.full((max(n, 1),), -7, dtype=torch.int32, device=cuda)
        r["perm_w"] = torch.empty(max(n, 1), dtype=torch.float32, device=cuda)
        r["x_perm"] = torch.empty((max(n, 1), wl.d), dtype=dt, device=cuda)
        B.dispatch(self.cfg, D["x"], r["idx"], r["offsets"], r["slot_of"], r["perm_token"],
                   r["x_perm"], self.ws, topk_w=r["w"], perm_w=r["perm_w"], stream=self.stream)
        r["y_perm"] = torch.empty((max(n, 1), wl.d), dtype=torch.float32, device=cuda)
        B.expert_ffn(self.cfg, r["x_perm"], r["offsets"], D["W1"], D["b1"], D["W2"], D["b2"],
                     r["y_perm"], self.ws, perm_w=r["perm_w"], stream=self.stream)
        r["y"] = torch.empty((T, wl.d), dtype=dt, device=cuda)
        B.combine(self.cfg, r["y_perm"], r["slot_of"], r["y"], stream=self.stream)
        torch.cuda.synchronize()
        return r

    def staged_ec(self, logits_in=None, noise=None):
        """Expert choice: route_expert_choice (with the gather), expert_ffn,
        combine."""
        wl, D, T, E = self.wl, self.dev, self.wl.T, self.wl.E
        C = B.expert_choice_capacity(self.cfg)
        R = max(E * C, 1)
        dt, cuda = D["x"].dtype, D["x"].device
        r = {"C": C}
        r["logits"] = torch.empty((T, E), dtype=torch.float32, device=cuda)
        r["offsets"] = torch.full((E + 1,), -7, dtype=torch.int32, device=cuda)
        r["perm_token"] = torch.full((R,), -7, dtype=torch.int32, device=cuda)
        r["perm_w"] = torch.empty(R, dtype=torch.float32, device=cuda)
        r["slot_of"] = torch.full((T, E), -7, dtype=torch.int32, device=cuda)
        r["x_perm"] = torch.empty((R, wl.d), dtype=dt, device=cuda)
        r["counts"] = torch.full((E,), -7, dtype=torch.int32, device=cuda)
        r["z"] = torch.full((1,), -1.0, dtype=torch.float32, device=cuda)
        B.route_expert_choice(self.cfg, D["x"], D["W_r"], r["offsets"], r["perm_token"],
                              r["perm_w"], r["slot_of"], self.ws, x_perm=r["x_perm"],
                              logit_bias=D["logit_bias"], logit_noise=noise,
                              logits_in=logits_in, logits_out=r["logits"],
                              expert_counts=r["counts"], z_loss_out=r["z"], stream=self.stream)
        r["y_perm"] = torch.empty((R, wl.d), dtype=torch.float32, device=cuda)
        B.expert_ffn(self.cfg, r["x_perm"], r["offsets"], D["W1"], D["b1"], D["W2"], D["b2"],
                     r["y_perm"], self.ws, perm_w=r["perm_w"], stream=self.stream)
        r["y"] = torch.empty((T, wl.d), dtype=dt, device=cuda)
        B.combine(self.cfg, r["y_perm"], r["slot_of"], r["y"], stream=self.stream)
        torch.cuda.synchronize()
        return r

    def forward(self, noise=None):
        D, wl = self.dev, self.wl
        y = torch.empty_like(D["x"])
        aux = torch.empty(1, dtype=torch.float32, device=y.device)
        counts = torch.empty(wl.E, dtype=torch.int32, device=y.device)
        logits = torch.empty((wl.T, wl.E - wl.n_shared), dtype=torch.float32, device=y.device)
        z = torch.full((1,), -1.0, dtype=torch.float32, device=y.device)
        B.forward(self.cfg, D["x"], D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], y, self.ws,
                  logit_bias=D["logit_bias"], aux_out=aux, expert_counts=counts,
                  logits_out=logits, z_loss_out=z, logit_noise=noise, stream=self.stream)
        torch.cuda.synchronize()
        return dict(y=y, aux=aux, counts=counts, logits=logits, z=z)


def oracle_on(inp, wl, logits=None, tokens=None, layout=True):
    """The oracle on stored inputs (optionally routing from given fp32 logits)."""
    return O.moe_forward(inp.as_f32("x"), inp.W_r, inp.as_f32("W1"), inp.as_f32("b1"),
                         inp.as_f32("W2"), inp.as_f32("b2"), k=wl.k,
                         renormalize=wl.renormalize, capacity=wl.capacity,
                         logit_bias=inp.logit_bias, logits=logits, tokens=tokens, layout=layout,
                         n_shared=wl.n_shared, reroute=wl.overflow == "reroute")


def sample_tokens(wl, ref_route, n_kept: int = 1024, tile: int = 256, per_tile: int = 4,
                  n_dropped: int = 64, seed: int = 0) -> np.ndarray:
    """A seeded token sample for the largest workloads: in every `tile`-row
    tile of every expert's segment of the permuted rows (the GEMMs' token
    tiles), the tokens of its first and last rows and of `per_tile` - 2 random
    rows; under a cap, the last kept and first and last dropped tokens of every
    expert that overflowed; then random tokens with at least one kept
    assignment until `n_kept` of them are in, and `n_dropped` random tokens
    whose every assignment was dropped (their output must be 0).
    `ref_route` is the oracle's result with the dispatch layout."""
    g = np.random.default_rng(seed)
    T = wl.T
    pick = set()
    off, perm = ref_route.offsets, ref_route.perm_token
    for e in range(len(off) - 1):
        for r0 in range(int(off[e]), int(off[e + 1]), tile):
            r1 = min(r0 + tile, int(off[e + 1]))
            rows = {r0, r1 - 1} | set(g.integers(r0, r1, size=max(per_tile - 2, 0)).tolist())
            pick |= {int(perm[r]) for r in rows}
    idx, kept = ref_route.idx, ref_route.kept
    if wl.capacity is not None:
        for e in range(wl.E):
            sel = (idx == e)
            kt = np.nonzero((sel & kept).any(axis=1))[0]
            dt = np.nonzero((sel & ~kept).any(axis=1))[0]
            if kt.size:
                pick.add(int(kt[-1]))
            if dt.size:
                pick.add(int(dt[0]))
                pick.add(int(dt[-1]))
    any_kept = kept.any(axis=1)
    kept_tokens = np.nonzero(any_kept)[0]
    have = sum(1 for t in pick if any_kept[t])
    if have < n_kept:
        rest = np.setdiff1d(kept_tokens, np.fromiter(pick, np.int64, len(pick)))
        pick |= set(g.choice(rest, size=min(n_kept - have, rest.size), replace=False).tolist())
    dropped = np.nonzero(~any_kept)[0]
    if dropped.size:
        pick |= set(g.choice(dropped, size=min(n_dropped, dropped.size), replace=False).tolist())
    return np.array(sorted(pick), np.int64)
