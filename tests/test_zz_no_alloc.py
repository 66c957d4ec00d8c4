"""moe_dispatch_noalloc, the dispatch call that needs no workspace, against
moe_dispatch on the same routing.

Callers whose GPU memory is all handed out up front by another component
(a serving engine's fixed pool, a plugin host that owns every allocation)
cannot give the library a workspace; this entry point runs the dispatch on a
fixed scratch array inside the library instead.  Its results must be the
ones moe_dispatch gives (bit-exact: the dispatch is integer bookkeeping and
row copies), on two calls in a row, so no state from one call leaks into the
next.  The file sorts last so that a stop-at-first-failure run has already
run every other test when it gets here.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300 import inputs as I
from sparse_mixture_experts_71_b300.layer import device_inputs

pytestmark = pytest.mark.gpu

CASES = [
    I.MEDIUM,                                                # 4096 tokens, top-2, E=8, no cap
    I.SWITCH.with_(name="switch-small", T=8192, d=256, F=512),  # top-1, E=64, capacity 640
]


def _routing(wl, D, cfg, ws):
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    B.route(cfg, D["x"], D["W_r"], idx, w, ws, logit_bias=D["logit_bias"])
    return idx, w


def _dispatch(wl, D, cfg, idx, w, ws=None):
    n = wl.T * wl.k
    out = dict(offsets=torch.full((wl.E + 1,), -5, dtype=torch.int32, device="cuda"),
               slot_of=torch.full((wl.T, wl.k), -5, dtype=torch.int32, device="cuda"),
               perm_token=torch.full((n,), -5, dtype=torch.int32, device="cuda"),
               perm_w=torch.full((n,), -5.0, dtype=torch.float32, device="cuda"),
               x_perm=torch.zeros((n, wl.d), dtype=D["x"].dtype, device="cuda"))
    if ws is None:
        B.dispatch_noalloc(cfg, D["x"], idx, out["offsets"], out["slot_of"], out["perm_token"],
                           out["x_perm"], topk_w=w, perm_w=out["perm_w"])
    else:
        B.dispatch(cfg, D["x"], idx, out["offsets"], out["slot_of"], out["perm_token"],
                   out["x_perm"], ws, topk_w=w, perm_w=out["perm_w"])
    torch.cuda.synchronize()
    return out


def _same(a, b):
    nk = int(a["offsets"][-1])
    assert torch.equal(a["offsets"], b["offsets"])
    assert torch.equal(a["slot_of"], b["slot_of"])
    assert torch.equal(a["perm_token"][:nk], b["perm_token"][:nk])
    assert torch.equal(a["perm_w"][:nk], b["perm_w"][:nk])
    assert torch.equal(a["x_perm"][:nk], b["x_perm"][:nk])
    return nk


def test_noalloc_dispatch_matches_workspace_dispatch():
    prepared = []
    for wl in CASES:
        D = device_inputs(I.make_inputs(wl, seed=2))
        cfg = B.config(wl.T, wl.d, wl.F, wl.E, wl.k, wl.dtype, wl.capacity, wl.renormalize)
        ws = B.workspace(cfg)
        idx, w = _routing(wl, D, cfg, ws)
        prepared.append((wl, D, cfg, idx, w, _dispatch(wl, D, cfg, idx, w, ws)))
    # two calls in a row on each case, the cases interleaved: no state carries over
    for _ in range(2):
        for wl, D, cfg, idx, w, ref in prepared:
            nk = _same(_dispatch(wl, D, cfg, idx, w), ref)
            assert 0 < nk <= wl.T * wl.k


def test_noalloc_dispatch_rejects_batches_beyond_its_scratch():
    lib = B.load()
    cfg = B.config(40000, 64, 64, 8, 2)  # 80000 assignments > 65536
    fake = 1 << 20                       # never dereferenced: the call fails first
    st = lib.moe_dispatch_noalloc(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, None,
                                  fake, None)
    assert st == 4  # MOE_ERR_UNSUPPORTED
    cfg = B.config(64, 64, 64, 300, 2)   # E > 256
    assert lib.moe_dispatch_noalloc(ctypes.byref(cfg), fake, fake, None, fake, fake, fake,
                                    None, fake, None) == 4
