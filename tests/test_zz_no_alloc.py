"""moe_dispatch_noalloc, the dispatch call that needs no workspace, against
moe_dispatch on the same routing.

Callers whose GPU memory is all handed out up front by another component
(a serving engine's fixed pool, a plugin host that owns every allocation)
cannot give the library a workspace; this entry point runs the dispatch on a
fixed scratch array inside the library instead.  Its results must be the
ones moe_dispatch gives (bit-exact: the dispatch is integer bookkeeping and
row copies), on two calls in a row, so no state from one call leaks into the
next, and rows past the kept ones must keep the caller's fill (a wrong
scratch layout would most likely show up as writes there).  The file sorts
last so that a stop-at-first-failure run has already run every other test
when it gets here.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300 import inputs as I
from sparse_mixture_experts_71_b300.layer import device_inputs

pytestmark = pytest.mark.gpu

FILL = -5

CASES = [
    I.MEDIUM,                                                   # 4096 tokens, top-2, E=8, no cap
    I.SWITCH.with_(name="switch-small", T=8192, d=256, F=512),  # top-1, E=64, capacity 640
    I.TINY,                                                     # fp32 rows
    # one shared expert: K = k + 1 = 3 assignments per token, the shared one never capped
    I.MEDIUM.with_(name="shared-capped", T=3000, d=128, F=256, E=9, n_shared=1, capacity=500),
    # exactly the scratch bound: T * k = 65536 assignments, 256 counting blocks
    I.MEDIUM.with_(name="at-bound", T=32768, d=64, F=64),
]


def _cfg(wl):
    return B.config(wl.T, wl.d, wl.F, wl.E, wl.k, wl.dtype, wl.capacity, wl.renormalize,
                    n_shared=wl.n_shared)


def _routing(wl, D, cfg, ws):
    K = wl.k + wl.n_shared
    idx = torch.empty((wl.T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, K), dtype=torch.float32, device="cuda")
    B.route(cfg, D["x"], D["W_r"], idx, w, ws, logit_bias=D["logit_bias"])
    return idx, w


def _dispatch(wl, D, cfg, idx, w, ws=None):
    K = wl.k + wl.n_shared
    n = wl.T * K
    out = dict(offsets=torch.full((wl.E + 1,), FILL, dtype=torch.int32, device="cuda"),
               slot_of=torch.full((wl.T, K), FILL, dtype=torch.int32, device="cuda"),
               perm_token=torch.full((n,), FILL, dtype=torch.int32, device="cuda"),
               perm_w=torch.full((n,), float(FILL), dtype=torch.float32, device="cuda"),
               x_perm=torch.full((n, wl.d), float(FILL), dtype=D["x"].dtype, device="cuda"))
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
    for name in ("perm_token", "perm_w", "x_perm"):
        assert torch.equal(a[name][:nk], b[name][:nk]), name
        tail = a[name][nk:]
        assert bool((tail == FILL).all()), f"{name}: rows past the {nk} kept ones were written"
    return nk


def test_noalloc_dispatch_matches_workspace_dispatch():
    prepared = []
    for wl in CASES:
        D = device_inputs(I.make_inputs(wl, seed=2))
        cfg = _cfg(wl)
        ws = B.workspace(cfg)
        idx, w = _routing(wl, D, cfg, ws)
        prepared.append((wl, D, cfg, idx, w, _dispatch(wl, D, cfg, idx, w, ws)))
    # two calls in a row on each case, the cases interleaved: no state carries over
    for _ in range(2):
        for wl, D, cfg, idx, w, ref in prepared:
            nk = _same(_dispatch(wl, D, cfg, idx, w), ref)
            assert 0 < nk <= wl.T * (wl.k + wl.n_shared)
            if wl.capacity is not None and wl.n_shared:
                # the shared expert keeps every token; routed experts at most capacity
                counts = torch.diff(ref["offsets"]).cpu().numpy()
                assert counts[0] == wl.T and counts[1:].max() <= wl.capacity


def test_noalloc_dispatch_rejects_batches_beyond_its_scratch():
    lib = B.load()
    fake = 1 << 20  # never dereferenced: the call fails first
    for cfg in (B.config(40000, 64, 64, 8, 2),             # 80000 assignments > 65536
                B.config(65537, 64, 64, 8, 1),             # one past the bound
                B.config(21846, 64, 64, 9, 2, n_shared=1),  # 65538 with the shared column
                B.config(64, 64, 64, 300, 2)):             # E > 256
        st = lib.moe_dispatch_noalloc(ctypes.byref(cfg), fake, fake, None, fake, fake, fake,
                                      None, fake, None)
        assert st == 4  # MOE_ERR_UNSUPPORTED


def _drv(res):
    """Unpack a cuda.bindings driver result, raising on an error code."""
    from cuda.bindings import driver as drv
    err, *rest = res if isinstance(res, tuple) else (res,)
    assert err == drv.CUresult.CUDA_SUCCESS, err
    return rest[0] if len(rest) == 1 else rest


def test_noalloc_dispatch_in_a_second_context():
    """A host that makes its own driver-API context (as a plugin host may)
    gets the scratch array's address in that context, not the one looked up
    in the primary context: the call made there gives the same result, and
    the primary context's next call is still right."""
    drv = pytest.importorskip("cuda.bindings.driver")
    wl = I.MEDIUM.with_(name="ctx", T=1000, d=64, F=64)
    D = device_inputs(I.make_inputs(wl, seed=3))
    cfg = _cfg(wl)
    ws = B.workspace(cfg)
    idx, w = _routing(wl, D, cfg, ws)
    ref = _dispatch(wl, D, cfg, idx, w, ws)
    _same(_dispatch(wl, D, cfg, idx, w), ref)  # primary context: the address is cached

    n = wl.T * wl.k
    host_in = {"x": D["x"].view(torch.int16).cpu().numpy(), "idx": idx.cpu().numpy(),
               "w": w.cpu().numpy()}
    sizes = {"offsets": 4 * (wl.E + 1), "slot_of": 4 * n, "perm_token": 4 * n, "perm_w": 4 * n,
             "x_perm": 2 * n * wl.d}
    _drv(drv.cuInit(0))
    dev = _drv(drv.cuDeviceGet(torch.cuda.current_device()))
    ctx = _drv(drv.cuCtxCreate(None, 0, dev))  # now current on this thread
    ptrs = {}
    try:
        for name, a in host_in.items():
            ptrs[name] = _drv(drv.cuMemAlloc(a.nbytes))
            _drv(drv.cuMemcpyHtoD(ptrs[name], np.ascontiguousarray(a), a.nbytes))
        for name, nbytes in sizes.items():
            ptrs[name] = _drv(drv.cuMemAlloc(nbytes))
            _drv(drv.cuMemsetD8(ptrs[name], 0xAB, nbytes))
        p = {k: int(v) for k, v in ptrs.items()}
        st = B.load().moe_dispatch_noalloc(ctypes.byref(cfg), p["x"], p["idx"], p["w"],
                                           p["offsets"], p["slot_of"], p["perm_token"],
                                           p["perm_w"], p["x_perm"], None)
        assert st == 0
        _drv(drv.cuCtxSynchronize())
        got = {}
        for name, dt, shape in (("offsets", np.int32, (wl.E + 1,)), ("slot_of", np.int32, (n,)),
                                ("perm_token", np.int32, (n,)), ("perm_w", np.float32, (n,)),
                                ("x_perm", np.int16, (n, wl.d))):
            a = np.empty(shape, dtype=dt)
            _drv(drv.cuMemcpyDtoH(a, ptrs[name], a.nbytes))
            got[name] = a
    finally:
        for v in ptrs.values():
            drv.cuMemFree(v)
        _drv(drv.cuCtxPopCurrent())
        _drv(drv.cuCtxDestroy(ctx))
    nk = int(ref["offsets"][-1])
    assert np.array_equal(got["offsets"], ref["offsets"].cpu().numpy())
    assert np.array_equal(got["slot_of"], ref["slot_of"].cpu().numpy().reshape(-1))
    assert np.array_equal(got["perm_token"][:nk], ref["perm_token"][:nk].cpu().numpy())
    assert np.array_equal(got["perm_w"][:nk], ref["perm_w"][:nk].cpu().numpy())
    assert np.array_equal(got["x_perm"][:nk],
                          ref["x_perm"][:nk].view(torch.int16).cpu().numpy())
    # back in the primary context: its cached address still serves it
    _same(_dispatch(wl, D, cfg, idx, w), ref)
