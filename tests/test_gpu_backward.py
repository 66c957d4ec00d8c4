"""GPU parity of the backward pass (moe_backward) against the oracle's fp64
gradients, routing from the kernels' own fp32 logits.

Tolerance: the kernels keep the expert pre-activations, activations and the
scaled upstream rows in bf16 (as the forward keeps H) and accumulate in fp32,
so each gradient is compared by its relative Frobenius error, at most 2e-2
(a handful of bf16 roundings, 2^-9 each, on the way), and its largest
element error relative to the gradient's largest magnitude, at most 5e-2.
fp32 layers keep every intermediate in fp32 and accumulate with fp32 FMA
over at most a few thousand terms (relative error ~ sqrt(n) 2^-24, a few
1e-6), so their bounds are 2e-5 (Frobenius) and 1e-4 (largest element)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from parity import LibRun, oracle_on, to_np
from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300 import inputs as I

pytestmark = pytest.mark.gpu

REL_FRO, REL_MAX = 2e-2, 5e-2
REL_FRO_F32, REL_MAX_F32 = 2e-5, 1e-4

CASES = [
    # name, T, d, F, E, k, capacity, renormalize, zipf, aux_grad, z_grad
    ("bwd-k2", 300, 256, 512, 8, 2, None, True, 0.0, 0.0, 0.0),
    ("bwd-k2-losses", 300, 256, 512, 8, 2, None, True, 0.0, 0.7, 0.3),
    ("bwd-top1-cap", 400, 128, 256, 8, 1, 40, False, 1.5, 0.5, 0.0),
    ("bwd-decode", 64, 256, 512, 8, 2, None, True, 0.0, 0.0, 0.0),     # single-CTA GEMMs
    ("bwd-e64-tc-router", 1100, 128, 128, 64, 2, 30, True, 1.0, 0.1, 0.1),
    ("bwd-ragged", 1500, 64, 192, 5, 2, 500, True, 1.0, 0.0, 0.0),
    # d and d_ff not multiples of 64: the 2-D box forms of the MN-major reads
    ("bwd-2d-boxes", 700, 136, 200, 6, 2, None, True, 0.5, 0.1, 0.0),
    # rows narrower than one 64-column box
    ("bwd-tiny-dims", 65, 24, 40, 5, 2, None, True, 0.0, 0.0, 0.0),
    # 20 routed experts (the dx product's tensor-core form, its K padded to
    # 24) and d not a multiple of its 128-column tiles
    ("bwd-e20", 700, 200, 256, 20, 2, None, True, 0.5, 0.1, 0.1),
    # mid size: ~1024 rows per expert, so the weight-gradient GEMMs' segment
    # reduction walks 8 K tiles of 128 per expert, on both GEMM kernels' wide path
    ("bwd-mid", 4096, 512, 2048, 8, 2, None, True, 0.0, 0.01, 0.001),
]


# The layer variants: shared experts, rerouting on overflow, expert choice.
VARIANTS = [
    # workload, aux_grad, z_grad
    (I.Workload("bwd-shared", 500, 128, 256, 9, 2, n_shared=1), 0.3, 0.1),
    (I.Workload("bwd-shared2-cap", 700, 128, 256, 10, 2, capacity=80, zipf_bias=1.0,
                n_shared=2), 0.2, 0.0),
    (I.Workload("bwd-reroute", 600, 128, 256, 8, 2, capacity=100, zipf_bias=1.0,
                overflow="reroute"), 0.5, 0.2),
    (I.Workload("bwd-reroute-top1-raw", 400, 128, 256, 8, 1, renormalize=False, capacity=40,
                zipf_bias=1.5, overflow="reroute"), 0.0, 0.0),
    (I.Workload("bwd-reroute-e64", 1100, 128, 128, 64, 2, capacity=30, zipf_bias=1.0,
                overflow="reroute"), 0.1, 0.1),
    (I.Workload("bwd-ec", 512, 128, 256, 8, 2, routing="expert"), 0.0, 0.3),
    (I.Workload("bwd-ec-cap", 300, 128, 256, 8, 2, capacity=40, zipf_bias=1.0,
                routing="expert"), 0.7, 0.0),   # aux_grad is ignored: no balancing loss
    (I.Workload("bwd-ec-e64", 1100, 128, 128, 64, 2, routing="expert"), 0.0, 0.1),
    # fp32 layers (the CUDA-core path): plain, capped top-1 with raw weights,
    # shared experts, rerouting, expert choice; ragged d_ff and segments
    (I.Workload("bwd-f32", 300, 256, 520, 8, 2, dtype="f32"), 0.3, 0.2),
    (I.Workload("bwd-f32-top1-cap", 400, 128, 264, 8, 1, dtype="f32", renormalize=False,
                capacity=40, zipf_bias=1.5), 0.5, 0.0),
    (I.Workload("bwd-f32-shared", 200, 64, 136, 6, 2, dtype="f32", capacity=50, n_shared=1),
     0.2, 0.1),
    (I.Workload("bwd-f32-reroute", 500, 128, 200, 8, 2, dtype="f32", capacity=80, zipf_bias=1.0,
                overflow="reroute"), 0.1, 0.1),
    (I.Workload("bwd-f32-ec", 256, 128, 192, 8, 2, dtype="f32", routing="expert"), 0.0, 0.2),
]


def test_segment_maps_match_driver_encoding():
    """The weight-gradient products read each expert segment through its own
    tensor map, edited on the device from a whole-buffer map; every edited map
    must equal the driver's encoding of the same segment (runs before any
    product loads through one)."""
    ws = torch.empty(3 << 20, dtype=torch.uint8, device="cuda")
    B.check_segment_maps(ws)


def _close(name, got, want, f32=False):
    got = np.asarray(got, np.float64)
    d = got - want
    fro = np.linalg.norm(d) / max(np.linalg.norm(want), 1e-30)
    mx = np.max(np.abs(d)) / max(np.max(np.abs(want)), 1e-30)
    bf, bm = (REL_FRO_F32, REL_MAX_F32) if f32 else (REL_FRO, REL_MAX)
    assert fro <= bf and mx <= bm, f"{name}: rel fro {fro:.3e}, rel max {mx:.3e}"
    return fro


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(case):
    name, T, d, F, E, k, cap, renorm, zipf, aux_grad, z_grad = case
    wl = I.Workload(name, T, d, F, E, k, capacity=cap, renormalize=renorm, zipf_bias=zipf)
    inp = I.make_inputs(wl, seed=41)
    run = LibRun(wl, inp)
    D = run.dev
    g = run.forward()["logits"]
    dy_np = I.router_noise(T, d, 1.0, seed=42)  # any seeded (T, d) draw serves as dy
    dy = torch.from_numpy(dy_np).to(torch.bfloat16).cuda()
    cfg = run.cfg
    ws = B.backward_workspace(cfg)
    f32 = dict(dtype=torch.float32, device="cuda")
    out = dict(dx=torch.empty_like(D["x"]), dW_r=torch.empty((E, d), **f32),
               dW1=torch.empty((E, F, d), **f32), db1=torch.empty((E, F), **f32),
               dW2=torch.empty((E, d, F), **f32), db2=torch.empty((E, d), **f32))
    B.backward(cfg, D["x"], D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], dy, out["dx"],
               out["dW_r"], out["dW1"], out["db1"], out["dW2"], out["db2"], ws,
               logit_bias=D["logit_bias"], aux_grad=aux_grad, z_grad=z_grad)
    torch.cuda.synchronize()
    assert B.get_device_error(ws)[0] == 0
    ref = O.moe_backward(inp.as_f32("x"), inp.W_r, inp.as_f32("W1"), inp.as_f32("b1"),
                         inp.as_f32("W2"), inp.as_f32("b2"),
                         dy.float().cpu().numpy(), k=k, renormalize=renorm, capacity=cap,
                         logit_bias=inp.logit_bias, logits=to_np(g), aux_grad=aux_grad,
                         z_grad=z_grad)
    errs = {n: _close(n, to_np(out[n]), ref[n]) for n in out}
    print(name, " ".join(f"{n} {v:.2e}" for n, v in errs.items()))
    # deterministic: a second call gives the same bits
    again = {n: torch.empty_like(v) for n, v in out.items()}
    B.backward(cfg, D["x"], D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], dy, again["dx"],
               again["dW_r"], again["dW1"], again["db1"], again["dW2"], again["db2"], ws,
               logit_bias=D["logit_bias"], aux_grad=aux_grad, z_grad=z_grad)
    torch.cuda.synchronize()
    for n in out:
        assert torch.equal(out[n], again[n]), n


def _lib_backward(run, dy, aux_grad, z_grad):
    D, wl = run.dev, run.wl
    ws = B.backward_workspace(run.cfg)
    f32 = dict(dtype=torch.float32, device="cuda")
    E, d, F = wl.E, wl.d, wl.F
    out = dict(dx=torch.empty_like(D["x"]), dW_r=torch.empty(tuple(D["W_r"].shape), **f32),
               dW1=torch.empty((E, F, d), **f32), db1=torch.empty((E, F), **f32),
               dW2=torch.empty((E, d, F), **f32), db2=torch.empty((E, d), **f32))
    B.backward(run.cfg, D["x"], D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], dy, out["dx"],
               out["dW_r"], out["dW1"], out["db1"], out["dW2"], out["db2"], ws,
               logit_bias=D["logit_bias"], aux_grad=aux_grad, z_grad=z_grad)
    torch.cuda.synchronize()
    assert B.get_device_error(ws)[0] == 0
    return out


@pytest.mark.parametrize("variant", VARIANTS, ids=[v[0].name for v in VARIANTS])
def test_variant_backward_matches_oracle(variant):
    """Shared experts, rerouting and expert choice: moe_backward against the
    oracle's gradients of the same variant, routing (and, for expert choice,
    the selection) taken from the kernels' forward pass."""
    wl, aux_grad, z_grad = variant
    inp = I.make_inputs(wl, seed=47)
    run = LibRun(wl, inp)
    dy = torch.from_numpy(I.router_noise(wl.T, wl.d, 1.0, seed=48)).to(run.dev["x"].dtype).cuda()
    args = (inp.as_f32("x"), inp.W_r, inp.as_f32("W1"), inp.as_f32("b1"), inp.as_f32("W2"),
            inp.as_f32("b2"), dy.float().cpu().numpy())
    if wl.routing == "expert":
        r = run.staged_ec()
        C = r["C"]
        sel = to_np(r["perm_token"])[:wl.E * C].reshape(wl.E, C).astype(np.int64)
        ref = O.expert_choice_backward(*args, k=wl.k, capacity=wl.capacity,
                                       logit_bias=inp.logit_bias, logits=to_np(r["logits"]),
                                       sel=sel, z_grad=z_grad)
    else:
        g = run.forward()["logits"]
        if wl.overflow == "reroute":  # the case moves slots to other experts
            fwd = oracle_on(inp, wl, logits=to_np(g), layout=False)
            assert np.any(fwd.idx[:, :wl.k] != O.top_k(to_np(g), wl.k))
        ref = O.moe_backward(*args, k=wl.k, renormalize=wl.renormalize, capacity=wl.capacity,
                             logit_bias=inp.logit_bias, logits=to_np(g), aux_grad=aux_grad,
                             z_grad=z_grad, n_shared=wl.n_shared,
                             reroute=wl.overflow == "reroute")
    out = _lib_backward(run, dy, aux_grad, z_grad)
    errs = {n: _close(n, to_np(out[n]), ref[n], wl.dtype == "f32") for n in out}
    print(wl.name, " ".join(f"{n} {v:.2e}" for n, v in errs.items()))
    again = _lib_backward(run, dy, aux_grad, z_grad)
    for n in out:
        assert torch.equal(out[n], again[n]), n


def test_backward_empty_batch_is_zero():
    wl = I.Workload("bwd-empty", 0, 64, 128, 4, 2)
    cfg = B.config(0, 64, 128, 4, 2)
    ws = B.backward_workspace(cfg)
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = [torch.full(s, 7.0, **f32) for s in ((4, 64), (4, 128, 64), (4, 128), (4, 64, 128),
                                                  (4, 64))]
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((4, 128, 64), dtype=torch.bfloat16, device="cuda")
    B.backward(cfg, x, torch.zeros((4, 64), **f32), w, torch.zeros((4, 128), dtype=torch.bfloat16,
               device="cuda"), torch.zeros((4, 64, 128), dtype=torch.bfloat16, device="cuda"),
               torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda"), x, x, *outs, ws)
    torch.cuda.synchronize()
    assert all(not o.any() for o in outs)
    assert wl.T == 0


def test_layer_backward_matches_the_c_call():
    """MoELayer.backward (the Python layer API) gives the C call's bits."""
    from sparse_mixture_experts_71_b300.layer import MoELayer
    wl = I.Workload("bwd-layer", 200, 128, 256, 8, 2)
    inp = I.make_inputs(wl, seed=43)
    run = LibRun(wl, inp)
    D = run.dev
    layer = MoELayer(D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], k=2,
                     logit_bias=D["logit_bias"])
    dy = torch.from_numpy(I.router_noise(200, 128, 1.0, seed=44)).to(torch.bfloat16).cuda()
    g = layer.backward(D["x"], dy, aux_grad=0.2, z_grad=0.05)
    ws = B.backward_workspace(run.cfg)
    want = {n: torch.empty_like(v) for n, v in g.items()}
    B.backward(run.cfg, D["x"], D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], dy, want["dx"],
               want["dW_r"], want["dW1"], want["db1"], want["dW2"], want["db2"], ws,
               logit_bias=D["logit_bias"], aux_grad=0.2, z_grad=0.05)
    torch.cuda.synchronize()
    for n in g:
        assert torch.equal(g[n], want[n]), n
