"""The decode-sized forward pass that evaluates every expert on all T tokens
(moe_forward on bf16 token-choice layers with T <= 64 and T k >= 4 E): its
outputs against the staged sparse calls (route, dispatch, expert_ffn,
combine) bit for bit - each (expert, token) row of the dense GEMMs is the
sparse path's row, and the combine applies the same weight and the same
drops in the same order - and against the oracle within the bf16 tolerances.

"Mixture of Experts: Scaling Parameters Without Scaling Compute", section
"The MoE layer" (the layer's output is the weighted sum of the chosen
experts' outputs; only the evaluation order of the experts changes here) and
"The central problem: load balancing" (the capacity drop in token order and
the auxiliary loss, which the dense path's combine and its finishing block
compute).
"""
import numpy as np
import pytest
import torch

from parity import LibRun, assert_y_close, oracle_on, to_np
from sparse_mixture_experts_71_b300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = [
    # T, d, F, E, k, capacity, renormalize, zipf
    I.Workload("dense-64", 64, 512, 1024, 8, 2),
    I.Workload("dense-40-cap", 40, 256, 768, 8, 2, capacity=9, zipf_bias=1.0),  # drops; T % 32 != 0
    I.Workload("dense-e48-k4", 64, 256, 512, 48, 4),                          # tile router (E > 32)
    I.Workload("dense-33-top1", 33, 128, 256, 8, 1, renormalize=False, capacity=3, zipf_bias=1.5),
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_dense_decode_forward(wl):
    assert wl.T <= 64 and wl.T * wl.k >= 4 * wl.E and wl.T * wl.k < 96 * wl.E
    inp = I.make_inputs(wl, seed=5)
    run = LibRun(wl, inp)
    staged = run.staged()
    f = run.forward()
    # routing outputs: the same router kernel, the same bits
    assert torch.equal(f["logits"], staged["logits"])
    assert torch.equal(f["counts"], staged["counts"])
    # the losses: the forward runs the router in fewer, larger blocks, so the
    # per-block partial sums of p and of the squared log-sum-exp add up in
    # another order - within two fp32 ulps of the staged calls' values
    for key in ("aux", "z"):
        a, b = float(f[key][0]), float(staged[key][0])
        assert abs(a - b) <= 2.4e-7 * max(abs(b), 1e-30), (key, a, b)
    # the layer output: the sparse path's bits
    assert torch.equal(f["y"], staged["y"]), (
        f"max |dense - sparse| {float((f['y'].float() - staged['y'].float()).abs().max()):.3e}")
    # and the oracle, routing from the kernels' logits
    ref = oracle_on(inp, wl, logits=to_np(f["logits"]), layout=False)
    max_abs, rel = assert_y_close(to_np(f["y"]), ref.y, wl.dtype)
    assert abs(float(f["aux"][0]) - ref.aux) <= 1e-5 * max(1.0, ref.aux)
    if wl.capacity is not None:
        dropped = ~ref.kept.any(axis=1)
        assert np.all(to_np(f["y"])[dropped] == 0.0)
    # deterministic
    assert torch.equal(run.forward()["y"], f["y"])
    print(f"{wl.name}: max|dy| {max_abs:.2e} rel {rel:.2e}")
