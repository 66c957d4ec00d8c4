"""GPU parity of expert-choice routing (each expert takes its top-C tokens by
router probability) against the oracle, routing from the kernels' own fp32
logits.

The oracle's probabilities are fp64 and the kernels' fp32, so where two
tokens' probabilities lie within rounding of an expert's C-th largest value
either may be chosen: the test accepts a different choice only there, checks
that the kernels' choice is otherwise exactly the oracle's, and evaluates the
oracle's layer on the kernels' choice.  Rows, slots, gathered rows and the
expert counts are then compared bit for bit, and y within the layer
tolerances."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from parity import LibRun, assert_y_close, to_np
from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300 import inputs as I

pytestmark = pytest.mark.gpu

P_RTOL = 4e-6  # fp32 softmax against fp64

CASES = [
    # name, T, d, F, E, k, dtype, capacity
    ("ec-bf16", 300, 256, 512, 8, 2, "bf16", None),
    ("ec-f32-ragged", 63, 64, 96, 4, 1, "f32", None),
    ("ec-e1-ties", 70, 32, 64, 1, 1, "f32", 10),
    ("ec-cap0", 50, 32, 64, 4, 2, "bf16", 0),
    ("ec-all-tokens", 90, 32, 64, 4, 4, "bf16", None),
    ("ec-e16-mma-router", 1100, 128, 256, 16, 2, "bf16", None),
    ("ec-e64-tc-router", 1100, 128, 128, 64, 2, "bf16", None),
    ("ec-e200-tile-router", 257, 40, 48, 200, 3, "f32", None),
    ("ec-chunks", 3000, 256, 512, 8, 1, "bf16", 700),
]


def _wl(name, T, d, F, E, k, dtype, cap):
    return I.Workload(name, T, d, F, E, k, dtype=dtype, capacity=cap, routing="expert",
                      init="uniform" if dtype == "f32" else "normal")


def _check_selection(r, ref, E):
    """The kernels' choice per expert: ascending, and the oracle's except
    between tokens whose probabilities are within rounding of the C-th."""
    C = ref.C
    gsel = to_np(r["perm_token"])[:E * C].reshape(E, C).astype(np.int64)
    for e in range(E):
        row = gsel[e]
        assert np.all(np.diff(row) > 0), f"expert {e}: not ascending"
        if np.array_equal(row, ref.sel[e]):
            continue
        p = ref.probs[:, e]
        thr = np.sort(p)[::-1][C - 1]
        for t in np.setxor1d(row, ref.sel[e]):
            assert abs(p[t] - thr) <= P_RTOL * thr, f"expert {e}, token {t}: not a near tie"
    return gsel


def _check(wl, inp, run, r):
    E, T = wl.E, wl.T
    g = to_np(r["logits"])
    ref = O.expert_choice_forward(inp.as_f32("x"), None, inp.as_f32("W1"), inp.as_f32("b1"),
                                  inp.as_f32("W2"), inp.as_f32("b2"), k=wl.k,
                                  capacity=wl.capacity, logits=g, tokens=np.array([], np.int64))
    C = ref.C
    assert r["C"] == C
    assert to_np(r["offsets"]).tolist() == [e * C for e in range(E + 1)]
    assert to_np(r["counts"]).tolist() == [C] * E
    gsel = _check_selection(r, ref, E)
    np.testing.assert_allclose(to_np(r["perm_w"])[:E * C],
                               np.take_along_axis(ref.probs.T, gsel, 1).ravel(), rtol=P_RTOL)
    slot = np.full((T, E), -1, np.int64)
    for e in range(E):
        slot[gsel[e], e] = e * C + np.arange(C)
    assert np.array_equal(to_np(r["slot_of"]), slot)
    assert np.array_equal(to_np(r["x_perm"])[:E * C], inp.as_f32("x")[gsel.ravel()])
    assert abs(float(r["z"][0]) - ref.z_loss) <= 1e-5 * max(1.0, ref.z_loss)
    full = O.expert_choice_forward(inp.as_f32("x"), None, inp.as_f32("W1"), inp.as_f32("b1"),
                                   inp.as_f32("W2"), inp.as_f32("b2"), k=wl.k,
                                   capacity=wl.capacity, logits=g, sel=gsel)
    max_abs, rel = assert_y_close(to_np(r["y"]), full.y, wl.dtype)
    print(f"{wl.name}: C {C}, max|dy| {max_abs:.3e}, rel {rel:.3e}")
    return ref, gsel


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_expert_choice_small_shapes(case):
    wl = _wl(*case)
    inp = I.make_inputs(wl, seed=21)
    run = LibRun(wl, inp)
    r = run.staged_ec()
    ref, gsel = _check(wl, inp, run, r)
    if wl.E == 1:  # equal probabilities: the first C tokens
        assert gsel.tolist() == [list(range(ref.C))]
    if wl.capacity == 0:
        assert not to_np(r["y"]).any()
    # the whole layer in one call: the same bits, aux 0, deterministic
    f = run.forward()
    assert torch.equal(f["y"], r["y"]) and torch.equal(f["logits"], r["logits"])
    assert float(f["aux"][0]) == 0.0 and torch.equal(f["counts"], r["counts"])
    assert torch.equal(f["z"], r["z"])
    assert torch.equal(run.forward()["y"], f["y"])


def test_expert_choice_full_workload():
    wl = I.EXPERTCHOICE
    inp = I.make_inputs(wl, seed=0)
    run = LibRun(wl, inp)
    r = run.staged_ec()
    g = to_np(r["logits"])
    ref_logits = O.router_logits(inp.as_f32("x"), inp.W_r, inp.logit_bias)
    assert np.max(np.abs(g - ref_logits)) <= 2e-5 * max(np.max(np.abs(ref_logits)), 1.0)
    _check(wl, inp, run, r)
    assert torch.equal(run.forward()["y"], r["y"])


def test_expert_choice_logits_in_and_noise():
    """Caller logits replace the router; noise shifts the logits it uses."""
    wl = _wl("ec-logits", 200, 64, 96, 8, 2, "bf16", None)
    inp = I.make_inputs(wl, seed=22)
    run = LibRun(wl, inp)
    base = run.staged_ec()
    again = run.staged_ec(logits_in=base["logits"])
    assert torch.equal(again["perm_token"], base["perm_token"])
    assert torch.equal(again["y"], base["y"])
    noise = torch.from_numpy(I.router_noise(wl.T, wl.E, 1.0, seed=5)).cuda()
    noisy = run.staged_ec(noise=noise)
    np.testing.assert_allclose(to_np(noisy["logits"]), to_np(base["logits"]) + to_np(noise),
                               rtol=1e-6, atol=1e-6)
    _check(wl, inp, run, noisy)
