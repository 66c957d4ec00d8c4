"""GPU parity of rerouting on overflow (a slot the capacity cap drops is
offered once, in token order, to the token's next-best expert) against the
oracle, routing from the kernels' own fp32 logits: the router's K2 ranked
experts, the drop pass, the offers, the row layout and the gather bit-exact,
the weights and the layer output within tolerance."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from parity import LibRun, assert_y_close, oracle_on, to_np
from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, d, F, E, k, dtype, capacity, renormalize, zipf
    ("rr-bf16-k2", 300, 256, 512, 8, 2, "bf16", 60, True, 1.5),
    ("rr-f32-top1", 200, 64, 96, 4, 1, "f32", 40, False, 2.0),
    ("rr-tc-router", 1100, 128, 128, 64, 2, "bf16", 30, True, 1.0),
    ("rr-mma-router-k4", 1024, 128, 256, 16, 4, "bf16", 200, True, 1.5),
    ("rr-tile-router", 257, 40, 48, 100, 3, "f32", 5, True, 1.0),
    ("rr-k-eq-E", 64, 32, 64, 2, 2, "f32", 10, True, 0.0),    # no next-best expert: drop only
    ("rr-cap0", 50, 32, 64, 4, 2, "bf16", 0, True, 0.0),      # every offer refused
    ("rr-no-cap", 90, 32, 64, 4, 2, "bf16", None, True, 0.0),  # nothing dropped
    ("rr-ragged", 2000, 64, 64, 8, 2, "bf16", 300, True, 2.0),
]


def _wl(name, T, d, F, E, k, dtype, cap, renorm, zipf):
    return I.Workload(name, T, d, F, E, k, dtype=dtype, capacity=cap, renormalize=renorm,
                      zipf_bias=zipf, overflow="reroute",
                      init="uniform" if dtype == "f32" else "normal")


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_reroute(case):
    wl = _wl(*case)
    T, E, k = wl.T, wl.E, wl.k
    inp = I.make_inputs(wl, seed=31)
    run = LibRun(wl, inp)
    r = run.staged()
    g = to_np(r["logits"])
    ref = oracle_on(inp, wl, logits=g)
    K2 = min(2 * k, E)
    # the router's ranking and weights (the next-best normalised as the choices)
    ranked = O.top_k(g, K2)
    assert np.array_equal(to_np(r["idx"]), ranked)
    den = (np.take_along_axis(ref.probs, ranked[:, :k], 1).sum(1, keepdims=True)
           if wl.renormalize else 1.0)
    np.testing.assert_allclose(to_np(r["w"]), np.take_along_axis(ref.probs, ranked, 1) / den,
                               rtol=3e-6, atol=1e-7)
    assert np.array_equal(to_np(r["counts"]), ref.counts)
    assert abs(float(r["aux"][0]) - ref.aux) <= 1e-5 * max(1.0, ref.aux)
    # drop pass, offers, rows: bit-exact
    assert np.array_equal(to_np(r["offsets"]), ref.offsets)
    assert np.array_equal(to_np(r["slot_of"]), ref.slot_of)
    nk = int(ref.offsets[-1])
    assert np.array_equal(to_np(r["perm_token"])[:nk], ref.perm_token)
    assert np.array_equal(to_np(r["x_perm"])[:nk], inp.as_f32("x")[ref.perm_token])
    rows = ref.slot_of[ref.kept]
    np.testing.assert_allclose(to_np(r["perm_w"])[rows], ref.w[ref.kept], rtol=3e-6, atol=1e-7)
    drop = O.moe_forward(inp.as_f32("x"), inp.W_r, inp.as_f32("W1"), inp.as_f32("b1"),
                         inp.as_f32("W2"), inp.as_f32("b2"), k=k, renormalize=wl.renormalize,
                         capacity=wl.capacity, logits=g, tokens=np.array([], np.int64))
    moved = int(ref.kept.sum() - drop.kept.sum())
    max_abs, rel = assert_y_close(to_np(r["y"]), ref.y, wl.dtype)
    print(f"{wl.name}: kept {nk}/{T * k}, rerouted {moved}, max|dy| {max_abs:.3e}")
    if wl.name == "rr-cap0":
        assert nk == 0 and not to_np(r["y"]).any()
    # the whole layer in one call: the same bits
    f = run.forward()
    assert torch.equal(f["y"], r["y"]) and torch.equal(f["counts"], r["counts"])
    assert torch.equal(f["aux"], r["aux"]) and torch.equal(f["z"], r["z"])


def test_reroute_moves_slots_on_a_skewed_router():
    """The skewed cases above reroute a good share of the dropped slots."""
    wl = _wl(*CASES[0])
    inp = I.make_inputs(wl, seed=31)
    r = LibRun(wl, inp).staged()
    ref = oracle_on(inp, wl, logits=to_np(r["logits"]), tokens=np.array([], np.int64))
    drop = O.moe_forward(inp.as_f32("x"), inp.W_r, inp.as_f32("W1"), inp.as_f32("b1"),
                         inp.as_f32("W2"), inp.as_f32("b2"), k=wl.k, capacity=wl.capacity,
                         logits=to_np(r["logits"]), tokens=np.array([], np.int64))
    assert ref.kept.sum() > drop.kept.sum() + 20


def test_reroute_full_switch_workload():
    """The Switch workload with rerouting at full size: layout bit-exact, y on
    a seeded token sample covering every expert and the drop boundaries."""
    from parity import sample_tokens
    wl = I.SWITCH_REROUTE
    inp = I.make_inputs(wl, seed=0)
    run = LibRun(wl, inp)
    r = run.staged()
    g = to_np(r["logits"])
    ref = oracle_on(inp, wl, logits=g, tokens=np.array([], np.int64))
    assert np.array_equal(to_np(r["idx"]), O.top_k(g, 2))
    assert np.array_equal(to_np(r["offsets"]), ref.offsets)
    assert np.array_equal(to_np(r["slot_of"]), ref.slot_of)
    nk = int(ref.offsets[-1])
    assert np.array_equal(to_np(r["perm_token"])[:nk], ref.perm_token)
    tokens = sample_tokens(wl, ref)
    # and the rerouted tokens among the sample
    moved = np.nonzero(ref.kept[:, 0] & (ref.idx[:, 0] != O.top_k(g, 1)[:, 0]))[0]
    tokens = np.unique(np.concatenate([tokens, moved[:64]]))
    full = oracle_on(inp, wl, logits=g, tokens=tokens, layout=False)
    max_abs, rel = assert_y_close(to_np(r["y"])[tokens], full.y, wl.dtype)
    print(f"{wl.name}: kept {nk}/{wl.T}, rerouted {len(moved)}, max|dy| {max_abs:.3e}")
    assert len(moved) > 0
    assert torch.equal(run.forward()["y"], r["y"])
