"""GPU parity on small and degenerate shapes: ragged token counts, one
expert, k = E, many experts, capacity 0 / 1 / >= T, empty experts, empty
batch, fp32 and bf16, plus the device-side error record."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from parity import LibRun, assert_y_close, oracle_on, to_np
from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300 import inputs as I

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, d, F, E, k, dtype, capacity, renormalize
    ("t1", 1, 64, 128, 8, 2, "bf16", None, True),
    ("t63-f32", 63, 64, 96, 8, 2, "f32", None, True),
    ("t65-ragged", 65, 24, 40, 5, 2, "bf16", None, True),
    ("e1-dense", 100, 32, 64, 1, 1, "f32", None, True),
    ("k-eq-e", 70, 32, 64, 4, 4, "f32", None, True),
    ("e64-top1-cap", 300, 64, 128, 64, 1, "bf16", 3, False),
    ("e256-top8", 130, 32, 64, 256, 8, "bf16", None, True),
    ("e200-top3-cap", 257, 40, 48, 200, 3, "f32", 2, True),
    ("cap0", 50, 32, 64, 4, 2, "bf16", 0, True),
    ("cap1-k2", 77, 32, 64, 3, 2, "f32", 1, True),
    ("cap-ge-T", 90, 32, 64, 4, 2, "bf16", 90, True),
    ("no-renorm-k2", 64, 64, 64, 8, 2, "f32", None, False),
    ("big-rows", 2000, 256, 512, 16, 2, "bf16", 200, True),
]


def _wl(name, T, d, F, E, k, dtype, cap, renorm, zipf=0.0):
    return I.Workload(name, T, d, F, E, k, dtype=dtype, renormalize=renorm, capacity=cap,
                      zipf_bias=zipf, init="uniform" if dtype == "f32" else "normal")


def _check(wl, inp, r):
    g_logits = to_np(r["logits"])
    ref = oracle_on(inp, wl, logits=g_logits)
    assert np.array_equal(to_np(r["idx"]), ref.idx)
    assert np.array_equal(to_np(r["counts"]), ref.counts)
    assert np.array_equal(to_np(r["offsets"]), ref.offsets)
    assert np.array_equal(to_np(r["slot_of"]), ref.slot_of)
    nk = int(ref.offsets[-1])
    assert np.array_equal(to_np(r["perm_token"])[:nk], ref.perm_token)
    assert abs(float(r["aux"][0]) - ref.aux) <= 1e-5 * max(1.0, ref.aux)
    assert abs(float(r["z"][0]) - ref.z_loss) <= 1e-5 * max(1.0, ref.z_loss)
    assert_y_close(to_np(r["y"]), ref.y, wl.dtype)
    return ref


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_small_shapes(case):
    wl = _wl(*case)
    inp = I.make_inputs(wl, seed=11)
    run = LibRun(wl, inp)
    r = run.staged()
    ref = _check(wl, inp, r)
    if wl.capacity == 0:
        assert not torch.any(r["y"].float() != 0)
    f = run.forward()
    assert torch.equal(f["y"], r["y"])
    assert torch.equal(f["z"], r["z"])
    assert B.get_device_error(run.ws)[0] == 0
    del ref


def test_empty_experts_and_zipf_skew():
    """A strong per-expert logit bias leaves most experts empty."""
    wl = _wl("zipf", 500, 64, 128, 16, 1, "bf16", 40, False, zipf=6.0)
    inp = I.make_inputs(wl, seed=3)
    r = LibRun(wl, inp).staged()
    ref = _check(wl, inp, r)
    assert np.sum(ref.counts == 0) >= 4 and np.any(~ref.kept)


def test_logits_in_routes_identically():
    """Routing from caller-given logits: ties go to the lower expert index."""
    wl = _wl("ties", 96, 32, 64, 8, 3, "f32", None, True)
    inp = I.make_inputs(wl, seed=5)
    logits = np.round(np.random.default_rng(0).standard_normal((96, 8)), 1).astype(np.float32)
    logits[::3, 5] = logits[::3, 2]  # exact ties
    run = LibRun(wl, inp)
    r = run.staged(logits_in=torch.from_numpy(logits).cuda())
    assert np.array_equal(to_np(r["logits"]), logits)
    ref = oracle_on(inp, wl, logits=logits)
    assert np.array_equal(to_np(r["idx"]), ref.idx)
    assert_y_close(to_np(r["y"]), ref.y, wl.dtype)


def test_empty_batch():
    wl = _wl("t0", 0, 32, 64, 4, 2, "bf16", None, True)
    inp = I.make_inputs(wl, seed=0)
    run = LibRun(wl, inp)
    r = run.staged()
    assert float(r["aux"][0]) == 0.0 and not torch.any(r["counts"] != 0)
    assert float(r["z"][0]) == 0.0
    assert not torch.any(r["offsets"] != 0)


def test_out_of_range_expert_is_flagged_not_written():
    """An expert index outside [0, E) given to moe_dispatch is skipped and
    recorded in the workspace; the other assignments are still dispatched."""
    wl = _wl("bad-idx", 40, 32, 64, 4, 2, "bf16", None, True)
    inp = I.make_inputs(wl, seed=1)
    run = LibRun(wl, inp)
    r = run.staged()
    idx = r["idx"].clone()
    idx[7, 1] = 9
    off = torch.empty(5, dtype=torch.int32, device="cuda")
    slot = torch.empty((40, 2), dtype=torch.int32, device="cuda")
    perm = torch.empty(80, dtype=torch.int32, device="cuda")
    xp = torch.empty((80, 32), dtype=torch.bfloat16, device="cuda")
    B.dispatch(run.cfg, run.dev["x"], idx, off, slot, perm, xp, run.ws)
    st, code, info = B.get_device_error(run.ws)
    assert (st, code, info) == (6, 1, 7 * 2 + 1)
    assert int(slot[7, 1]) == -1 and int(off[-1]) == 79
    assert B.get_device_error(run.ws)[0] == 0  # the record was cleared


SEGMENTS = {
    # 16 experts: every expert on the CTA-pair GEMMs, all tile kinds in one launch
    "pair-tiles": [0, 1, 127, 128, 129, 255, 256, 257, 300, 640, 31, 32, 33, 95, 96, 97],
    # 20 experts: full, partial and nearly empty experts side by side
    "e20-mixed": [640, 300, 256, 129, 128, 127, 100, 64, 63, 33, 32, 31, 17, 5, 1, 1, 0, 0,
                  200, 400],
    "e20-all-150": [150] * 20,  # one full and one partial token tile each
    "e20-all-100": [100] * 20,  # every expert a single partial token tile
}


@pytest.mark.parametrize("name", list(SEGMENTS))
def test_segment_sizes_around_tile_boundaries(name):
    """Expert segments of chosen sizes around the grouped GEMMs' token-tile
    sizes (32, 64, 128, 256 rows) in one batch, routed from caller-given
    logits with the experts interleaved in token order, on the wide-batch
    GEMM path (T*k >= 96*E)."""
    sizes = SEGMENTS[name]
    T, E = sum(sizes), len(sizes)
    wl = _wl(name, T, 128, 384, E, 1, "bf16", None, False)
    assert T * wl.k >= 96 * E
    inp = I.make_inputs(wl, seed=4)
    expert = np.repeat(np.arange(E), sizes)
    np.random.default_rng(1).shuffle(expert)
    logits = np.random.default_rng(2).standard_normal((T, E)).astype(np.float32)
    logits[np.arange(T), expert] = 8.0  # the chosen expert is the top-1
    run = LibRun(wl, inp)
    r = run.staged(logits_in=torch.from_numpy(logits).cuda())
    ref = oracle_on(inp, wl, logits=logits)
    assert np.array_equal(to_np(r["counts"]), np.array(sizes))
    assert np.array_equal(to_np(r["offsets"]), ref.offsets)
    assert np.array_equal(to_np(r["perm_token"])[:T], ref.perm_token)
    assert_y_close(to_np(r["y"]), ref.y, wl.dtype)
    assert B.get_device_error(run.ws)[0] == 0


def test_stalled_pipeline_wait_reports_time_out_and_context_survives():
    """The bounded mbarrier wait the tensor-core pipelines use, on a barrier
    nothing completes, gives up after its limit and records code 2 (time-out)
    in the workspace; the error record reads back, clears, and the next layer
    call on the same workspace and context runs normally."""
    wl = _wl("after-timeout", 2048, 64, 128, 8, 2, "bf16", None, True)
    inp = I.make_inputs(wl, seed=6)
    run = LibRun(wl, inp)
    B.check_wait_timeout(run.ws, 2_000_000)  # 2 ms
    assert B.get_device_error(run.ws) == (6, 2, 900)
    assert B.get_device_error(run.ws)[0] == 0  # cleared
    r = run.staged()
    _check(wl, inp, r)
    assert B.get_device_error(run.ws)[0] == 0


NOISY = [
    # name, T, d, F, E, k, dtype: one case per router kernel
    ("noise-mma", 2048, 256, 256, 8, 2, "bf16"),    # mma.sync router (E <= 16)
    ("noise-tc", 2048, 256, 256, 40, 2, "bf16"),    # tcgen05 router (16 < E <= 64)
    # tcgen05 router on a large batch with a ragged last block (33000 = 257 x 128 + 104)
    ("noise-tc-large", 33000, 128, 128, 40, 2, "bf16"),
    ("noise-warp", 300, 64, 64, 8, 2, "f32"),       # warp router
    ("noise-tile", 200, 64, 64, 100, 3, "bf16"),    # tile router (E > 64)
]


@pytest.mark.parametrize("case", NOISY, ids=[c[0] for c in NOISY])
def test_noisy_gating(case):
    """Caller-drawn noise added to the router logits (noisy gating): the
    logits used for routing match the oracle's x W_r + noise, routing from
    them is bit-exact, and forward equals the staged calls."""
    name, T, d, F, E, k, dt = case
    wl = _wl(name, T, d, F, E, k, dt, None, True)
    inp = I.make_inputs(wl, seed=12)
    noise_np = I.router_noise(T, E, 0.5, seed=3)
    noise = torch.from_numpy(noise_np).cuda()
    run = LibRun(wl, inp)
    r = run.staged(noise=noise)
    g = to_np(r["logits"])
    want = O.router_logits(inp.as_f32("x"), inp.W_r, None, noise_np)
    assert np.max(np.abs(g - want)) <= 2e-5 * max(1.0, float(np.max(np.abs(want))))
    assert np.max(np.abs(g - O.router_logits(inp.as_f32("x"), inp.W_r))) > 0.1  # noise applied
    _check(wl, inp, r)
    f = run.forward(noise=noise)
    assert torch.equal(f["y"], r["y"]) and torch.equal(f["logits"], r["logits"])


def test_balance_bias_update_matches_oracle_and_evens_out_load():
    """Auxiliary-loss-free balancing: the bias step from a routed batch's
    counts equals the oracle's, and repeating route + step on a Zipf-skewed
    router brings the first-choice loads toward balance."""
    wl = _wl("balance", 2048, 64, 64, 16, 2, "bf16", None, True, zipf=1.0)
    inp = I.make_inputs(wl, seed=9)
    run = LibRun(wl, inp)
    bias = run.dev["logit_bias"].clone()
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    counts = torch.empty(wl.E, dtype=torch.int32, device="cuda")

    def route():
        B.route(run.cfg, run.dev["x"], run.dev["W_r"], idx, w, run.ws, logit_bias=bias,
                expert_counts=counts)
        top1 = torch.bincount(idx[:, 0].long(), minlength=wl.E)
        return float(top1.max()) / (wl.T / wl.E)

    first = route()
    want = O.balance_bias_update(to_np(bias), to_np(counts), 0.02)
    B.update_balance_bias(run.cfg, counts, bias, 0.02)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(bias), want)
    for _ in range(99):
        route()
        B.update_balance_bias(run.cfg, counts, bias, 0.02)
    last = route()
    assert first > 3.0 and last < 1.6


SHARED = [
    # name, T, d, F, E, k, n_shared, dtype, capacity
    ("shared1-tc", 2048, 128, 256, 9, 2, 1, "bf16", None),    # CTA-pair GEMMs, mma router
    ("shared2-cap", 600, 64, 128, 10, 2, 2, "bf16", 50),      # capacity: shared experts uncapped
    ("shared1-f32", 100, 32, 64, 6, 1, 1, "f32", None),       # SIMT path
]


@pytest.mark.parametrize("case", SHARED, ids=[c[0] for c in SHARED])
def test_shared_experts(case):
    """Shared experts (always active, weight 1, never capped) beside k routed
    ones: routing, counts, the dispatch layout and y against the oracle, and
    forward equal to the staged calls."""
    name, T, d, F, E, k, ns, dt, cap = case
    wl = I.Workload(name, T, d, F, E, k, dtype=dt, renormalize=True, capacity=cap,
                    init="uniform" if dt == "f32" else "normal", n_shared=ns)
    inp = I.make_inputs(wl, seed=13)
    run = LibRun(wl, inp)
    r = run.staged()
    ref = _check(wl, inp, r)
    assert np.array_equal(to_np(r["idx"])[:, k:], np.tile(np.arange(ns), (T, 1)))
    assert np.all(to_np(r["w"])[:, k:] == 1.0)
    assert np.all(ref.kept[:, k:]) and np.all(ref.kept_count[:ns] == T)
    f = run.forward()
    assert torch.equal(f["y"], r["y"]) and torch.equal(f["counts"], r["counts"])
    assert torch.equal(f["aux"], r["aux"]) and torch.equal(f["z"], r["z"])
