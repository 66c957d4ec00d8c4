"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test names the passage or the closed form it checks.  None of them
re-types an oracle formula: expected values come from the pages' worked
examples, from exact special cases, from brute force with plain loops, or
from library routines (torch on CPU, fp64).
"""
import math
import random

import numpy as np
import pytest
import torch
import torch.nn.functional as TF

from conftest import read_golden
from oracle import moe_oracle as O
from sparse_mixture_experts_71_b300.inputs import SWITCH

rng = np.random.default_rng(1234)


def _rand_layer(T, d, F, E, seed=0):
    g = np.random.default_rng(seed)
    return dict(
        x=g.standard_normal((T, d)),
        W_r=g.standard_normal((E, d)) * 0.5,
        W1=g.standard_normal((E, F, d)) / math.sqrt(d),
        b1=g.uniform(-0.3, 0.3, (E, F)),
        W2=g.standard_normal((E, d, F)) / math.sqrt(F),
        b2=g.uniform(-0.3, 0.3, (E, d)),
    )


# ---------------------------------------------------------------- routing pins

def test_day59_worked_top2_example():
    """day-59 "Replace one MLP with many experts": probabilities of Experts
    1..8 -> the token goes to Experts 2 and 4."""
    gold = read_golden("day59_top2_example.txt")
    p = np.array([float(v) for v in gold["probs"]])
    logits = np.log(p).astype(np.float32)[None, :]
    idx = O.top_k(logits, 2)
    assert [int(i) + 1 for i in idx[0]] == [int(v) for v in gold["top2_1based"]]
    # softmax of ln p gives p back (the printed probabilities sum to 1)
    probs = O.softmax(logits)
    np.testing.assert_allclose(probs[0], p, rtol=1e-6)
    # renormalised over the two chosen experts: 0.51/0.82 and 0.31/0.82
    w = O.gate_weights(probs, idx, True)
    np.testing.assert_allclose(w[0], [0.51 / 0.82, 0.31 / 0.82], rtol=1e-6)
    # not renormalised: the router probabilities themselves
    np.testing.assert_allclose(O.gate_weights(probs, idx, False)[0], [0.51, 0.31], rtol=1e-6)


def test_ratish_router_table():
    """ratishfolio "How does MoE work?" Part 1: scores A .10 B .75 C .15 ->
    top-1 B; top-2 B and C."""
    gold = read_golden("ratish_router_table.txt")
    s = np.array([float(v) for v in gold["scores"]])
    names = "ABC"
    logits = np.log(s).astype(np.float32)[None, :]
    assert [names[i] for i in O.top_k(logits, 1)[0]] == gold["top1"]
    assert [names[i] for i in O.top_k(logits, 2)[0]] == gold["top2"]
    w = O.gate_weights(O.softmax(logits), O.top_k(logits, 2), True)
    np.testing.assert_allclose(w[0], [0.75 / 0.90, 0.15 / 0.90], rtol=1e-6)


def test_aiinbed_router_demo():
    """aiinbed "Experts and the router": Gaussian router scores (stdlib RNG,
    seed 7, 8 experts, 4 tokens), softmax, top-2, shares renormalised over the
    two.  The expected picks are computed here with plain Python floats by the
    procedure the page states; the oracle routes the same scores as fp32
    logits and must agree on picks and rounded percentages."""
    random.seed(7)
    E, k = 8, 2
    for _ in range(4):
        scores = [random.gauss(0, 1) for _ in range(E)]
        ex = [math.exp(v) for v in scores]
        tot = sum(ex)
        probs = [v / tot for v in ex]
        best = sorted(range(E), key=lambda i: probs[i], reverse=True)[:k]
        share = sum(probs[i] for i in best)
        want = [(i, round(100 * probs[i] / share)) for i in best]
        logits = np.array(scores, np.float32)[None, :]
        idx = O.top_k(logits, k)[0]
        w = O.gate_weights(O.softmax(logits), idx[None, :], True)[0]
        got = [(int(i), round(100 * float(v))) for i, v in zip(idx, w)]
        assert got == want


def test_top_k_ties_go_to_lower_index():
    """Equal logits: lower expert index first (stable descending order)."""
    g = np.array([[1.0, 3.0, 3.0, 0.0, 3.0]], np.float32)
    assert O.top_k(g, 2)[0].tolist() == [1, 2]
    assert O.top_k(g, 3)[0].tolist() == [1, 2, 4]
    z = np.zeros((1, 6), np.float32)
    assert O.top_k(z, 4)[0].tolist() == [0, 1, 2, 3]


def test_top_k_brute_force():
    """Top-k against an explicit selection loop on random fp32 logits."""
    g = rng.standard_normal((50, 7)).astype(np.float32)
    g[:, 3] = g[:, 5]  # force some ties
    for k in (1, 2, 3, 7):
        idx = O.top_k(g, k)
        for t in range(g.shape[0]):
            left = list(range(g.shape[1]))
            want = []
            for _ in range(k):
                b = left[0]
                for e in left:
                    if g[t, e] > g[t, b]:
                        b = e
                want.append(b)
                left.remove(b)
            assert idx[t].tolist() == want


def test_renormalised_weights_sum_to_one():
    """Renormalised weights of every token sum to 1 (fp64 round-off)."""
    g = (rng.standard_normal((200, 16)) * 3).astype(np.float32)
    for k in (2, 4, 16):
        w = O.gate_weights(O.softmax(g), O.top_k(g, k), True)
        assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 4e-16
        assert np.all(w > 0)


def test_softmax_matches_torch():
    g = (rng.standard_normal((40, 64)) * 5).astype(np.float32)
    want = torch.softmax(torch.from_numpy(g).double(), dim=-1).numpy()
    np.testing.assert_allclose(O.softmax(g), want, rtol=1e-13, atol=0)


# ---------------------------------------------------------- bias balancing pins

def test_balance_bias_update_by_hand():
    """Loads 10/2/2/2 (mean 4): the overloaded expert's bias drops by the step,
    the others rise by it; loads at the mean keep their bias."""
    b = np.array([0.5, -1.0, 0.0, 2.0], np.float32)
    np.testing.assert_array_equal(O.balance_bias_update(b, [10, 2, 2, 2], 0.25),
                                  np.array([0.25, -0.75, 0.25, 2.25], np.float32))
    np.testing.assert_array_equal(O.balance_bias_update(b, [4, 4, 4, 4], 0.25), b)
    np.testing.assert_array_equal(O.balance_bias_update(b, [6, 4, 2, 4], 1.0),
                                  np.array([-0.5, -1.0, 1.0, 2.0], np.float32))


def test_balance_bias_updates_even_out_a_skewed_router():
    """Repeated updates on a router skewed by a Zipf-like logit offset bring
    the top-1 loads toward balance (the purpose of the mechanism)."""
    g = np.random.default_rng(21)
    T, d, E = 2048, 32, 8
    x, W = g.standard_normal((T, d)), g.standard_normal((E, d)) * 0.05
    skew = -1.5 * np.log(np.arange(1, E + 1))
    b = np.zeros(E, np.float32)
    def imbalance(bias):
        idx = O.top_k(O.router_logits(x, W, skew + bias), 1)
        c = np.bincount(idx[:, 0], minlength=E)
        return c, c.max() / (T / E)
    c0, first = imbalance(b)
    for _ in range(60):
        c, _ = imbalance(b)
        b = O.balance_bias_update(b, c, 0.05)
    _, last = imbalance(b)
    assert first > 3.0 and last < 1.5


# ---------------------------------------------------------- noisy gating pins

def test_noise_equal_to_a_bias_row_is_the_bias_and_zero_noise_is_none():
    """Noise that is the same per-expert offset for every token gives exactly
    the logits of that offset as logit bias; zero noise changes nothing."""
    g = np.random.default_rng(8)
    x, W = g.standard_normal((40, 32)), g.standard_normal((6, 32))
    c = g.standard_normal(6)
    assert np.array_equal(O.router_logits(x, W, logit_noise=np.tile(c, (40, 1))),
                          O.router_logits(x, W, logit_bias=c))
    assert np.array_equal(O.router_logits(x, W, logit_noise=np.zeros((40, 6))),
                          O.router_logits(x, W))


def test_large_noise_on_one_expert_selects_it():
    """Noise far above the logit spread on expert j makes j every token's
    first choice (the noise is there to make the router explore)."""
    g = np.random.default_rng(9)
    x, W = g.standard_normal((64, 16)), g.standard_normal((8, 16)) * 0.1
    noise = np.zeros((64, 8))
    noise[:, 5] = 1e3
    r = O.moe_forward(x, W, np.zeros((8, 4, 16)), np.zeros((8, 4)), np.zeros((8, 16, 4)),
                      np.zeros((8, 16)), k=2, logit_noise=noise)
    assert np.all(r.idx[:, 0] == 5)


# ---------------------------------------------------------- router z-loss pins

@pytest.mark.parametrize("E,c", [(1, 0.0), (8, 0.0), (8, -2.5), (64, 3.25)])
def test_z_loss_equal_logits_closed_form(E, c):
    """All logits equal to c: log-sum-exp = c + ln E for every token, so the
    z-loss is (c + ln E)^2 (the term that keeps router logits small)."""
    g = np.full((50, E), c, np.float32)
    assert abs(O.router_z_loss(g) - (c + math.log(E)) ** 2) <= 1e-12 * max(1.0, (c + math.log(E)) ** 2)


def test_z_loss_matches_library_logsumexp():
    """Reduces to torch.logsumexp (fp64) squared and averaged over tokens."""
    g = (rng.standard_normal((333, 16)) * 4.0).astype(np.float32)
    lse = torch.logsumexp(torch.from_numpy(g).double(), dim=1)
    want = float((lse * lse).mean())
    assert abs(O.router_z_loss(g) - want) <= 1e-12 * want


def test_z_loss_dominant_logit_and_empty_batch():
    """One logit L far above the others: log-sum-exp -> L, z -> L^2; and an
    empty batch contributes 0."""
    g = np.zeros((10, 8), np.float32)
    g[:, 3] = 60.0
    assert abs(O.router_z_loss(g) - 3600.0) <= 1e-9
    assert O.router_z_loss(np.zeros((0, 8), np.float32)) == 0.0


# ---------------------------------------------------------- auxiliary loss pins

@pytest.mark.parametrize("E,k", [(1, 1), (4, 2), (8, 2), (64, 1), (8, 8)])
def test_aux_loss_uniform_routing_is_one(E, k):
    """All logits equal -> P_i = 1/E, so E * sum f_i / E = 1 exactly, whatever
    the tie-break ("The central problem: load balancing")."""
    g = np.zeros((96, E), np.float32)
    p = O.softmax(g)
    assert abs(O.aux_loss(p, O.top_k(g, k), E) - 1.0) <= 1e-14


def test_aux_loss_balanced_top1_is_one():
    """Top-1 counts exactly balanced (f_i = 1/E) -> aux = sum_i P_i = 1."""
    E, T = 8, 256
    g = rng.standard_normal((T, E)).astype(np.float32)
    g[np.arange(T), np.arange(T) % E] += 20.0
    p = O.softmax(g)
    idx = O.top_k(g, 2)
    assert np.all(np.bincount(idx[:, 0], minlength=E) == T // E)
    assert abs(O.aux_loss(p, idx, E) - 1.0) <= 1e-13


def test_aux_loss_day59_imbalance():
    """day-59 "The router can create traffic jams": 8 experts, 8000 tokens,
    loads 4700/800/.../200.  With one-hot routing probabilities P_i = f_i, so
    aux = 8 * sum f_i^2 = 2.995 (derived from the printed loads)."""
    gold = read_golden("day59_imbalance_loads.txt")
    E, T = int(gold["experts"][0]), int(gold["tokens"][0])
    loads = [int(v) for v in gold["loads"]]
    assert sum(loads) == T
    top1 = np.repeat(np.arange(E), loads)
    np.random.default_rng(5).shuffle(top1)
    g = np.zeros((T, E), np.float32)
    g[np.arange(T), top1] = 80.0
    p = O.softmax(g)
    idx = O.top_k(g, 2)
    assert np.array_equal(idx[:, 0], top1)
    assert abs(O.aux_loss(p, idx, E) - 2.995) <= 1e-12


def test_aux_loss_counts_top1_slot_only():
    """f_i counts the first (highest) choice only: moving a token's second
    choice does not change aux."""
    E = 4
    g = np.array([[4.0, 3.0, 0.0, 0.0], [4.0, 0.0, 3.0, 0.0]], np.float32)
    p = O.softmax(g)
    idx = O.top_k(g, 2)
    # f = (1, 0, 0, 0): aux = E * P_0
    assert abs(O.aux_loss(p, idx, E) - E * p[:, 0].mean()) <= 1e-15


# ------------------------------------------------------------- capacity pins

def test_switch_capacity_value():
    """C = ceil(1.25 * T / E) for the Switch workload: 1.25 * 32768 / 64 = 640."""
    assert O.expert_capacity(1.25, 32768, 64) == 640 == SWITCH.capacity
    assert O.expert_capacity(1.0, 10, 3) == 4


def test_capacity_day59_loads():
    """day-59 loads 4700/800/.../200 with C = ceil(1.25 * 8000 / 8) = 1250:
    expert 0 keeps its first 1250 tokens in token order, every other expert
    keeps all of its tokens; the 3450 later tokens of expert 0 are dropped."""
    gold = read_golden("day59_imbalance_loads.txt")
    E, T = int(gold["experts"][0]), int(gold["tokens"][0])
    loads = [int(v) for v in gold["loads"]]
    C = O.expert_capacity(1.25, T, E)
    assert C == 1250
    top1 = np.repeat(np.arange(E), loads)
    np.random.default_rng(9).shuffle(top1)
    kept = O.capacity_keep(top1[:, None], E, C)[:, 0]
    for e in range(E):
        toks = np.nonzero(top1 == e)[0]
        n = min(loads[e], C)
        assert kept[toks[:n]].all() and not kept[toks[n:]].any()
    assert int((~kept).sum()) == 3450


def test_capacity_slot_order_for_k2():
    """Cap 1: in (token, slot) order the first assignment to an expert wins."""
    idx = np.array([[1, 0], [0, 1], [2, 1]])
    kept = O.capacity_keep(idx, 3, 1)
    assert kept.tolist() == [[True, True], [False, False], [True, False]]


def test_dispatch_layout_brute_force():
    """Segments are expert-major and token-ascending inside an expert; every
    kept assignment has one slot, every dropped one has -1."""
    T, k, E = 37, 2, 5
    g = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.top_k(g, k)
    kept = O.capacity_keep(idx, E, 9)
    counts, kc, off, slot_of, perm = O.dispatch_layout(idx, kept, E)
    want_perm = []
    for e in range(E):
        assert counts[e] == sum(int(idx[t, j] == e) for t in range(T) for j in range(k))
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e and kept[t, j]:
                    assert slot_of[t, j] == off[0] + len(want_perm)
                    want_perm.append(t)
                elif not kept[t, j]:
                    assert slot_of[t, j] == -1
        assert off[e + 1] == len(want_perm)
    assert perm.tolist() == want_perm


# ------------------------------------------------------------------ GELU pins

def test_gelu_values():
    """GELU(0) = 0; GELU(+-1) = +-Phi(+-1); matches torch's exact GELU."""
    assert O.gelu(np.array([0.0]))[0] == 0.0
    assert abs(O.gelu(np.array([1.0]))[0] - 0.8413447460685429) <= 1e-15
    assert abs(O.gelu(np.array([-1.0]))[0] + 0.15865525393145707) <= 1e-15
    u = np.linspace(-8, 8, 1001)
    want = TF.gelu(torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(O.gelu(u), want, rtol=1e-14, atol=1e-15)


# ------------------------------------------------------- whole-layer pins

def _brute_force_dense(L, k, renormalize, capacity):
    """Run every expert on every token with plain loops, then mask by the
    gate weights (0 off the top-k and for dropped assignments)."""
    x, W_r, W1, b1, W2, b2 = (L[n] for n in ("x", "W_r", "W1", "b1", "W2", "b2"))
    T, d = x.shape
    E, F, _ = W1.shape
    logits = np.zeros((T, E), np.float32)
    for t in range(T):
        for e in range(E):
            logits[t, e] = np.float32(sum(float(W_r[e, j]) * float(x[t, j]) for j in range(d)))
    y = np.zeros((T, d))
    taken = [0] * E
    for t in range(T):
        m = max(logits[t])
        ex = [math.exp(float(v) - float(m)) for v in logits[t]]
        s = sum(ex)
        p = [v / s for v in ex]
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        share = sum(p[e] for e in order) if renormalize else 1.0
        gate = [0.0] * E
        for e in order:
            if capacity is None or taken[e] < capacity:
                taken[e] += 1
                gate[e] = p[e] / share
        for e in range(E):
            h = [0.0] * F
            for f in range(F):
                u = b1[e, f] + sum(W1[e, f, j] * x[t, j] for j in range(d))
                h[f] = 0.5 * u * (1.0 + math.erf(u / math.sqrt(2.0)))
            for i in range(d):
                o = b2[e, i] + sum(W2[e, i, f] * h[f] for f in range(F))
                y[t, i] += gate[e] * o
    return logits, y


@pytest.mark.parametrize("k,renorm,cap", [(1, False, None), (2, True, None), (2, True, 3),
                                          (3, True, 2), (1, False, 0)])
def test_forward_equals_dense_masked_brute_force(k, renorm, cap):
    """Loop-over-experts forward == every expert on every token, masked."""
    L = _rand_layer(T=9, d=5, F=6, E=4, seed=k * 10 + (cap or 0))
    logits, want = _brute_force_dense(L, k, renorm, cap)
    r = O.moe_forward(**L, k=k, renormalize=renorm, capacity=cap)
    assert np.array_equal(r.logits, logits)
    np.testing.assert_allclose(r.y, want, rtol=1e-12, atol=1e-12)


def test_shared_experts_add_their_dense_ffn():
    """n_shared experts always active ("Design variations": shared experts):
    y = the routed layer over experts n_shared.. (the pinned path above) +
    sum over the shared experts of their plain FFN (torch, fp64), and the
    routing, weights and loss are those of the routed layer alone."""
    L = _rand_layer(T=17, d=8, F=12, E=5, seed=31)
    W_r = L["W_r"][:3]  # router over the 3 routed experts
    both = dict(L, W_r=W_r)
    r = O.moe_forward(**both, k=2, renormalize=True, n_shared=2)
    routed = O.moe_forward(L["x"], W_r, L["W1"][2:], L["b1"][2:], L["W2"][2:], L["b2"][2:],
                           k=2, renormalize=True)
    t = {n: torch.from_numpy(v) for n, v in L.items()}
    shared = sum(TF.linear(TF.gelu(TF.linear(t["x"], t["W1"][e], t["b1"][e])), t["W2"][e],
                           t["b2"][e]) for e in range(2))
    np.testing.assert_allclose(r.y, routed.y + shared.numpy(), rtol=1e-12, atol=1e-12)
    assert np.array_equal(r.idx[:, :2], routed.idx + 2)
    assert np.array_equal(r.idx[:, 2:], np.tile([0, 1], (17, 1)))
    assert np.array_equal(r.w[:, 2:], np.ones((17, 2))) and np.array_equal(r.w[:, :2], routed.w)
    assert r.aux == routed.aux and r.z_loss == routed.z_loss
    assert np.array_equal(r.counts, np.concatenate([[17, 17], routed.counts]))


def test_shared_experts_are_not_capped():
    """Capacity 1: each routed expert keeps one assignment, the shared
    expert keeps every token."""
    L = _rand_layer(T=10, d=6, F=5, E=4, seed=32)
    r = O.moe_forward(**dict(L, W_r=L["W_r"][:3]), k=1, renormalize=False, capacity=1,
                      n_shared=1)
    assert r.kept[:, 1].all() and r.kept_count[0] == 10
    assert np.all(r.kept_count[1:] <= 1) and r.kept[:, 0].sum() == r.kept_count[1:].sum()


def test_single_expert_is_dense_ffn():
    """E = 1, k = 1, renormalised -> the plain Linear-GELU-Linear FFN
    (torch.nn.functional on CPU, fp64)."""
    L = _rand_layer(T=33, d=16, F=40, E=1, seed=3)
    r = O.moe_forward(**L, k=1, renormalize=True)
    t = {n: torch.from_numpy(v) for n, v in L.items()}
    want = TF.linear(TF.gelu(TF.linear(t["x"], t["W1"][0], t["b1"][0])), t["W2"][0], t["b2"][0])
    np.testing.assert_allclose(r.y, want.numpy(), rtol=1e-12, atol=1e-12)
    assert abs(r.aux - 1.0) <= 1e-15


def test_k_equals_E_is_soft_mixture():
    """k = E, renormalised -> y = sum_e p_e f_e(x) (torch, fp64)."""
    L = _rand_layer(T=21, d=12, F=20, E=5, seed=4)
    r = O.moe_forward(**L, k=5, renormalize=True)
    t = {n: torch.from_numpy(v) for n, v in L.items()}
    logits = torch.from_numpy(r.logits).double()
    p = torch.softmax(logits, -1)
    want = torch.zeros_like(t["x"])
    for e in range(5):
        fe = TF.linear(TF.gelu(TF.linear(t["x"], t["W1"][e], t["b1"][e])), t["W2"][e], t["b2"][e])
        want += p[:, e:e + 1] * fe
    np.testing.assert_allclose(r.y, want.numpy(), rtol=1e-12, atol=1e-12)
    # and the fp32 logits are the fp64 product rounded once
    want_g = (t["x"] @ t["W_r"].T).float().numpy()
    assert np.array_equal(r.logits, want_g)


def test_capacity_extremes():
    """C >= T -> same as no cap; C = 0 -> every assignment dropped, y = 0."""
    L = _rand_layer(T=30, d=8, F=16, E=4, seed=5)
    a = O.moe_forward(**L, k=2)
    b = O.moe_forward(**L, k=2, capacity=30)
    assert np.array_equal(a.y, b.y) and np.array_equal(a.slot_of, b.slot_of)
    z = O.moe_forward(**L, k=2, capacity=0)
    assert not z.y.any() and np.all(z.slot_of == -1) and z.offsets[-1] == 0
    assert z.aux == a.aux  # the loss is taken before any drop


def test_token_permutation():
    """No cap: permuting tokens permutes y and keeps aux.  With a cap the
    drop is in token order, so a permutation changes which token is dropped."""
    L = _rand_layer(T=25, d=8, F=12, E=3, seed=6)
    perm = np.random.default_rng(2).permutation(25)
    a = O.moe_forward(**L, k=2)
    Lp = dict(L, x=L["x"][perm])
    b = O.moe_forward(**Lp, k=2)
    np.testing.assert_allclose(b.y, a.y[perm], rtol=1e-12, atol=1e-13)
    assert abs(a.aux - b.aux) <= 1e-13
    ca = O.moe_forward(**L, k=1, capacity=4)
    cb = O.moe_forward(**Lp, k=1, capacity=4)
    assert not np.array_equal(ca.kept[perm], cb.kept)


def test_token_subset_matches_full():
    """Computing only some token rows gives those rows of the full output."""
    L = _rand_layer(T=40, d=8, F=12, E=4, seed=7)
    full = O.moe_forward(**L, k=2, capacity=12)
    sub = np.array([39, 0, 17, 5])
    part = O.moe_forward(**L, k=2, capacity=12, tokens=sub)
    np.testing.assert_allclose(part.y, full.y[sub], rtol=1e-12, atol=1e-13)


# ------------------------------------------- the pins catch planted mistakes

def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)


def test_planted_mistakes_are_caught(monkeypatch):
    """Plausible oracle mistakes, planted on the CPU, each fail a pin above."""
    good_topk, good_gate, good_aux = O.top_k, O.gate_weights, O.aux_loss

    # ties to the higher index
    _planted(monkeypatch, "top_k", lambda g, k: np.argsort(-np.asarray(g)[:, ::-1], axis=1,
                                                            kind="stable")[:, :k] * -1
             + np.asarray(g).shape[1] - 1)
    with pytest.raises(AssertionError):
        test_top_k_ties_go_to_lower_index()
    monkeypatch.setattr(O, "top_k", good_topk)

    # weights not renormalised
    _planted(monkeypatch, "gate_weights", lambda p, i, r: good_gate(p, i, False))
    with pytest.raises(AssertionError):
        test_day59_worked_top2_example()
    monkeypatch.setattr(O, "gate_weights", good_gate)

    # aux loss with f over all k slots instead of the top-1 choice
    def aux_all_slots(p, idx, E):
        idx = np.asarray(idx)
        f = np.bincount(idx.ravel(), minlength=E) / idx.size
        return float(E * np.sum(f * np.asarray(p).mean(0)))
    _planted(monkeypatch, "aux_loss", aux_all_slots)
    with pytest.raises(AssertionError):
        test_aux_loss_counts_top1_slot_only()
    monkeypatch.setattr(O, "aux_loss", good_aux)

    # tanh GELU instead of the exact one
    good_gelu = O.gelu
    _planted(monkeypatch, "gelu", lambda u: 0.5 * np.asarray(u) * (1 + np.tanh(
        math.sqrt(2 / math.pi) * (np.asarray(u) + 0.044715 * np.asarray(u) ** 3))))
    with pytest.raises(AssertionError):
        test_single_expert_is_dense_ffn()
    monkeypatch.setattr(O, "gelu", good_gelu)


# ---- expert-choice routing ("Design variations": experts choose their top
# tokens); the readings are listed in the oracle's header

def test_expert_choice_capacity_values():
    """C = ceil(T k / E) without a cap, the cap when given, never above T."""
    assert O.expert_choice_capacity(4096, 8, 2) == 1024
    assert O.expert_choice_capacity(10, 3, 1) == 4      # ceil(10/3)
    assert O.expert_choice_capacity(10, 3, 2) == 7      # ceil(20/3)
    assert O.expert_choice_capacity(5, 1, 2) == 5       # ceil(10/1) > T
    assert O.expert_choice_capacity(10, 3, 1, capacity=2) == 2
    assert O.expert_choice_capacity(10, 3, 1, capacity=50) == 10
    assert O.expert_choice_capacity(10, 3, 1, capacity=0) == 0


def test_expert_choice_hand_worked():
    """Two experts, four tokens, logits (a_t, 0): p[t, 0] = sigmoid(a_t).
    a = (2, -1, 0.5, 0): p0 = (.881, .269, .622, .5), p1 = 1 - p0; C = 2.
    Expert 0 takes tokens 0 and 2, expert 1 tokens 1 and 3 (worked by hand);
    each token's output is its one expert's FFN scaled by that p."""
    L = _rand_layer(T=4, d=3, F=5, E=2, seed=41)
    g = np.array([[2.0, 0.0], [-1.0, 0.0], [0.5, 0.0], [0.0, 0.0]], np.float32)
    r = O.expert_choice_forward(**L, k=1, logits=g)
    assert r.C == 2
    assert r.sel.tolist() == [[0, 2], [1, 3]]
    assert r.slot_of.tolist() == [[0, -1], [-1, 2], [1, -1], [-1, 3]]
    sig = [1 / (1 + math.exp(-a)) for a in (2.0, -1.0, 0.5, 0.0)]
    assert np.allclose(r.w, [[sig[0], sig[2]], [1 - sig[1], 1 - sig[3]]], rtol=1e-15)
    t = {n: torch.from_numpy(v) for n, v in L.items()}
    for tok, e in ((0, 0), (1, 1), (2, 0), (3, 1)):
        fe = TF.linear(TF.gelu(TF.linear(t["x"][tok], t["W1"][e], t["b1"][e])), t["W2"][e],
                       t["b2"][e]).numpy()
        pe = sig[tok] if e == 0 else 1 - sig[tok]
        np.testing.assert_allclose(r.y[tok], pe * fe, rtol=1e-12, atol=1e-15)


def test_expert_choice_ties_go_to_lower_token():
    """Equal logits: p = 1/E everywhere, so every expert takes tokens 0..C-1;
    E = 1 is the same (p = 1) and tokens from C on get y = 0."""
    r = O.expert_choice_select(np.full((9, 3), 1 / 3), 4)
    assert r.tolist() == [[0, 1, 2, 3]] * 3
    L = _rand_layer(T=7, d=4, F=6, E=1, seed=42)
    r1 = O.expert_choice_forward(**L, k=1, capacity=3)
    assert r1.sel.tolist() == [[0, 1, 2]]
    assert not r1.y[3:].any()
    t = {n: torch.from_numpy(v) for n, v in L.items()}
    want = TF.linear(TF.gelu(TF.linear(t["x"][:3], t["W1"][0], t["b1"][0])), t["W2"][0],
                     t["b2"][0])
    np.testing.assert_allclose(r1.y[:3], want.numpy(), rtol=1e-12, atol=1e-15)


def test_expert_choice_brute_force_selection():
    """With distinct probabilities each expert's chosen set is the unique
    C-subset of tokens with the largest total probability (enumerated)."""
    import itertools
    rng = np.random.default_rng(43)
    for T, E, C in ((6, 3, 2), (7, 2, 3), (5, 4, 1), (6, 2, 6)):
        p = rng.random((T, E))
        sel = O.expert_choice_select(p, C)
        for e in range(E):
            best = max(itertools.combinations(range(T), C), key=lambda s: sum(p[i, e] for i in s))
            assert sel[e].tolist() == list(best)


def test_expert_choice_all_tokens_is_soft_mixture():
    """C = T (every expert takes every token): y = sum_e p_e f_e(x), the soft
    mixture (torch, fp64); balance: every expert takes exactly C tokens."""
    L = _rand_layer(T=13, d=6, F=10, E=4, seed=44)
    r = O.expert_choice_forward(**L, k=4)  # ceil(13 * 4 / 4) = 13 = T
    assert r.C == 13 and all(sorted(s) == list(range(13)) for s in r.sel.tolist())
    t = {n: torch.from_numpy(v) for n, v in L.items()}
    p = torch.softmax(torch.from_numpy(r.logits).double(), -1)
    want = torch.zeros_like(t["x"])
    for e in range(4):
        fe = TF.linear(TF.gelu(TF.linear(t["x"], t["W1"][e], t["b1"][e])), t["W2"][e], t["b2"][e])
        want += p[:, e:e + 1] * fe
    np.testing.assert_allclose(r.y, want.numpy(), rtol=1e-12, atol=1e-12)


def test_expert_choice_dense_masked_brute_force():
    """Every expert on every token with plain loops, masked by the column-wise
    top-C of p computed by sorting each column in pure Python."""
    L = _rand_layer(T=11, d=4, F=5, E=3, seed=45)
    logits, _ = _brute_force_dense(L, 1, False, None)
    r = O.expert_choice_forward(**L, k=2)  # C = ceil(22 / 3) = 8
    assert np.array_equal(r.logits, logits) and r.C == 8
    T, E = logits.shape
    p = [[0.0] * E for _ in range(T)]
    for t in range(T):
        m = max(float(v) for v in logits[t])
        ex = [math.exp(float(v) - m) for v in logits[t]]
        p[t] = [v / sum(ex) for v in ex]
    x, W1, b1, W2, b2 = (L[n] for n in ("x", "W1", "b1", "W2", "b2"))
    want = np.zeros_like(r.y)
    for e in range(E):
        chosen = sorted(range(T), key=lambda t: (-p[t][e], t))[:8]
        for tok in chosen:
            h = [0.5 * u * (1 + math.erf(u / math.sqrt(2)))
                 for u in (b1[e, f] + sum(W1[e, f, j] * x[tok, j] for j in range(4))
                           for f in range(5))]
            for i in range(4):
                want[tok, i] += p[tok][e] * (b2[e, i] + sum(W2[e, i, f] * h[f] for f in range(5)))
    np.testing.assert_allclose(r.y, want, rtol=1e-12, atol=1e-12)
    # a token outside every expert's choice gets zero; counts per expert are C
    assert (r.slot_of >= 0).sum(axis=0).tolist() == [8, 8, 8]


def test_expert_choice_token_subset_and_given_selection():
    """Restricting output rows or passing the oracle's own selection back
    changes nothing."""
    L = _rand_layer(T=20, d=6, F=8, E=4, seed=46)
    a = O.expert_choice_forward(**L, k=2, capacity=7)
    b = O.expert_choice_forward(**L, k=2, capacity=7, tokens=[19, 3, 8])
    np.testing.assert_allclose(b.y, a.y[[19, 3, 8]], rtol=1e-12, atol=1e-14)
    c = O.expert_choice_forward(**L, k=2, capacity=7, sel=a.sel)
    np.testing.assert_array_equal(c.y, a.y)


def test_planted_expert_choice_mistakes_are_caught(monkeypatch):
    """Plausible expert-choice mistakes, planted on the CPU, fail a pin."""
    good = O.expert_choice_select

    def ties_to_higher(p, C):  # equal probabilities: the higher token first
        p = np.asarray(p)
        T, E = p.shape
        return np.array([np.sort(np.lexsort((-np.arange(T), -p[:, e]))[:C]) for e in range(E)])
    monkeypatch.setattr(O, "expert_choice_select", ties_to_higher)
    with pytest.raises(AssertionError):
        test_expert_choice_ties_go_to_lower_token()

    def by_logit_rank_per_token(p, C):  # top-C of the token-wise rank instead of p
        p = np.asarray(p)
        r = np.argsort(np.argsort(-p, axis=1), axis=1).astype(float)
        return good(-r + 1e-9 * p, C)
    monkeypatch.setattr(O, "expert_choice_select", by_logit_rank_per_token)
    with pytest.raises(AssertionError):
        test_expert_choice_brute_force_selection()
    monkeypatch.setattr(O, "expert_choice_select", good)

    good_cap = O.expert_choice_capacity
    monkeypatch.setattr(O, "expert_choice_capacity",
                        lambda T, E, k, capacity=None: good_cap(T, E, 1, capacity))  # k ignored
    with pytest.raises(AssertionError):
        test_expert_choice_all_tokens_is_soft_mixture()


# ---- rerouting on overflow (overflow sent to the next-ranked expert); the reading
# (one hop, offers after the drop pass, in token order) is in the oracle's header

def test_reroute_hand_worked():
    """Capacity 1, three experts, four tokens that all prefer expert 0, with
    second choices 1, 1, 2, 1.  Drop pass: token 0 keeps expert 0, tokens
    1-3 are dropped.  Offers in token order: token 1 -> expert 1 (room),
    token 2 -> expert 2 (room), token 3 -> expert 1 (full: dropped).
    Rows: expert 0 [t0], expert 1 [t1], expert 2 [t2]."""
    ranked = np.array([[0, 1], [0, 1], [0, 2], [0, 1]])
    final, phase = O.reroute_keep(ranked, 1, 3, 1)
    assert final[:, 0].tolist() == [0, 1, 2, -1]
    assert phase[:, 0].tolist() == [1, 2, 2, 0]
    offsets, slot_of, perm_token = O.reroute_layout(final, phase, 3)
    assert offsets.tolist() == [0, 1, 2, 3]
    assert slot_of[:, 0].tolist() == [0, 1, 2, -1]
    assert perm_token.tolist() == [0, 1, 2]


def test_reroute_two_slot_order_and_rows():
    """k = 2, capacity 2, E = 4.  Token choices (best first, then next-best):
    t0 (0,1 | 2,3), t1 (0,1 | 3,2), t2 (0,1 | 2,3), t3 (1,0 | 2,3).
    Drop pass keeps t0 and t1 on experts 0 and 1 and drops all of t2, t3.
    Offers: t2 slot 0 -> its 3rd expert 2 (ok), t2 slot 1 -> its 4th expert 3
    (ok), t3 slot 0 -> 2 (ok: 2 is at 1 of 2), t3 slot 1 -> 3 (ok).  Expert 2
    rows [t2, t3] and expert 3 rows [t2, t3], all after the (empty) drop-pass
    rows."""
    ranked = np.array([[0, 1, 2, 3], [0, 1, 3, 2], [0, 1, 2, 3], [1, 0, 2, 3]])
    final, phase = O.reroute_keep(ranked, 2, 4, 2)
    assert final.tolist() == [[0, 1], [0, 1], [2, 3], [2, 3]]
    assert phase.tolist() == [[1, 1], [1, 1], [2, 2], [2, 2]]
    offsets, slot_of, perm_token = O.reroute_layout(final, phase, 4)
    assert offsets.tolist() == [0, 2, 4, 6, 8]
    assert perm_token.tolist() == [0, 1, 0, 1, 2, 3, 2, 3]
    assert slot_of.tolist() == [[0, 2], [1, 3], [4, 6], [5, 7]]


@pytest.mark.parametrize("n0,C", [(700, 400), (300, 400), (900, 300), (1000, 1000), (500, 0)])
def test_reroute_two_experts_closed_form(n0, C):
    """Top-1 over two experts, n0 of 1000 tokens prefer expert 0: the drop
    pass keeps min(n0, C) and min(n1, C); each expert then accepts the other's
    overflow up to its spare room, so the kept totals are
    min(n0, C) + min(n1 - min(n1, C), C - min(n0, C)) on expert 0 and the
    mirror on expert 1."""
    T = 1000
    rng = np.random.default_rng(n0 + C)
    first = np.zeros(T, np.int64)
    first[rng.permutation(T)[:T - n0]] = 1
    ranked = np.stack([first, 1 - first], axis=1)
    final, _ = O.reroute_keep(ranked, 1, 2, C)
    n1 = T - n0
    k0, k1 = min(n0, C), min(n1, C)
    want0 = k0 + min(n1 - k1, C - k0)
    want1 = k1 + min(n0 - k0, C - k1)
    assert int(np.sum(final == 0)) == want0 and int(np.sum(final == 1)) == want1
    # invariants: a moved token went to its other expert, none exceeds C
    assert np.all((final[:, 0] == -1) | (final[:, 0] == first) | (final[:, 0] == 1 - first))


def test_reroute_invariants_random():
    """Random rankings: the drop pass is capacity_keep's, no expert exceeds
    the cap, a moved slot lands on the token's (k + r)-th expert, and an offer
    is refused only when its expert was full at that point in token order."""
    rng = np.random.default_rng(47)
    for T, E, k, C in ((40, 5, 2, 6), (60, 8, 1, 5), (30, 4, 2, 3), (25, 6, 3, 4)):
        ranked = np.array([rng.permutation(E)[:min(2 * k, E)] for _ in range(T)])
        final, phase = O.reroute_keep(ranked, k, E, C)
        kept1 = O.capacity_keep(ranked[:, :k], E, C)
        assert np.array_equal(phase == 1, kept1)
        assert np.all(np.bincount(final[final >= 0], minlength=E) <= C)
        load = np.bincount(ranked[:, :k][kept1], minlength=E)
        for t in range(T):
            r = 0
            for j in range(k):
                if kept1[t, j]:
                    continue
                if k + r < ranked.shape[1]:
                    e = ranked[t, k + r]
                    if phase[t, j] == 2:
                        assert final[t, j] == e and load[e] < C
                        load[e] += 1
                    else:
                        assert final[t, j] == -1 and load[e] >= C
                r += 1


def test_reroute_forward():
    """No cap or a cap >= T: rerouting changes nothing.  With a cap: the
    moved slot carries the new expert's renormalised probability, the layer
    equals the dense masked evaluation with those gates (torch, fp64), and
    it keeps at least as many assignments as dropping."""
    L = _rand_layer(T=24, d=6, F=8, E=4, seed=48)
    a = O.moe_forward(**L, k=2)
    b = O.moe_forward(**L, k=2, capacity=24, reroute=True)
    assert np.array_equal(a.y, b.y) and np.array_equal(a.slot_of, b.slot_of)
    bias = np.array([2.0, 0.0, 0.0, -1.0], np.float32)  # expert 0 overflows, 3 has room
    r = O.moe_forward(**L, k=2, capacity=14, reroute=True, logit_bias=bias)
    d = O.moe_forward(**L, k=2, capacity=14, logit_bias=bias)
    assert r.kept.sum() > d.kept.sum()
    assert np.array_equal(r.counts, d.counts)  # counts are the k choices'
    p = r.probs
    top = O.top_k(r.logits, 2)
    den = np.take_along_axis(p, top, 1).sum(1)
    t = {n: torch.from_numpy(v) for n, v in L.items()}
    want = np.zeros_like(r.y)
    for tok in range(24):
        for j in range(2):
            if not r.kept[tok, j]:
                continue
            e = int(r.idx[tok, j])
            assert abs(r.w[tok, j] - p[tok, e] / den[tok]) <= 1e-15
            fe = TF.linear(TF.gelu(TF.linear(t["x"][tok], t["W1"][e], t["b1"][e])), t["W2"][e],
                           t["b2"][e]).numpy()
            want[tok] += r.w[tok, j] * fe
    np.testing.assert_allclose(r.y, want, rtol=1e-12, atol=1e-14)
    # the moved slots are exactly the dropped slots whose next-best had room
    moved = r.kept & ~d.kept
    assert moved.sum() > 0 and np.all(r.idx[moved] != top[moved])


def test_planted_reroute_mistakes_are_caught(monkeypatch):
    """Offers that ignore the drop pass's load, or that go to the token's
    (k+1)-th expert for every dropped slot, fail a reroute pin."""
    good = O.reroute_keep

    def fresh_load(ranked, k, E, capacity):  # room counted from zero, not after the drop pass
        ranked = np.asarray(ranked)
        final, phase = good(ranked, k, E, capacity)
        kept = O.capacity_keep(ranked[:, :k], E, capacity)
        load = np.zeros(E, np.int64)
        for t in range(ranked.shape[0]):
            r = 0
            for j in range(k):
                if kept[t, j]:
                    continue
                if k + r < ranked.shape[1] and load[ranked[t, k + r]] < capacity:
                    load[ranked[t, k + r]] += 1
                    final[t, j], phase[t, j] = ranked[t, k + r], 2
                r += 1
        return final, phase
    monkeypatch.setattr(O, "reroute_keep", fresh_load)
    with pytest.raises(AssertionError):
        test_reroute_two_experts_closed_form(700, 400)
    monkeypatch.setattr(O, "reroute_keep", good)

    def same_alternate(ranked, k, E, capacity):  # every dropped slot offered to rank k
        ranked = np.array(ranked)
        ranked[:, k + 1:] = ranked[:, k:k + 1]
        return good(ranked, k, E, capacity)
    monkeypatch.setattr(O, "reroute_keep", same_alternate)
    with pytest.raises(AssertionError):
        test_reroute_two_slot_order_and_rows()


# ---- backward pass: the oracle's hand-derived gradients against torch
# autograd of the same layer (routing decisions held fixed), and against
# central finite differences

def _torch_loss(L, dy, k, renorm, cap, aux_grad, z_grad, bias=None):
    """<dy, y> + aux_grad aux + z_grad z in torch fp64, the routing (top-k and
    capacity keep) taken from the oracle as constants; the fp32 rounding of
    the oracle's logits is added as a constant so the values match."""
    r = O.moe_forward(**L, k=k, renormalize=renorm, capacity=cap, logit_bias=bias)
    t = {n: torch.tensor(np.asarray(v, np.float64), requires_grad=True) for n, v in L.items()}
    g64 = t["x"] @ t["W_r"].T
    if bias is not None:
        g64 = g64 + torch.tensor(np.asarray(bias, np.float64))
    g = g64 + (torch.tensor(r.logits.astype(np.float64)) - g64).detach()
    p = torch.softmax(g, dim=1)
    idx = torch.tensor(r.idx, dtype=torch.int64)
    sel = p.gather(1, idx)
    w = sel / sel.sum(1, keepdim=True) if renorm else sel
    T, E = g.shape
    ys = []
    for tok in range(T):
        yt = torch.zeros(t["x"].shape[1], dtype=torch.float64)
        for j in range(k):
            if r.kept[tok, j]:
                e = int(r.idx[tok, j])
                h = TF.gelu(t["W1"][e] @ t["x"][tok] + t["b1"][e])
                yt = yt + w[tok, j] * (t["W2"][e] @ h + t["b2"][e])
        ys.append(yt)
    y = torch.stack(ys)
    f = torch.tensor(np.bincount(r.idx[:, 0], minlength=E) / T)
    aux = E * (f * p.mean(0)).sum()
    z = torch.logsumexp(g, dim=1).pow(2).mean()
    loss = (torch.tensor(dy) * y).sum() + aux_grad * aux + z_grad * z
    loss.backward()
    return {n: t[n].grad.numpy() for n in t}, float(loss.detach())


@pytest.mark.parametrize("k,renorm,cap,aux_grad,z_grad", [
    (2, True, None, 0.0, 0.0), (1, False, None, 0.0, 0.0), (2, True, 3, 0.3, 0.0),
    (1, False, 4, 0.01, 0.5), (3, True, None, 1.0, 1.0), (2, False, 2, 0.0, 2.0)])
def test_backward_matches_torch_autograd(k, renorm, cap, aux_grad, z_grad):
    L = _rand_layer(T=11, d=6, F=7, E=4, seed=50 + k)
    dy = np.random.default_rng(51).standard_normal((11, 6))
    want, _ = _torch_loss(L, dy, k, renorm, cap, aux_grad, z_grad)
    got = O.moe_backward(**L, dy=dy, k=k, renormalize=renorm, capacity=cap, aux_grad=aux_grad,
                         z_grad=z_grad)
    for n, gname in (("x", "dx"), ("W_r", "dW_r"), ("W1", "dW1"), ("b1", "db1"), ("W2", "dW2"),
                     ("b2", "db2")):
        np.testing.assert_allclose(got[gname], want[n], rtol=1e-10, atol=1e-12, err_msg=gname)


def test_backward_with_logit_bias_and_dense_expert():
    """A logit bias shifts the routing but not the formulas; E = 1 is the
    plain FFN's backward."""
    L = _rand_layer(T=9, d=5, F=6, E=3, seed=52)
    dy = np.random.default_rng(53).standard_normal((9, 5))
    bias = np.array([0.4, -0.2, 0.0], np.float32)
    want, _ = _torch_loss(L, dy, 2, True, 4, 0.2, 0.1, bias=bias)
    got = O.moe_backward(**L, dy=dy, k=2, renormalize=True, capacity=4, logit_bias=bias,
                         aux_grad=0.2, z_grad=0.1)
    np.testing.assert_allclose(got["dx"], want["x"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got["dW_r"], want["W_r"], rtol=1e-10, atol=1e-12)
    L1 = _rand_layer(T=7, d=4, F=5, E=1, seed=54)
    dy1 = np.random.default_rng(55).standard_normal((7, 4))
    got1 = O.moe_backward(**L1, dy=dy1, k=1, renormalize=True)
    t = {n: torch.tensor(np.asarray(v, np.float64), requires_grad=True) for n, v in L1.items()}
    y = TF.linear(TF.gelu(TF.linear(t["x"], t["W1"][0], t["b1"][0])), t["W2"][0], t["b2"][0])
    (torch.tensor(dy1) * y).sum().backward()
    np.testing.assert_allclose(got1["dW1"][0], t["W1"].grad[0].numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(got1["dx"], t["x"].grad.numpy(), rtol=1e-10, atol=1e-13)
    assert not got1["dW_r"].any()  # one expert: w = 1 whatever the logit


def test_backward_finite_differences():
    """Central differences of the loss in x, W1, W_r and b2 (steps small
    enough to keep the routing, large enough that the fp32 rounding of the
    logits stays below the tolerance) agree with the oracle's gradients."""
    L = _rand_layer(T=6, d=4, F=5, E=3, seed=56)
    dy = np.random.default_rng(57).standard_normal((6, 4))
    kw = dict(k=2, renormalize=True, capacity=None)
    got = O.moe_backward(**L, dy=dy, aux_grad=0.5, z_grad=0.25, **kw)

    def loss(LL):
        r = O.moe_forward(**LL, **kw)
        f = np.bincount(r.idx[:, 0], minlength=3) / 6
        return float((dy * r.y).sum() + 0.5 * 3 * (f * r.probs.mean(0)).sum()
                     + 0.25 * r.z_loss)

    base = O.moe_forward(**L, **kw)
    eps = 1e-3
    for name, gname, pos in (("x", "dx", (2, 1)), ("W1", "dW1", (1, 3, 2)), ("W_r", "dW_r", (0, 3)),
                             ("b2", "db2", (2, 0))):
        a = {n: np.array(v, np.float64) for n, v in L.items()}
        b = {n: np.array(v, np.float64) for n, v in L.items()}
        a[name][pos] += eps
        b[name][pos] -= eps
        for LL in (a, b):  # the steps keep every routing decision
            assert np.array_equal(O.moe_forward(**LL, **kw).idx, base.idx)
        fd = (loss(a) - loss(b)) / (2 * eps)
        assert abs(fd - got[gname][pos]) <= 5e-5 * max(1.0, abs(fd)), (name, fd, got[gname][pos])


def test_planted_backward_mistakes_are_caught(monkeypatch):
    """A GELU derivative without its u phi(u) term fails the autograd pin."""
    good = O.gelu_grad
    monkeypatch.setattr(O, "gelu_grad", lambda u: 0.5 * (1.0 + O.erf(np.asarray(u) / math.sqrt(2))))
    with pytest.raises(AssertionError):
        test_backward_matches_torch_autograd(2, True, None, 0.0, 0.0)
    monkeypatch.setattr(O, "gelu_grad", good)


# ---- backward of the layer variants: shared experts, rerouting on overflow,
# expert choice; each against torch autograd of the same layer with its
# routing decisions held fixed (the oracle's fp32 logit rounding added as a
# constant, as in _torch_loss)

def _torch_router(t, r_logits, bias=None):
    g64 = t["x"] @ t["W_r"].T
    if bias is not None:
        g64 = g64 + torch.tensor(np.asarray(bias, np.float64))
    return g64 + (torch.tensor(r_logits.astype(np.float64)) - g64).detach()


def _torch_variant_loss(L, dy, k, renorm, cap, aux_grad, z_grad, n_shared=0, reroute=False,
                        bias=None):
    """The layer in torch: routed slot j of token t has final expert f_j (the
    oracle's decision, held fixed) and weight p_{f_j} / sum over the token's
    k choices of p (renormalised) or p_{f_j}; shared experts weight 1."""
    r = O.moe_forward(**L, k=k, renormalize=renorm, capacity=cap, n_shared=n_shared,
                      reroute=reroute, logit_bias=bias)
    t = {n: torch.tensor(np.asarray(v, np.float64), requires_grad=True) for n, v in L.items()}
    g = _torch_router(t, r.logits, bias)
    p = torch.softmax(g, dim=1)
    choices = torch.tensor(O.top_k(r.logits, k), dtype=torch.int64)
    S = p.gather(1, choices).sum(1) if renorm else torch.ones(g.shape[0], dtype=torch.float64)
    T = g.shape[0]
    ys = []
    for tok in range(T):
        yt = torch.zeros(t["x"].shape[1], dtype=torch.float64)
        for j in range(r.idx.shape[1]):
            if not r.kept[tok, j]:
                continue
            e = int(r.idx[tok, j])
            w = 1.0 if j >= k else p[tok, e - n_shared] / S[tok]
            h = TF.gelu(t["W1"][e] @ t["x"][tok] + t["b1"][e])
            yt = yt + w * (t["W2"][e] @ h + t["b2"][e])
        ys.append(yt)
    y = torch.stack(ys)
    assert np.allclose(y.detach().numpy(), r.y, rtol=1e-12, atol=1e-12)  # the oracle's forward
    E_r = g.shape[1]
    f = torch.tensor(np.bincount(O.top_k(r.logits, k)[:, 0], minlength=E_r) / T)
    aux = E_r * (f * p.mean(0)).sum()
    z = torch.logsumexp(g, dim=1).pow(2).mean()
    loss = (torch.tensor(dy) * y).sum() + aux_grad * aux + z_grad * z
    loss.backward()
    return {n: t[n].grad.numpy() for n in t}


_GRADS = (("x", "dx"), ("W_r", "dW_r"), ("W1", "dW1"), ("b1", "db1"), ("W2", "dW2"), ("b2", "db2"))


@pytest.mark.parametrize("k,renorm,cap,aux_grad,z_grad,ns", [
    (2, True, None, 0.0, 0.0, 1), (1, False, None, 0.2, 0.0, 1), (2, True, 3, 0.3, 0.4, 2),
    (1, True, 2, 0.0, 1.0, 1)])
def test_backward_shared_experts_matches_torch_autograd(k, renorm, cap, aux_grad, z_grad, ns):
    E = 5
    L = _rand_layer(T=12, d=6, F=7, E=E, seed=60 + ns)
    L["W_r"] = L["W_r"][: E - ns]  # the router covers the routed experts
    dy = np.random.default_rng(61).standard_normal((12, 6))
    want = _torch_variant_loss(L, dy, k, renorm, cap, aux_grad, z_grad, n_shared=ns)
    got = O.moe_backward(**L, dy=dy, k=k, renormalize=renorm, capacity=cap, aux_grad=aux_grad,
                         z_grad=z_grad, n_shared=ns)
    for n, gname in _GRADS:
        np.testing.assert_allclose(got[gname], want[n], rtol=1e-10, atol=1e-12, err_msg=gname)
    assert got["dW_r"].shape == (E - ns, 6)
    # the shared experts see every token
    assert np.all(np.abs(got["db2"][:ns]).sum(axis=1) > 0)


@pytest.mark.parametrize("k,renorm,cap,aux_grad,z_grad", [
    (1, False, 3, 0.0, 0.0), (2, True, 4, 0.0, 0.0), (2, True, 3, 0.5, 0.3), (1, True, 2, 0.1, 0.0),
    (2, False, 4, 0.0, 0.2)])
def test_backward_reroute_matches_torch_autograd(k, renorm, cap, aux_grad, z_grad):
    L = _rand_layer(T=12, d=5, F=6, E=6, seed=70 + k)
    bias = np.array([1.5, 1.0, 0.2, -0.5, -1.0, -1.5], np.float32)  # skewed load: overflow
    dy = np.random.default_rng(71).standard_normal((12, 5))
    r = O.moe_forward(**L, k=k, renormalize=renorm, capacity=cap, reroute=True, logit_bias=bias)
    moved = r.kept & (r.idx != O.top_k(r.logits, k))
    assert moved.any()  # the cap moves some slots to their next-best expert
    want = _torch_variant_loss(L, dy, k, renorm, cap, aux_grad, z_grad, reroute=True, bias=bias)
    got = O.moe_backward(**L, dy=dy, k=k, renormalize=renorm, capacity=cap, aux_grad=aux_grad,
                         z_grad=z_grad, reroute=True, logit_bias=bias)
    for n, gname in _GRADS:
        np.testing.assert_allclose(got[gname], want[n], rtol=1e-10, atol=1e-12, err_msg=gname)


def test_backward_reroute_without_moves_equals_drop():
    """No slot moves (a cap no expert reaches): rerouting's gradients are the
    dropping layer's."""
    L = _rand_layer(T=8, d=4, F=5, E=4, seed=75)
    dy = np.random.default_rng(76).standard_normal((8, 4))
    a = O.moe_backward(**L, dy=dy, k=2, capacity=8, reroute=True, aux_grad=0.2)
    b = O.moe_backward(**L, dy=dy, k=2, capacity=8, reroute=False, aux_grad=0.2)
    for _, gname in _GRADS:
        np.testing.assert_array_equal(a[gname], b[gname])


def _torch_ec_loss(L, dy, k, cap, z_grad):
    r = O.expert_choice_forward(**L, k=k, capacity=cap)
    t = {n: torch.tensor(np.asarray(v, np.float64), requires_grad=True) for n, v in L.items()}
    g = _torch_router(t, r.logits)
    p = torch.softmax(g, dim=1)
    T, E = g.shape
    rows = [[] for _ in range(T)]
    for e in range(E):
        for j in range(r.C):
            rows[int(r.sel[e, j])].append(e)
    ys = []
    for tok in range(T):
        yt = torch.zeros(t["x"].shape[1], dtype=torch.float64)
        for e in rows[tok]:
            h = TF.gelu(t["W1"][e] @ t["x"][tok] + t["b1"][e])
            yt = yt + p[tok, e] * (t["W2"][e] @ h + t["b2"][e])
        ys.append(yt)
    y = torch.stack(ys)
    assert np.allclose(y.detach().numpy(), r.y, rtol=1e-12, atol=1e-12)
    z = torch.logsumexp(g, dim=1).pow(2).mean()
    ((torch.tensor(dy) * y).sum() + z_grad * z).backward()
    return {n: t[n].grad.numpy() for n in t}


@pytest.mark.parametrize("k,cap,z_grad", [(2, None, 0.0), (1, 3, 0.5), (2, 9, 0.0), (3, None, 1.0)])
def test_backward_expert_choice_matches_torch_autograd(k, cap, z_grad):
    L = _rand_layer(T=9, d=5, F=6, E=4, seed=80 + k)
    dy = np.random.default_rng(81).standard_normal((9, 5))
    want = _torch_ec_loss(L, dy, k, cap, z_grad)
    got = O.expert_choice_backward(**L, dy=dy, k=k, capacity=cap, z_grad=z_grad)
    for n, gname in _GRADS:
        np.testing.assert_allclose(got[gname], want[n], rtol=1e-10, atol=1e-12, err_msg=gname)


def test_backward_expert_choice_every_token_is_the_soft_mixture():
    """C = T: every expert takes every token, y = sum_e p_e f_e(x), whose
    router gradient is the softmax's: dg = s - p sum s (finite differences in
    W_r agree)."""
    L = _rand_layer(T=5, d=4, F=5, E=3, seed=85)
    dy = np.random.default_rng(86).standard_normal((5, 4))
    got = O.expert_choice_backward(**L, dy=dy, k=3, capacity=5)
    eps = 1e-3
    for pos in ((0, 1), (2, 3)):
        a = {n: np.array(v, np.float64) for n, v in L.items()}
        b = {n: np.array(v, np.float64) for n, v in L.items()}
        a["W_r"][pos] += eps
        b["W_r"][pos] -= eps
        la = float((dy * O.expert_choice_forward(**a, k=3, capacity=5).y).sum())
        lb = float((dy * O.expert_choice_forward(**b, k=3, capacity=5).y).sum())
        fd = (la - lb) / (2 * eps)
        assert abs(fd - got["dW_r"][pos]) <= 5e-5 * max(1.0, abs(fd)), (pos, fd, got["dW_r"][pos])


def test_planted_variant_backward_mistakes_are_caught(monkeypatch):
    """Planted in the oracle's forward (which its backward differentiates): a
    rerouted slot keeping the weight of the choice it was dropped from, and
    shared experts weighted by 1/2 instead of 1 - each fails its autograd pin."""
    good = O.moe_forward

    def wrong_reroute_weight(*a, **kw):
        r = good(*a, **kw)
        if kw.get("reroute"):
            ch = O.top_k(r.logits, kw["k"])
            p = np.take_along_axis(r.probs, ch, axis=1)
            S = p.sum(axis=1, keepdims=True) if kw.get("renormalize", True) else 1.0
            moved = r.kept & (r.idx != ch)
            r.w = np.where(moved, p / S, r.w)
        return r

    monkeypatch.setattr(O, "moe_forward", wrong_reroute_weight)
    with pytest.raises(AssertionError):
        test_backward_reroute_matches_torch_autograd(2, True, 4, 0.0, 0.0)

    def wrong_shared_weight(*a, **kw):
        r = good(*a, **kw)
        if kw.get("n_shared"):
            r.w = r.w.copy()
            r.w[:, kw["k"]:] = 0.5
        return r

    monkeypatch.setattr(O, "moe_forward", wrong_shared_weight)
    with pytest.raises(AssertionError):
        test_backward_shared_experts_matches_torch_autograd(2, True, None, 0.0, 0.0, 1)
    monkeypatch.setattr(O, "moe_forward", good)
