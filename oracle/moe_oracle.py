"""CPU oracle of the sparsely-gated Mixture-of-Experts FFN layer forward pass.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the layer computes.  Only the test-suite, the package smoke
check and the benchmark's CPU-baseline leg may import it; the product path
never does.  It shares no code with the CUDA path.

Arithmetic is fp64 (numpy), on stored inputs widened exactly.  Each function
cites the passage it follows.  Page titles used in citations:

* [LECTURE]  "Mixture of Experts: Scaling Parameters Without Scaling Compute"
* [DAY59]    "Mixture-of-Experts -- making a model wider without using all of
             it for every token"
* [RATISH]   "Mixture of Experts" (learn.ratishfolio.com)
* [GLOSSARY] "Mixture of Experts (MoE)" (inferensys glossary)
* [AIINBED]  "Mixture of experts: big models, small bills"

Readings taken where the pages are silent or garbled (the display formulas of
the combine and of the auxiliary loss did not survive extraction):

* routing decisions are taken on the fp32 router logits (softmax is
  monotone), ties going to the lower expert index;
* k >= 2 weights are renormalised over the selected experts; with
  ``renormalize=False`` (Switch top-1) the weight is the router probability;
* the capacity cap keeps, per expert, the first ``capacity`` assignments in
  (token, slot) ascending order; a dropped assignment contributes 0 (the
  residual add is outside the layer) and surviving weights are not
  renormalised again;
* f_i of the auxiliary loss counts the top-1 choice only, before any drop;
* the router z-loss, which the pages name without a formula (a penalty that
  keeps the router logits small), is the mean over tokens of the squared log-sum-exp of the
  token's router logits (the logits that enter the softmax, bias included);
* noisy gating adds a caller-drawn (T, E) noise tensor to the router logits
  before the softmax and the top-k (the pages give no distribution; the
  caller chooses it);
* auxiliary-loss-free balancing moves the per-expert logit bias by a fixed
  step toward balanced load after a batch: minus the step for an expert
  above the mean assignment count, plus it below, unchanged at the mean;
* rerouting on overflow (an overflowing token goes to its next-ranked
  expert instead of being dropped) is one hop: after
  the drop pass above, the r-th dropped slot of a token (r = 0, 1, ...) is
  offered to the token's (k + r)-th ranked expert (the best one it does not
  use); offers are visited in (token, slot) order and an expert accepts them
  while its kept assignments plus accepted offers stay below the capacity;
  a refused offer is dropped.  The slot's weight becomes the new expert's
  probability, with the same normalisation as the token's other weights
  (divided by the sum over its k choices when renormalising).  An expert's
  rows are its first-pass assignments in token order, then the offers it
  accepted in token order;
* the backward pass (gradients of the layer, which the pages name as part
  of training) treats the routing decisions (top-k, capacity) as constants,
  as autograd does: the loss is <dy, y> + aux_grad * aux + z_grad * z_loss
  for caller-given dy and scalar weights; the gate weights carry gradient to
  the logits through the softmax (and the renormalisation), the auxiliary
  loss through P (f holds counts) and the z-loss through the log-sum-exp;
* expert-choice routing (the experts, not the tokens, do the selecting)
  ranks, for each
  expert, the batch's tokens by their router probability p[t, e] (the same
  softmax over experts as token choice), larger first and the lower token
  index first among equals, and keeps the first C; C is the capacity when one
  is given, else ceil(T k / E) (the average load top-k token choice would
  put on an expert), at most T.  A token's output is the sum, over the
  experts that chose it, of p[t, e] times the expert's output (no
  renormalisation); a token no expert chose gets 0.  Balance holds by
  construction, so no balancing loss is defined (reported as 0).

Parity: the routing, capacity, auxiliary-loss and combine functions are pinned
by the pages' worked examples, closed forms and brute force (tests).  The
full-layer numeric output is pinned by invariants and by special cases that
reduce to library routines, not by any printed value: the pages print no layer
output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
from scipy.special import erf

f64 = np.float64


def router_logits(x, W_r, logit_bias=None, logit_noise=None) -> np.ndarray:
    """g = W_r x (+ per-expert bias) (+ per-token noise), computed in fp64 and
    rounded to fp32.

    [LECTURE] "The MoE layer", step 1 (router logits, an ``nn.Linear`` with no
    bias in its listing).  The optional additive per-expert bias is the fixed
    logit offset of the Switch workload (the mechanism [LECTURE] "The central
    problem: load balancing" names for bias-based balancing).  The optional
    (T, E) noise is noisy gating ("The central problem: load balancing":
    random perturbation of the router's logits while training, so that it
    explores); the caller draws it.
    x: (T, d); W_r: (E, d); returns (T, E) fp32.
    """
    g = np.asarray(x, f64) @ np.asarray(W_r, f64).T
    if logit_bias is not None:
        g = g + np.asarray(logit_bias, f64)[None, :]
    if logit_noise is not None:
        g = g + np.asarray(logit_noise, f64)
    return g.astype(np.float32)


def softmax(logits) -> np.ndarray:
    """p = softmax(g) over experts, fp64, max-subtracted.

    [LECTURE] "The MoE layer", step 1; [AIINBED] "Experts and the router".
    """
    g = np.asarray(logits, f64)
    z = np.exp(g - g.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def top_k(logits, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, largest first.

    [LECTURE] "The MoE layer", step 2; [DAY59] "Replace one MLP with many
    experts" (top-2 example).  Equal logits: the lower expert index comes
    first (a stable descending sort, as the router demo of [AIINBED] does).
    Returns (T, k) int32.
    """
    g = np.asarray(logits)
    order = np.argsort(-g, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gate_weights(probs, idx, renormalize: bool) -> np.ndarray:
    """Weights of the selected experts: p_sel / sum(p_sel), or p_sel as is.

    [LECTURE] "The MoE layer" (the chosen experts' probabilities, usually
    rescaled to sum to one);
    [DAY59] "Replace one MLP with many experts".  Returns (T, k) fp64.
    """
    sel = np.take_along_axis(np.asarray(probs, f64), np.asarray(idx, np.int64), axis=1)
    if renormalize:
        return sel / sel.sum(axis=1, keepdims=True)
    return sel


def expert_capacity(capacity_factor: float, T: int, E: int) -> int:
    """C = ceil(capacity_factor * T / E).

    [LECTURE] "The central problem: load balancing" (the capacity factor
    scales each expert's even share of the tokens); rounding up is the
    reading taken (the display formula of
    [DAY59] "Experts also have capacity limits" is lost).
    """
    return int(math.ceil(capacity_factor * T / E))


def capacity_keep(idx, E: int, capacity: int | None, n_shared: int = 0) -> np.ndarray:
    """Which assignments survive the per-expert capacity cap.

    [LECTURE] "The central problem: load balancing" (overflow tokens are
    dropped); [GLOSSARY] expert capacity.  Assignments are visited in token
    order, then slot order; each expert keeps its first ``capacity``.
    ``capacity=None`` keeps everything.  Shared experts (ids below
    ``n_shared``, always active) are not capped.  Returns (T, k) bool.
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    kept = np.ones((T, k), dtype=bool)
    if capacity is None:
        return kept
    taken = [0] * E
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if e < n_shared:
                continue
            if taken[e] < capacity:
                taken[e] += 1
            else:
                kept[t, j] = False
    return kept


def reroute_keep(ranked, k: int, E: int, capacity: int | None):
    """Drop, then offer each dropped slot once to the token's next-best expert.

    [LECTURE] "The central problem: load balancing" (an overflowing token is
    either dropped or sent elsewhere); [GLOSSARY] expert capacity (one option
    sends it to its next-ranked expert).  ``ranked`` (T, K2) lists each token's experts best
    first, its k choices then the next K2 - k.  First pass: ``capacity_keep``
    on the k choices.  Second pass: the r-th dropped slot of token t is
    offered to ranked[t, k + r] (when k + r < K2); offers in (token, slot)
    order; expert e accepts while first-pass keeps + accepted offers <
    capacity.  Returns final (T, k) expert ids (-1: dropped) and the pass
    (T, k) that placed each slot (1, 2; 0 if dropped).
    """
    ranked = np.asarray(ranked)
    T, K2 = ranked.shape
    first = ranked[:, :k]
    kept = capacity_keep(first, E, capacity)
    final = np.where(kept, first, -1).astype(np.int64)
    phase = kept.astype(np.int64)
    if capacity is None:
        return final, phase
    load = np.bincount(first[kept].astype(np.int64), minlength=E)
    for t in range(T):
        r = 0
        for j in range(k):
            if kept[t, j]:
                continue
            if k + r < K2:
                e = int(ranked[t, k + r])
                if load[e] < capacity:
                    load[e] += 1
                    final[t, j] = e
                    phase[t, j] = 2
            r += 1
    return final, phase


def reroute_layout(final, phase, E: int):
    """Rows of a rerouted batch: per expert, its first-pass slots in token
    order, then the offers it accepted in token order.  Returns offsets
    (E+1,), slot_of (T, k) and perm_token (n_kept,)."""
    final, phase = np.asarray(final), np.asarray(phase)
    T, k = final.shape
    offsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + int(np.sum(final == e))
    slot_of = np.full((T, k), -1, np.int64)
    perm_token = np.zeros(int(offsets[E]), np.int64)
    for e in range(E):
        pos = int(offsets[e])
        for ph in (1, 2):
            for t in range(T):
                for j in range(k):
                    if final[t, j] == e and phase[t, j] == ph:
                        slot_of[t, j] = pos
                        perm_token[pos] = t
                        pos += 1
    return offsets, slot_of, perm_token


def gelu(u) -> np.ndarray:
    """Exact GELU, 0.5 u (1 + erf(u / sqrt 2)) (``nn.GELU()`` default).

    [LECTURE] "The MoE layer" (each expert is Linear, GELU, Linear).
    """
    u = np.asarray(u, f64)
    return 0.5 * u * (1.0 + erf(u / math.sqrt(2.0)))


def expert_ffn(X, W1e, b1e, W2e, b2e) -> np.ndarray:
    """One expert: Linear(d, F) + bias, GELU, Linear(F, d) + bias, in fp64.

    [LECTURE] "The MoE layer" (expert definition); [DAY59] "Replace one MLP
    with many experts" (each expert is an ordinary feed-forward network).
    X: (n, d); W1e: (F, d); b1e: (F,); W2e: (d, F); b2e: (d,).
    """
    U = np.asarray(X, f64) @ np.asarray(W1e, f64).T + np.asarray(b1e, f64)[None, :]
    H = gelu(U)
    return H @ np.asarray(W2e, f64).T + np.asarray(b2e, f64)[None, :]


def aux_loss(probs, idx, E: int) -> float:
    """Switch load-balancing loss E * sum_i f_i P_i.

    [LECTURE] "The central problem: load balancing" (f_i = fraction of tokens
    routed to expert i, P_i = mean router probability) and the loss lines of
    its listing (f from the top-1 choice, P = mean of the softmax); [DAY59]
    "Load-balancing losses encourage better routing".
    """
    idx = np.asarray(idx)
    T = idx.shape[0]
    f = np.bincount(idx[:, 0].astype(np.int64), minlength=E).astype(f64) / T
    P = np.asarray(probs, f64).mean(axis=0)
    return float(E * np.sum(f * P))


def balance_bias_update(logit_bias, counts, gamma: float) -> np.ndarray:
    """Auxiliary-loss-free balancing: move each expert's logit bias by gamma
    toward balanced load.

    [LECTURE] "The central problem: load balancing" (per-expert bias terms
    that follow the observed load).  An expert with more assignments than
    the mean loses gamma, one with fewer gains gamma, one at the mean keeps
    its bias.  Returns the new (E,) fp32 bias.
    """
    b = np.asarray(logit_bias, f64)
    c = np.asarray(counts, np.int64)
    E = c.shape[0]
    total = int(c.sum())
    step = np.where(c * E > total, -1.0, np.where(c * E < total, 1.0, 0.0))
    return (b + gamma * step).astype(np.float32)


def router_z_loss(logits) -> float:
    """Router z-loss: mean over tokens of (log sum_e exp g_{t,e})^2.

    [LECTURE] "The central problem: load balancing" (a z-loss term on the
    router that keeps its logits small, for numerical stability).  The log-sum-exp is taken stably around the row
    maximum.  Returns 0 for an empty batch.
    """
    g = np.asarray(logits, f64)
    if g.shape[0] == 0:
        return 0.0
    m = g.max(axis=1)
    lse = m + np.log(np.exp(g - m[:, None]).sum(axis=1))
    return float(np.mean(lse * lse))


def dispatch_layout(idx, kept, E: int):
    """Expert-contiguous order of the kept assignments.

    [LECTURE] "The MoE layer", the dispatch loop of its listing: for each
    expert in turn, the rows (tokens) routed to it, in ascending token order.
    Returns
      counts     (E,)   assignments routed to each expert, before the cap
      kept_count (E,)   assignments kept per expert
      offsets    (E+1,) start of each expert's segment (exclusive prefix sum)
      slot_of    (T, k) segment position of each assignment, -1 if dropped
      perm_token (n_kept,) token of each segment position
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(E, np.int64)
    kept_count = np.zeros(E, np.int64)
    for e in range(E):
        counts[e] = int(np.sum(idx == e))
        kept_count[e] = int(np.sum((idx == e) & kept))
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(kept_count)
    slot_of = np.full((T, k), -1, np.int64)
    perm_token = np.zeros(int(offsets[E]), np.int64)
    for e in range(E):
        pos = int(offsets[e])
        for t in np.nonzero(((idx == e) & kept).any(axis=1))[0]:
            j = int(np.nonzero(idx[t] == e)[0][0])
            slot_of[t, j] = pos
            perm_token[pos] = t
            pos += 1
    return counts, kept_count, offsets, slot_of, perm_token


@dataclass
class OracleResult:
    logits: np.ndarray      # (T, E) fp32 routing input
    probs: np.ndarray       # (T, E) fp64
    idx: np.ndarray         # (T, k) int32
    w: np.ndarray           # (T, k) fp64
    kept: np.ndarray        # (T, k) bool
    counts: np.ndarray      # (E,)
    kept_count: np.ndarray  # (E,)
    offsets: np.ndarray     # (E+1,)
    slot_of: np.ndarray     # (T, k)
    perm_token: np.ndarray  # (n_kept,)
    aux: float
    y: np.ndarray           # (len(tokens), d) fp64
    tokens: np.ndarray      # rows of the layer output held in y
    z_loss: float = 0.0     # router z-loss


def moe_forward(x, W_r, W1, b1, W2, b2, k: int, renormalize: bool = True,
                capacity: int | None = None, logit_bias=None, logits=None,
                tokens=None, layout: bool = True, logit_noise=None,
                n_shared: int = 0, reroute: bool = False) -> OracleResult:
    """The MoE layer forward pass, looping over experts.

    [LECTURE] "The MoE layer": router logits and softmax, top-k selection,
    output = sum over the selected experts of weight x expert output; its
    listing's loop dispatches each expert's tokens and accumulates the
    weighted outputs; "The central problem: load balancing" gives the
    capacity drop and the auxiliary loss.  [RATISH] "How does MoE work?"
    (router, experts, combine).

    ``logits`` (T, E fp32) replaces the router GEMM when given (routing from
    identical logits).  ``tokens`` restricts the expert computation (not the
    routing, cap or loss, which always cover the whole batch) to a subset of
    token rows; ``y`` then holds those rows in that order.

    ``n_shared`` > 0: experts 0 .. n_shared-1 of the E in W1..b2 are shared
    ([LECTURE] "Design variations": always active for every token, weight 1,
    never capped); the router (W_r with E - n_shared rows, the logits, the
    softmax, the top-k, the loss) covers the routed experts n_shared .. E-1.
    idx, w and kept then have k + n_shared columns: the k routed choices, then
    the shared experts.

    ``reroute``: an assignment the cap drops is offered to the token's
    next-best expert (``reroute_keep``); ``idx`` then holds each slot's final
    expert (the original choice when not dropped), ``w`` its weight and
    ``kept`` whether it survived; ``counts`` stay those of the k choices; the
    layout follows ``reroute_layout``.  Not combined with shared experts.
    """
    x = np.asarray(x)
    T, d = x.shape
    if logits is None:
        logits = router_logits(x, W_r, logit_bias, logit_noise)
    logits = np.asarray(logits, np.float32)
    E_r = logits.shape[1]
    E = E_r + n_shared
    probs = softmax(logits)
    idx_r = top_k(logits, k)
    w = gate_weights(probs, idx_r, renormalize)
    aux = aux_loss(probs, idx_r, E_r)
    idx = idx_r + n_shared
    if n_shared:
        idx = np.concatenate([idx, np.tile(np.arange(n_shared, dtype=idx.dtype), (T, 1))], 1)
        w = np.concatenate([w, np.ones((T, n_shared))], 1)
    if reroute:
        if n_shared:
            raise ValueError("rerouting is not combined with shared experts")
        ranked = top_k(logits, min(2 * k, E))
        final, phase = reroute_keep(ranked, k, E, capacity)
        counts = np.bincount(idx.ravel().astype(np.int64), minlength=E)
        rows = np.arange(T)[:, None]
        den = probs[rows, idx].sum(axis=1, keepdims=True) if renormalize else np.ones((T, 1))
        moved = phase == 2
        w = np.where(moved, probs[rows, np.maximum(final, 0)] / den, w)
        idx = np.where(moved, final, idx).astype(idx.dtype)
        kept = final >= 0
        kept_count = np.bincount(final[kept], minlength=E)
        if layout:
            offsets, slot_of, perm_token = reroute_layout(final, phase, E)
        else:
            offsets = slot_of = perm_token = None
    elif layout:
        kept = capacity_keep(idx, E, capacity, n_shared)
        counts, kept_count, offsets, slot_of, perm_token = dispatch_layout(idx, kept, E)
    else:
        kept = capacity_keep(idx, E, capacity, n_shared)
        counts = kept_count = offsets = slot_of = perm_token = None
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, np.int64)
    y = np.zeros((len(tokens), d), f64)
    sub_idx, sub_kept, sub_w = idx[tokens], kept[tokens], w[tokens]
    for e in range(E):
        sel = (sub_idx == e) & sub_kept                 # (n, k)
        rows = np.nonzero(sel.any(axis=1))[0]
        if rows.size == 0:
            continue
        out = expert_ffn(x[tokens[rows]], W1[e], b1[e], W2[e], b2[e])
        we = (sub_w * sel)[rows].sum(axis=1)
        y[rows] += we[:, None] * out
    return OracleResult(logits, probs, idx, w, kept, counts, kept_count, offsets, slot_of,
                        perm_token, aux, y, tokens, router_z_loss(logits))


def expert_choice_capacity(T: int, E: int, k: int, capacity: int | None = None) -> int:
    """C, the tokens each expert takes under expert-choice routing.

    [LECTURE] "Design variations" (expert-choice routing) and "The central
    problem: load balancing" (capacity as a multiple of the even share): the
    given
    capacity, else ceil(T k / E), the load top-k token choice averages per
    expert; never more than the T tokens of the batch.
    """
    c = int(math.ceil(T * k / E)) if capacity is None else int(capacity)
    return max(0, min(c, T))


def expert_choice_select(probs, C: int) -> np.ndarray:
    """For each expert, the C tokens with the largest router probability.

    [LECTURE] "Design variations": each expert chooses its top tokens (a
    top-C over the token axis of p instead of a top-k over the expert axis).
    Among equal probabilities the lower token index ranks first.  Each row
    of the result lists the chosen tokens in ascending token order.
    probs: (T, E); returns (E, C) int64.
    """
    p = np.asarray(probs, f64)
    T, E = p.shape
    sel = np.zeros((E, C), np.int64)
    for e in range(E):
        order = np.lexsort((np.arange(T), -p[:, e]))  # by -p, then by token
        sel[e] = np.sort(order[:C])
    return sel


@dataclass
class ExpertChoiceResult:
    logits: np.ndarray      # (T, E) fp32 routing input
    probs: np.ndarray       # (T, E) fp64
    C: int                  # tokens per expert
    sel: np.ndarray         # (E, C) chosen tokens, ascending
    w: np.ndarray           # (E, C) fp64 p[sel, e]
    slot_of: np.ndarray     # (T, E) row e*C + j of (token, expert), -1 if not chosen
    y: np.ndarray           # (len(tokens), d) fp64
    tokens: np.ndarray
    z_loss: float


def expert_choice_forward(x, W_r, W1, b1, W2, b2, k: int, capacity: int | None = None,
                          logit_bias=None, logit_noise=None, logits=None, sel=None,
                          tokens=None) -> ExpertChoiceResult:
    """The MoE layer with expert-choice routing, looping over experts.

    [LECTURE] "Design variations" (each expert selects the tokens it takes,
    which balances the load by construction) on the layer of "The MoE layer"
    (router logits and
    softmax, expert FFNs, weighted sum of the experts' outputs).  ``logits``
    replaces the router GEMM when given; ``sel`` (E, C) replaces the
    selection (to evaluate the layer on another valid choice among equal
    probabilities); ``tokens`` restricts the output rows as in moe_forward.
    """
    x = np.asarray(x)
    T, d = x.shape
    if logits is None:
        logits = router_logits(x, W_r, logit_bias, logit_noise)
    logits = np.asarray(logits, np.float32)
    E = logits.shape[1]
    probs = softmax(logits)
    C = expert_choice_capacity(T, E, k, capacity)
    if sel is None:
        sel = expert_choice_select(probs, C)
    sel = np.asarray(sel, np.int64)
    w = np.take_along_axis(probs.T, sel, axis=1) if C else np.zeros((E, 0))
    slot_of = np.full((T, E), -1, np.int64)
    for e in range(E):
        slot_of[sel[e], e] = e * C + np.arange(C)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, np.int64)
    pos = {int(t): i for i, t in enumerate(tokens)}
    y = np.zeros((len(tokens), d), f64)
    for e in range(E):
        rows = [j for j in range(C) if int(sel[e, j]) in pos]
        if not rows:
            continue
        toks = sel[e, rows]
        out = expert_ffn(x[toks], W1[e], b1[e], W2[e], b2[e])
        for r, t in enumerate(toks):
            y[pos[int(t)]] += w[e, rows[r]] * out[r]
    return ExpertChoiceResult(logits, probs, C, sel, w, slot_of, y, tokens,
                              router_z_loss(logits))


def gelu_grad(u) -> np.ndarray:
    """d/du of the exact GELU: Phi(u) + u phi(u).

    Derivative of [LECTURE] "The MoE layer"'s GELU (``nn.GELU()``)."""
    u = np.asarray(u, f64)
    return 0.5 * (1.0 + erf(u / math.sqrt(2.0))) + u * np.exp(-0.5 * u * u) / math.sqrt(2 * math.pi)


def moe_backward(x, W_r, W1, b1, W2, b2, dy, k: int, renormalize: bool = True,
                 capacity: int | None = None, logit_bias=None, logits=None,
                 aux_grad: float = 0.0, z_grad: float = 0.0, n_shared: int = 0,
                 reroute: bool = False) -> dict:
    """Gradients of L = <dy, y> + aux_grad * aux + z_grad * z_loss.

    The training step behind [LECTURE] "The MoE layer" (the layer is trained
    end to end with the load-balancing loss of "The central problem: load
    balancing"; [DAY59] "Load-balancing losses encourage better routing").
    Routing decisions (top-k, capacity, rerouting) are constants.  Per kept
    assignment (token t, expert e, weight w): u = W1_e x + b1_e, h = GELU(u),
    o = W2_e h + b2_e, y_t += w o; hence do = w dy_t, dW2_e += do h^T,
    db2_e += do, du = (W2_e^T do) * GELU'(u), dW1_e += du x^T, db1_e += du,
    dx_t += W1_e^T du, and s = <dy_t, w o> feeds the logits through w.

    A routed slot j of token t has final expert f_j (its choice c_j, or with
    ``reroute`` the expert a dropped slot moved to) and weight w_j = p_{f_j} / S
    with S the sum of p over the token's k choices (renormalised; S = 1
    otherwise).  With p the softmax of g:
        dw_j/dg_m = w_j [m = f_j] - w_j p_m ([m in choices] / S   (renormalised)
                                             1                    (otherwise)),
    so dg_m = sum over the kept slots with f_j = m of s_j - (sum_j s_j) *
    (p_m / S if m is a choice, else 0) when renormalised, and
    dg_m = sum_{f_j = m} s_j - p_m sum_j s_j otherwise; a dropped slot has
    s_j = 0 but its choice still counts in S.  Shared experts (``n_shared``,
    [LECTURE] "Design variations") have weight 1: their slots add to the
    expert gradients and dx but not to the logits, which cover the routed
    experts only.  The auxiliary loss adds aux_grad E / T * p_e (f_e -
    sum_i f_i p_i) (f from the first choice), the z-loss
    z_grad 2 / T * lse_t p_e.  Then dW_r = dg^T x and dx += dg W_r.
    ``logits`` replaces the router GEMM as in moe_forward (W_r still gets
    its gradient from dg).  Returns dx (T, d), dW_r (E - n_shared, d), dW1,
    db1, dW2, db2, all fp64, and dg (T, E - n_shared).
    """
    x = np.asarray(x, f64)
    dy = np.asarray(dy, f64)
    T, d = x.shape
    r = moe_forward(x, W_r, W1, b1, W2, b2, k=k, renormalize=renormalize, capacity=capacity,
                    logit_bias=logit_bias, logits=logits, layout=False, n_shared=n_shared,
                    reroute=reroute)
    E_r = r.logits.shape[1]
    p = r.probs
    g = np.asarray(r.logits, f64)
    choices = top_k(r.logits, k)  # (T, k) routed expert ids, the weights' normaliser
    W1, b1, W2, b2 = (np.asarray(a, f64) for a in (W1, b1, W2, b2))
    K = r.idx.shape[1]
    dx = np.zeros((T, d))
    dW1, db1 = np.zeros_like(W1), np.zeros_like(b1)
    dW2, db2 = np.zeros_like(W2), np.zeros_like(b2)
    s = np.zeros((T, K))  # <dy_t, w o> per slot (0 when dropped)
    for t in range(T):
        for j in range(K):
            if not r.kept[t, j]:
                continue
            e, w = int(r.idx[t, j]), r.w[t, j]
            u = W1[e] @ x[t] + b1[e]
            h = gelu(u)
            o = W2[e] @ h + b2[e]
            s[t, j] = w * float(dy[t] @ o)
            do = w * dy[t]
            dW2[e] += np.outer(do, h)
            db2[e] += do
            du = (W2[e].T @ do) * gelu_grad(u)
            dW1[e] += np.outer(du, x[t])
            db1[e] += du
            dx[t] += W1[e].T @ du
    dg = np.zeros((T, E_r))
    for t in range(T):
        tot = s[t, :k].sum()  # the routed slots
        for j in range(k):
            if r.kept[t, j]:
                dg[t, int(r.idx[t, j]) - n_shared] += s[t, j]
        if renormalize:
            S = p[t, choices[t]].sum()
            for c in choices[t]:
                dg[t, c] -= tot * p[t, c] / S
        else:
            dg[t] -= p[t] * tot
    if aux_grad:
        f = np.bincount(np.asarray(choices[:, 0], np.int64), minlength=E_r) / T
        fp = (p * f[None, :]).sum(axis=1, keepdims=True)
        dg += aux_grad * E_r / T * p * (f[None, :] - fp)
    if z_grad:
        m = g.max(axis=1, keepdims=True)
        lse = m + np.log(np.exp(g - m).sum(axis=1, keepdims=True))
        dg += z_grad * 2.0 / T * lse * p
    dW_r = dg.T @ x
    dx += dg @ np.asarray(W_r, f64)
    return dict(dx=dx, dW_r=dW_r, dW1=dW1, db1=db1, dW2=dW2, db2=db2, dg=dg)


def expert_choice_backward(x, W_r, W1, b1, W2, b2, dy, k: int, capacity: int | None = None,
                           logit_bias=None, logits=None, sel=None, z_grad: float = 0.0) -> dict:
    """Gradients of L = <dy, y> + z_grad * z_loss for the expert-choice layer
    (expert_choice_forward; [LECTURE] "Design variations"), the selection
    held constant.  Each chosen (token t, expert e) adds y_t += p_{t,e} o_e(x_t):
    the expert gradients as in moe_backward with w = p_{t,e}, and with
    s_{t,e} = <dy_t, p_{t,e} o> the softmax gives dg_{t,m} = s_{t,m} [m chose t]
    - p_{t,m} sum_e s_{t,e}.  There is no balancing loss.  Returns dx, dW_r,
    dW1, db1, dW2, db2 (fp64) and dg (T, E)."""
    x = np.asarray(x, f64)
    dy = np.asarray(dy, f64)
    T, d = x.shape
    r = expert_choice_forward(x, W_r, W1, b1, W2, b2, k=k, capacity=capacity,
                              logit_bias=logit_bias, logits=logits, sel=sel)
    E = r.logits.shape[1]
    p = r.probs
    g = np.asarray(r.logits, f64)
    W1, b1, W2, b2 = (np.asarray(a, f64) for a in (W1, b1, W2, b2))
    dx = np.zeros((T, d))
    dW1, db1 = np.zeros_like(W1), np.zeros_like(b1)
    dW2, db2 = np.zeros_like(W2), np.zeros_like(b2)
    s = np.zeros((T, E))
    for e in range(E):
        for j in range(r.C):
            t, w = int(r.sel[e, j]), r.w[e, j]
            u = W1[e] @ x[t] + b1[e]
            h = gelu(u)
            o = W2[e] @ h + b2[e]
            s[t, e] = w * float(dy[t] @ o)
            do = w * dy[t]
            dW2[e] += np.outer(do, h)
            db2[e] += do
            du = (W2[e].T @ do) * gelu_grad(u)
            dW1[e] += np.outer(du, x[t])
            db1[e] += du
            dx[t] += W1[e].T @ du
    dg = s - p * s.sum(axis=1, keepdims=True)
    if z_grad:
        m = g.max(axis=1, keepdims=True)
        lse = m + np.log(np.exp(g - m).sum(axis=1, keepdims=True))
        dg += z_grad * 2.0 / T * lse * p
    dW_r = dg.T @ x
    dx += dg @ np.asarray(W_r, f64)
    return dict(dx=dx, dW_r=dW_r, dW1=dW1, db1=db1, dW2=dW2, db2=db2, dg=dg)
