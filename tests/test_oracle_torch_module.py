"""The oracle against the layer as "Mixture of Experts: Scaling Parameters
Without Scaling Compute", section "The MoE layer", defines it, written here
as a torch module of its own (CPU, fp32, on the tiny fp32 workload's stored
weights): router Linear without bias, softmax over the experts, the k most
probable experts renormalised to sum to one, each expert Linear-GELU-Linear
on the tokens that chose it, the outputs summed with those weights, and the
Switch auxiliary loss E * sum_e f_e P_e with f_e the share of tokens whose
first choice is e and P_e the mean probability of e.

The module computes in fp32 (as such a module runs), the oracle in fp64 on the
same stored values, so they agree to fp32 rounding: max |dy| <= 1e-5 on every
token whose k-th and (k+1)-th probabilities are not near-tied (those may pick a
different expert under the module's tie order), and the routing and the loss
agree exactly / to 1e-6.  Unlike the E = 1 and k = E special cases checked
elsewhere, this is the whole layer at the workload's own shape, k < E.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import moe_oracle as O
from sparse_mixture_experts_71_b300 import inputs as I


class TorchMoELayer(torch.nn.Module):
    """Sparse MoE FFN layer: gate -> softmax -> top-k (renormalised) ->
    per-expert FFN on the tokens routed to it -> weighted sum; plus the
    Switch balancing loss."""

    def __init__(self, W_r, W1, b1, W2, b2, k):
        super().__init__()
        E, d_ff, d = W1.shape
        self.k = k
        self.gate = torch.nn.Linear(d, E, bias=False)
        self.up = torch.nn.ModuleList(torch.nn.Linear(d, d_ff) for _ in range(E))
        self.down = torch.nn.ModuleList(torch.nn.Linear(d_ff, d) for _ in range(E))
        with torch.no_grad():
            self.gate.weight.copy_(torch.as_tensor(W_r))
            for e in range(E):
                self.up[e].weight.copy_(torch.as_tensor(W1[e]))
                self.up[e].bias.copy_(torch.as_tensor(b1[e]))
                self.down[e].weight.copy_(torch.as_tensor(W2[e]))
                self.down[e].bias.copy_(torch.as_tensor(b2[e]))

    def forward(self, x):
        T = x.shape[0]
        E = len(self.up)
        scores = self.gate(x).softmax(dim=1)                 # (T, E)
        top_p, top_e = torch.topk(scores, self.k, dim=1)     # most probable first
        gates = top_p / top_p.sum(dim=1, keepdim=True)
        y = torch.zeros_like(x)
        for e in range(E):
            tok, slot = torch.nonzero(top_e == e, as_tuple=True)
            if tok.numel() == 0:
                continue
            out = self.down[e](F.gelu(self.up[e](x[tok])))
            y.index_add_(0, tok, gates[tok, slot].unsqueeze(1) * out)
        first = torch.bincount(top_e[:, 0], minlength=E).to(x.dtype) / T
        loss = E * torch.dot(first, scores.mean(dim=0))
        return y, loss, top_e


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_equals_the_torch_layer_on_the_tiny_workload(seed):
    wl = I.TINY
    inp = I.make_inputs(wl, seed=seed)
    x, W1, b1, W2, b2 = (inp.as_f32(n) for n in ("x", "W1", "b1", "W2", "b2"))
    layer = TorchMoELayer(inp.W_r, W1, b1, W2, b2, wl.k)
    with torch.no_grad():
        y_t, aux_t, top_e = layer(torch.from_numpy(x))
    ref = O.moe_forward(x, inp.W_r, W1, b1, W2, b2, k=wl.k, renormalize=True, layout=False)
    s = -np.sort(-ref.probs, axis=1)
    ok = (s[:, wl.k - 1] - s[:, wl.k]) >= 1e-6
    assert ok.mean() > 0.9
    assert np.array_equal(top_e.numpy()[ok], ref.idx[ok])
    d = np.abs(y_t.double().numpy() - ref.y)[ok]
    assert d.max() <= 1e-5, d.max()
    assert np.abs(ref.y).max() > 0.1  # a non-trivial output
    if ok.all():
        assert abs(float(aux_t) - ref.aux) <= 1e-6


def test_torch_layer_catches_a_planted_oracle_mistake():
    """The comparison is sharp enough to see a dropped renormalisation."""
    wl = I.TINY
    inp = I.make_inputs(wl, seed=0)
    x, W1, b1, W2, b2 = (inp.as_f32(n) for n in ("x", "W1", "b1", "W2", "b2"))
    with torch.no_grad():
        y_t, _, _ = TorchMoELayer(inp.W_r, W1, b1, W2, b2, wl.k)(torch.from_numpy(x))
    wrong = O.moe_forward(x, inp.W_r, W1, b1, W2, b2, k=wl.k, renormalize=False, layout=False)
    assert np.abs(y_t.double().numpy() - wrong.y).max() > 1e-2
