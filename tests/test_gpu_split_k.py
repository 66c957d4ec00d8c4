"""The second expert GEMM with each tile's K split in two halves: the fused
expert-FFN kernel (both GEMMs in one launch of CTA pairs) does this when the
half tiles fill the last wave of the 74 CTA pairs clearly better than whole
tiles (the first half stores (acc + b2) w, the second adds acc w once the
first half's epilogue warps have counted themselves), so the layer output
must still match the oracle and repeat bit for bit.  The second-GEMM tiles
also wait on the first GEMM's per-token-tile ready counts, which every
forward test exercises.

"Mixture of Experts: Scaling Parameters Without Scaling Compute", section
"The MoE layer": y_t = sum over the chosen experts of w_e (W2_e GELU(W1_e x_t
+ b1_e) + b2_e); splitting the sum over d_ff changes only its rounding.
"""
import math

import numpy as np
import pytest
import torch

from parity import LibRun, assert_y_close, oracle_on, to_np
from sparse_mixture_experts_71_b300 import inputs as I

pytestmark = pytest.mark.gpu

PAIRS = 74  # CTA pairs of the pair kernel's grid (148 SMs)


def _splits(offsets, d, d_ff):
    """The kernel's rule, restated: whole tiles = 256-token tiles x 256-row
    weight tiles; split when 2w / ceil(2w) > w / ceil(w) + 0.05, w = tiles /
    pairs, and d_ff is a multiple of 256 (two stages of 128)."""
    rows = np.diff(np.asarray(offsets, np.int64))
    tiles = int(sum((r + 255) // 256 for r in rows)) * ((d + 255) // 256)
    w = tiles / PAIRS
    return d_ff % 256 == 0 and 0 < tiles <= 512 and \
        2 * w / math.ceil(2 * w) > w / math.ceil(w) + 0.05


CASES = [
    # 640 rows per expert: 3 token tiles x 4 weight tiles x 8 experts = 96
    # tiles, 1.3 waves whole, 2.6 waves in halves
    I.Workload("splitk-96-tiles", 2560, 1024, 2048, 8, 2),
    # capped and skewed: fewer tiles than pairs (0.46 waves whole), ragged
    # token tiles, two experts with no rows
    I.Workload("splitk-capped", 3000, 512, 1024, 16, 2, capacity=300, zipf_bias=1.0),
    # capped, four experts full: 104 tiles, 1.4 waves whole
    I.Workload("splitk-capped-104", 6000, 1024, 1024, 16, 2, capacity=600, zipf_bias=1.0),
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_split_second_gemm_matches_oracle(wl):
    inp = I.make_inputs(wl, seed=17)
    run = LibRun(wl, inp)
    staged = run.staged()
    assert _splits(to_np(staged["offsets"]), wl.d, wl.F), "the case must take the split path"
    f = run.forward()
    assert torch.equal(f["y"], staged["y"])  # the same kernels, the same bits
    g = to_np(f["logits"])
    tokens = np.arange(0, wl.T, 3)
    ref = oracle_on(inp, wl, logits=g, tokens=tokens, layout=False)
    max_abs, rel = assert_y_close(to_np(f["y"])[tokens], ref.y, wl.dtype)
    if wl.capacity is not None:
        dropped = ~ref.kept[tokens].any(axis=1)  # kept covers every token
        assert np.all(to_np(f["y"])[tokens][dropped] == 0.0)
    assert torch.equal(run.forward()["y"], f["y"])  # deterministic
    print(f"{wl.name}: max|dy| {max_abs:.2e} rel {rel:.2e}")
