"""The first grouped GEMM's GELU epilogue on the GPU, element by element,
over pre-activations spanning [-8, 8].

"Mixture of Experts: Scaling Parameters Without Scaling Compute", section
"The MoE layer": h = GELU(x W1^T + b1) with the exact-erf GELU.  The bf16
kernels evaluate erf with Abramowitz & Stegun 7.1.26 and round h to bf16.
To read h through the public C ABI, one expert with W1 = W2 = I and zero
biases runs through moe_expert_ffn: U = x_perm exactly (one nonzero product
per output), and y_perm = h exactly (fp32 sums of one bf16 value and zeros),
so y_perm holds the kernels' bf16 h for every U.  U walks every bf16 value
in [-8, 8].

Bound (derived, not fitted): |h - GELU(U)| <= half a bf16 ulp of h (the
rounding of the fp32 result) + 7e-8 |U| (the formula's error, pinned on the
CPU by tests/test_gelu_approx.py) + 2e-6 |GELU(U)| + 1e-30 (fp32 evaluation:
the base-2 exponential, the reciprocal, five fused multiply-adds).
Both GEMM kernels are covered: the CTA-pair kernel (2048 rows) and the
single-CTA kernel for small batches (64 rows).
"""
import numpy as np
import pytest
import torch
from scipy.special import erf

from sparse_mixture_experts_71_b300 import binding as B
from sparse_mixture_experts_71_b300 import inputs as I

pytestmark = pytest.mark.gpu

D = 256  # d = d_ff: W1 and W2 are 256 x 256 identities


def _bf16_grid():
    """Every finite bf16 value in [-8, 8] (as fp32)."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    v = I.bf16_bits_to_f32(bits)
    v = v[np.isfinite(v) & (np.abs(v) <= 8.0)]
    return np.unique(v)


def _ulp_bf16(v):
    """Spacing of bf16 values at |v| (the normal-range exponent of v)."""
    a = np.maximum(np.abs(v.astype(np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("rows", [2048, 64], ids=["pair-kernel", "single-cta-kernel"])
def test_first_gemm_gelu_over_the_bf16_grid(rows):
    grid = _bf16_grid()
    vals = np.resize(grid, rows * D).astype(np.float32)  # the grid, cycled through the rows
    if rows * D < grid.size:  # the small case: an even subsample that keeps both ends
        vals = grid[np.linspace(0, grid.size - 1, rows * D).astype(np.int64)].astype(np.float32)
    x = torch.from_numpy(I.f32_to_bf16_bits(vals).view(np.int16)).view(torch.bfloat16)
    x = x.reshape(rows, D).cuda()
    eye = torch.eye(D, dtype=torch.bfloat16, device="cuda").reshape(1, D, D).contiguous()
    zb = torch.zeros((1, D), dtype=torch.bfloat16, device="cuda")
    cfg = B.config(rows, D, D, 1, 1)
    ws = B.workspace(cfg)
    offsets = torch.tensor([0, rows], dtype=torch.int32, device="cuda")
    y_perm = torch.full((rows, D), float("nan"), dtype=torch.float32, device="cuda")
    B.expert_ffn(cfg, x, offsets, eye, zb, eye.clone(), zb.clone(), y_perm, ws)
    torch.cuda.synchronize()
    assert B.get_device_error(ws)[0] == 0
    h = y_perm.cpu().numpy().reshape(-1).astype(np.float64)
    u = x.float().cpu().numpy().reshape(-1).astype(np.float64)
    assert np.array_equal(I.f32_to_bf16_bits(h.astype(np.float32)).astype(np.uint32) << 16,
                          h.astype(np.float32).view(np.uint32)), "h is not a bf16 value"
    exact = 0.5 * u * (1.0 + erf(u / np.sqrt(2.0)))
    bound = 0.5 * _ulp_bf16(h) + 7e-8 * np.abs(u) + 2e-6 * np.abs(exact) + 1e-30
    err = np.abs(h - exact)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (f"u={u[worst]!r}: h={h[worst]!r}, GELU={exact[worst]!r}, "
                                  f"|err|={err[worst]:.3e} > {bound[worst]:.3e}")
    # where the formula's error is far below half an ulp (|u| <= 3), h is the
    # correctly rounded bf16 GELU nearly everywhere
    mid = np.abs(u) <= 3.0
    rounded = I.bf16_bits_to_f32(I.f32_to_bf16_bits(exact[mid].astype(np.float32)))
    assert np.mean(h[mid] == rounded) >= 0.99
    assert np.all(h[u == 0.0] == 0.0)
