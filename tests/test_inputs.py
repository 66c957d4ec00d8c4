"""The seeded input generator: stored bf16 values and reproducibility."""
import numpy as np
import torch

from sparse_mixture_experts_71_b300 import inputs as I


def test_bf16_rounding_matches_torch():
    a = np.random.default_rng(0).standard_normal(100_000).astype(np.float32) * 7
    a[:4] = [0.0, -0.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8]  # exact ties, both parities
    bits = I.f32_to_bf16_bits(a)
    want = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, want)
    back = I.bf16_bits_to_f32(bits)
    assert np.array_equal(back, torch.from_numpy(a).to(torch.bfloat16).float().numpy())


def test_draws_do_not_depend_on_thread_count(monkeypatch):
    n = 3 * I._CHUNK + 17
    a = I._draw(3, 9, n, "normal", 1.0)
    monkeypatch.setattr(I, "_threads", lambda: 1)
    b = I._draw(3, 9, n, "normal", 1.0)
    assert np.array_equal(a, b)
    assert abs(float(a.std()) - 1.0) < 1e-2


def test_workload_recipes():
    w = I.TINY.with_(T=8)
    inp = I.make_inputs(w, seed=0)
    assert inp.x.dtype == np.float32 and inp.x.shape == (8, 256)
    assert np.all(np.abs(inp.W1) <= 1 / 16) and inp.logit_bias is None
    s = I.make_inputs(I.SWITCH.with_(T=16, d=64, F=128), seed=0)
    assert s.x.dtype == np.uint16 and s.W1.shape == (64, 128, 64)
    assert s.logit_bias[0] == 0.0 and np.all(np.diff(s.logit_bias) < 0)
    np.testing.assert_allclose(s.logit_bias[1], 1.5 * np.log(0.5), rtol=1e-7)
    # same seed, same values; another seed, other values
    assert np.array_equal(I.make_inputs(w, 0).W2, inp.W2)
    assert not np.array_equal(I.make_inputs(w, 1).W2, inp.W2)
