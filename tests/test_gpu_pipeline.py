"""GPU: the host-buffer executor (moe_pipeline_*).  Every batch's y and loss
must equal moe_forward's on the same batch bit for bit (the same kernels on
the same inputs), whatever the overlap depth and whether the host buffers are
pinned; the first batch is also checked against the oracle."""
import numpy as np
import pytest
import torch

from parity import assert_y_close, oracle_on, to_np
from sparse_mixture_experts_71_b300 import inputs as I
from sparse_mixture_experts_71_b300.layer import MoELayer, device_inputs, to_torch

pytestmark = pytest.mark.gpu

WORKLOADS = [
    I.MEDIUM.with_(name="pipe-bf16", T=300, d=256, F=512),
    I.TINY,
    I.SWITCH.with_(name="pipe-switch", T=500, d=128, F=256, capacity=9),
]


def _host(a, pinned):
    t = to_torch(a, "cpu")
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("wl", WORKLOADS, ids=[w.name for w in WORKLOADS])
@pytest.mark.parametrize("depth,pinned", [(1, True), (2, True), (3, True), (2, False)])
def test_pipeline_equals_forward(wl, depth, pinned):
    inp = I.make_inputs(wl, seed=0)
    D = device_inputs(inp, "cuda")
    layer = MoELayer(D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], k=wl.k, capacity=wl.capacity,
                     renormalize=wl.renormalize, logit_bias=D["logit_bias"])
    nb = 5
    xs = [inp.x] + [I.make_inputs(wl, seed=100 + s).x for s in range(1, nb)]
    x_host = [_host(x, pinned) for x in xs]
    dt = D["x"].dtype
    y_host = [torch.full((wl.T, wl.d), float("nan"), dtype=dt) for _ in range(nb)]
    y_host = [y.pin_memory() if pinned else y for y in y_host]
    aux_host = [torch.full((1,), float("nan")) for _ in range(nb)]
    aux_host = [a.pin_memory() if pinned else a for a in aux_host]

    pipe = layer.host_pipeline(wl.T, depth=depth)
    for s in range(3):  # a first round of three batches, joined
        pipe.submit(x_host[s], y_host[s], aux_host[s])
    pipe.join()
    for s in range(3, nb):  # a second round after the join
        pipe.submit(x_host[s], y_host[s], aux_host[s])
    pipe.join()
    torch.cuda.current_stream().synchronize()
    pipe.close()

    for s in range(nb):
        x_dev = x_host[s].to("cuda")
        y_ref, aux_ref = layer.forward(x_dev)
        torch.cuda.synchronize()
        assert torch.equal(y_host[s], y_ref.cpu()), f"batch {s}"
        assert aux_host[s][0].item() == aux_ref[0].item(), f"batch {s}"
    # the oracle routed from the kernels' fp32 logits (near ties decided alike)
    logits = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    layer.forward(x_host[0].to("cuda"), logits_out=logits)
    torch.cuda.synchronize()
    ref = oracle_on(inp, wl, logits=to_np(logits))
    assert_y_close(to_np(y_host[0]), ref.y, wl.dtype)
    assert abs(aux_host[0][0].item() - ref.aux) <= 1e-5 * max(1.0, ref.aux)


def test_pipeline_without_aux_and_more_batches_than_slots():
    wl = WORKLOADS[0]
    inp = I.make_inputs(wl, seed=0)
    D = device_inputs(inp, "cuda")
    layer = MoELayer(D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], k=wl.k, capacity=wl.capacity,
                     renormalize=wl.renormalize, logit_bias=D["logit_bias"])
    x = _host(inp.x, True)
    nb = 9
    ys = [torch.empty((wl.T, wl.d), dtype=D["x"].dtype).pin_memory() for _ in range(nb)]
    pipe = layer.host_pipeline(wl.T, depth=2)
    for s in range(nb):  # one host input read by every batch
        pipe.submit(x, ys[s])
    pipe.join()
    torch.cuda.current_stream().synchronize()
    y_ref, _ = layer.forward(x.to("cuda"))
    torch.cuda.synchronize()
    for s in range(nb):
        assert torch.equal(ys[s], y_ref.cpu()), f"batch {s}"
    assert np.isfinite(to_np(ys[-1]).astype(np.float32)).all()
