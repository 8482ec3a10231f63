"""GPU: the autograd integration.  A loss scaled after the call must scale
both gradients (the backward only distributes the gradients computed in the
forward), and the results must match the fp64 oracle."""
import numpy as np
import pytest

from linear_cross_entropy_ce_gb300 import workloads as wl
from oracle import flce_oracle
from tests.helpers import LOSS_RTOL, GRAD_FROB_RTOL, to_device, frob_rel, loss_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_ce_gb300 import flce
    try:
        flce.library()
    except RuntimeError:
        import __graft_entry__
        __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("scale", [1.0, 2.5, -0.75])
def test_autograd_matches_oracle(dev, scale):
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    p = wl.random_problem(600, 128, 1000, seed=31, ignore_frac=0.1)
    h, w, t = to_device(p, dev)
    h = h.clone().requires_grad_(True)
    w = w.clone().requires_grad_(True)
    loss = flce.linear_cross_entropy(h, w, t)
    (scale * loss).backward()
    ref = flce_oracle(p["hidden"], p["weight"], p["targets"])
    assert loss_rel(float(loss.item()), ref["loss"]) <= LOSS_RTOL
    assert h.grad.dtype == torch.bfloat16
    assert frob_rel(h.grad.float().cpu().double().numpy(), scale * ref["grad_hidden"]) <= GRAD_FROB_RTOL
    assert frob_rel(w.grad.float().cpu().double().numpy(), scale * ref["grad_weight"]) <= GRAD_FROB_RTOL


def test_module_with_fp32_master_weight_grad(dev):
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    p = wl.random_problem(300, 64, 512, seed=32, ignore_frac=0.2)
    h, w, t = to_device(p, dev)
    m = flce.LinearCrossEntropy(w.clone())
    loss = m(h, t)
    loss.backward()
    ref = flce_oracle(p["hidden"], p["weight"], p["targets"])
    assert loss_rel(float(loss.item()), ref["loss"]) <= LOSS_RTOL
    assert frob_rel(m.weight.grad.float().cpu().double().numpy(), ref["grad_weight"]) <= GRAD_FROB_RTOL


def test_scale_grads_kernel(dev):
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    gh = torch.randn(37, 64, device=dev).to(torch.bfloat16)
    gw = torch.randn(10, 64, device=dev)
    gh0, gw0 = gh.clone(), gw.clone()
    flce.scale_grads(gh, gw, torch.tensor([3.0], device=dev))
    torch.testing.assert_close(gh.float(), (gh0.float() * 3.0).to(torch.bfloat16).float(), rtol=0, atol=0)
    torch.testing.assert_close(gw, gw0 * 3.0, rtol=0, atol=0)
