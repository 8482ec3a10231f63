"""GPU parity of the final RMSNorm fused in front of the LM head against the
fp64 oracle (same tolerances as the plain path; grad_gain to 1e-2 Frobenius)."""
import numpy as np
import pytest

from linear_cross_entropy_ce_gb300 import workloads as wl
from oracle import rmsnorm_flce_oracle
from tests.helpers import LOSS_RTOL, GRAD_FROB_RTOL, to_device, frob_rel, loss_rel, gh_np

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


def _gain(H, seed):
    rng = np.random.default_rng(seed)
    return wl.f32_to_bf16_bits((1.0 + 0.2 * rng.standard_normal(H)).astype(np.float32))


@pytest.mark.parametrize("N,H,V,ign,seed,eps", [
    (300, 64, 512, 0.1, 1, 1e-6),
    (1000, 200, 1000, 0.2, 2, 1e-5),
    (700, 512, 16000, 0.05, 3, 1e-6),
    (257, 8, 300, 0.0, 4, 1e-3),
])
def test_rmsnorm_matches_oracle(dev, N, H, V, ign, seed, eps):
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    p = wl.random_problem(N, H, V, seed=seed, ignore_frac=ign, hidden_std=3.0)
    g = _gain(H, seed)
    h, w, t = to_device(p, dev)
    gt = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).to(dev)
    out = flce.rmsnorm_fwd_bwd(h, gt, w, t, eps=eps, row_loss=True)
    assert flce.query_status(out["workspace"]) == flce.FLCE_OK
    ref = rmsnorm_flce_oracle(p["hidden"], g, p["weight"], p["targets"], eps)
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert loss_rel(float(out["loss"].item()), ref["loss"]) <= LOSS_RTOL
    assert frob_rel(gh_np(out["grad_hidden"]), ref["grad_hidden"]) <= GRAD_FROB_RTOL
    assert frob_rel(out["grad_gain"].cpu().double().numpy(), ref["grad_gain"]) <= GRAD_FROB_RTOL
    assert frob_rel(out["grad_weight"].cpu().double().numpy(), ref["grad_weight"]) <= GRAD_FROB_RTOL
    ign_rows = torch.from_numpy(p["targets"] == -100).to(dev)
    if bool(ign_rows.any()):
        assert int(out["grad_hidden"].view(torch.int16)[ign_rows].abs().max().item()) == 0
    again = flce.rmsnorm_fwd_bwd(h, gt, w, t, eps=eps)
    for k in ("loss", "grad_hidden", "grad_gain", "grad_weight"):
        assert torch.equal(out[k], again[k]), k


def test_rmsnorm_unit_gain_equals_plain_on_normalised_input(dev):
    # with gain = 1 and the hidden rows already at unit RMS (eps = 0), the loss
    # and grad_weight equal those of the plain path on the same rows
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    w_ = wl.WORKLOADS["llama3_8b_head"].with_shape(N=256, H=512, V=3000)
    p = wl.make_inputs(w_)
    h, w, t = to_device(p, dev)
    g = torch.ones(512, dtype=torch.bfloat16, device=dev)
    a = flce.rmsnorm_fwd_bwd(h, g, w, t, eps=0.0)
    b = flce.fwd_bwd(h, w, t)
    assert abs(float(a["loss"].item()) - float(b["loss"].item())) <= 2e-3 * abs(float(b["loss"].item()))
    assert frob_rel(a["grad_weight"].cpu().double().numpy(), b["grad_weight"].cpu().double().numpy()) <= 1e-2


def test_rmsnorm_bf16_grad_weight(dev):
    # FLCE_GW_BF16 on the fused-RMSNorm entry point: the same fp32 accumulation, rounded once
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    p = wl.random_problem(600, 128, 900, seed=5, ignore_frac=0.1, hidden_std=3.0)
    g = _gain(128, 5)
    h, w, t = to_device(p, dev)
    gt = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).to(dev)
    a = flce.rmsnorm_fwd_bwd(h, gt, w, t)
    b = flce.rmsnorm_fwd_bwd(h, gt, w, t, grad_weight_dtype=torch.bfloat16)
    assert flce.query_status(b["workspace"]) == flce.FLCE_OK
    assert b["grad_weight"].dtype == torch.bfloat16
    assert torch.equal(b["grad_weight"], a["grad_weight"].to(torch.bfloat16))
    assert torch.equal(a["grad_hidden"], b["grad_hidden"]) and torch.equal(a["grad_gain"], b["grad_gain"])
    ref = rmsnorm_flce_oracle(p["hidden"], g, p["weight"], p["targets"], 1e-6)
    assert frob_rel(b["grad_weight"].double().cpu().numpy(), ref["grad_weight"]) <= GRAD_FROB_RTOL
