"""Pins for the fp64 oracle of the final RMSNorm fused in front of the LM head.

* PyTorch CPU autograd in fp64 of the unfused composition (normalise, scale
  by the gain, linear, cross_entropy with ignore_index).
* Central finite differences on a tiny problem.
* With eps = 0, RMSNorm is invariant to scaling a row of h, so the loss does
  not change and each gradient row is orthogonal to its hidden row.
* A planted mistake (the projection term dropped from dh) is caught.
"""
import numpy as np
import pytest

import oracle.flce_fp64 as ofl
from oracle import rmsnorm_flce_oracle_f64


def _problem(N, H, V, seed, ign=0):
    rng = np.random.default_rng(seed)
    Hs = rng.standard_normal((N, H)) * 2.0
    g = 1.0 + 0.3 * rng.standard_normal(H)
    W = rng.standard_normal((V, H)) * 0.4
    t = rng.integers(0, V, size=N).astype(np.int32)
    if ign:
        t[rng.choice(N, size=ign, replace=False)] = -100
    return Hs, g, W, t


def _torch_ref(Hs, g, W, t, eps, red):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    h = torch.tensor(Hs, requires_grad=True)
    gg = torch.tensor(g, requires_grad=True)
    w = torch.tensor(W, requires_grad=True)
    x = h * torch.rsqrt(h.pow(2).mean(-1, keepdim=True) + eps) * gg
    loss = F.cross_entropy(x @ w.T, torch.tensor(t, dtype=torch.long), ignore_index=-100, reduction=red)
    loss.backward()
    return loss.item(), h.grad.numpy(), gg.grad.numpy(), w.grad.numpy()


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def check_against_torch(orc):
    for (N, H, V, seed, ign, eps, red) in [(9, 8, 13, 1, 2, 1e-6, "mean"), (20, 16, 7, 2, 0, 1e-2, "sum"),
                                            (5, 4, 30, 3, 1, 0.0, "mean")]:
        Hs, g, W, t = _problem(N, H, V, seed, ign)
        l, dh, dg, dw = _torch_ref(Hs, g, W, t, eps, red)
        o = orc(Hs, g, W, t, eps, -100, red)
        if abs(o["loss"] - l) > 1e-12 * max(1, abs(l)):
            return False
        if _rel(o["grad_hidden"], dh) > 1e-11 or _rel(o["grad_gain"], dg) > 1e-11 or _rel(o["grad_weight"], dw) > 1e-11:
            return False
    return True


def check_finite_differences(orc):
    Hs, g, W, t = _problem(4, 3, 5, 7, 1)
    eps_fd = 1e-6
    o = orc(Hs, g, W, t, 1e-3)
    for name, A, G in (("h", Hs, o["grad_hidden"]), ("g", g, o["grad_gain"])):
        for idx in np.ndindex(A.shape):
            Ap, Am = A.copy(), A.copy()
            Ap[idx] += eps_fd
            Am[idx] -= eps_fd
            args_p = (Ap, g) if name == "h" else (Hs, Ap)
            args_m = (Am, g) if name == "h" else (Hs, Am)
            fd = (orc(*args_p, W, t, 1e-3)["loss"] - orc(*args_m, W, t, 1e-3)["loss"]) / (2 * eps_fd)
            if abs(fd - G[idx]) > 1e-7 * max(1.0, abs(G[idx])):
                return False
    return True


def check_scale_invariance(orc):
    Hs, g, W, t = _problem(12, 16, 9, 11, 3)
    a = orc(Hs, g, W, t, 0.0)
    c = np.exp(np.random.default_rng(5).standard_normal(12))[:, None]
    b = orc(Hs * c, g, W, t, 0.0)
    if abs(a["loss"] - b["loss"]) > 1e-12:
        return False
    dots = np.abs((a["grad_hidden"] * Hs).sum(axis=1))
    return bool(np.all(dots <= 1e-12 * np.linalg.norm(a["grad_hidden"]) * np.linalg.norm(Hs)))


PINS = [check_against_torch, check_finite_differences, check_scale_invariance]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_rmsnorm_oracle_pin(pin):
    assert pin(rmsnorm_flce_oracle_f64)


def test_planted_mistake_caught(monkeypatch):
    def wrong_backward(dX, xhat, r, gain):
        return r[:, None] * dX * gain[None, :], (dX * xhat).sum(axis=0)   # projection term dropped
    monkeypatch.setattr(ofl, "rmsnorm_backward", wrong_backward)
    assert not all(p(ofl.rmsnorm_flce_oracle_f64) for p in PINS)
