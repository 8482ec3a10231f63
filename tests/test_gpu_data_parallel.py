"""GPU: the data-parallel split of one batch over P simulated ranks.

Each "rank" calls flce_fwd_bwd with FLCE_REDUCE_SUM on its contiguous token
shard (sequential calls on one GPU, no kernel waits on another); the host then
does the exchange a data-parallel step would do with a collective -- sum of
the loss sums, of the valid counts and of grad_weight, in rank order -- and
rescales by 1/n_valid.  The result must match the unsplit mean call."""
import numpy as np
import pytest

from linear_cross_entropy_ce_gb300 import workloads as wl
from linear_cross_entropy_ce_gb300 import dist as fdist
from tests.helpers import to_device, frob_rel, gh_np

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


@pytest.mark.parametrize("world", [2, 3])
def test_token_shards_match_unsplit(dev, world):
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    p = wl.random_problem(1000, 256, 3000, seed=41, ignore_frac=0.15)
    h, w, t = to_device(p, dev)
    full = flce.fwd_bwd(h, w, t)
    loss_sum, n_valid = 0.0, 0
    gw = torch.zeros_like(full["grad_weight"], dtype=torch.float64)
    gh_parts = []
    for r in range(world):
        sl = fdist.shard_rows(1000, r, world)
        o = flce.fwd_bwd(h[sl].contiguous(), w, t[sl].contiguous(), reduction="sum")
        loss_sum += float(o["loss"].item())
        n_valid += int(o["n_valid"].item())
        gw += o["grad_weight"].double()
        gh_parts.append(o["grad_hidden"].double())
    assert n_valid == int(full["n_valid"].item())
    assert abs(loss_sum / n_valid - float(full["loss"].item())) <= 1e-5 * abs(float(full["loss"].item()))
    assert frob_rel((gw / n_valid).cpu().numpy(), full["grad_weight"].cpu().double().numpy()) <= 2e-3
    gh = torch.cat(gh_parts) / n_valid
    assert frob_rel(gh.cpu().numpy(), gh_np(full["grad_hidden"])) <= 1e-2
