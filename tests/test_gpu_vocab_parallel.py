"""GPU: the vocabulary-parallel LM head, with P ranks simulated as sequential
calls on one GPU and the collectives played by the test in rank order.
Shards are uneven and not multiples of any tile; the result must match the
fp64 oracle of the unsharded loss."""
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


@pytest.mark.parametrize("N,H,V,bounds,ign,seed", [
    (600, 128, 3001, [0, 1000, 2001, 3001], 0.1, 51),
    (300, 512, 16000, [0, 8000, 16000], 0.0, 52),
    (257, 64, 700, [0, 256, 264, 700], 0.3, 53),
])
def test_vocab_parallel_matches_oracle(dev, N, H, V, bounds, ign, seed):
    import torch
    from linear_cross_entropy_ce_gb300 import flce
    p = wl.random_problem(N, H, V, seed=seed, ignore_frac=ign)
    h, w, t = to_device(p, dev)
    shards = [(a, b) for a, b in zip(bounds, bounds[1:])]
    stats = [flce.vocab_shard_stats(h, w[a:b].contiguous(), t, a, V) for a, b in shards]
    m_glob = stats[0]["row_max"].clone()
    for s in stats[1:]:
        m_glob = torch.maximum(m_glob, s["row_max"])          # all-reduce MAX
    for s in stats:
        flce.vocab_rescale(s["row_max"], m_glob, s["row_sumexp"])
    d = sum(s["row_sumexp"] for s in stats)                   # all-reduce SUM (rank order)
    zt = sum(s["row_target_logit"] for s in stats)
    fin = flce.vocab_finish(m_glob, d, zt, t)
    parts = [flce.vocab_shard_bwd(h, w[a:b].contiguous(), t, fin["lse"], a, V) for a, b in shards]
    gh = sum(q["grad_hidden_partial"].double() for q in parts)   # all-reduce SUM
    gw = torch.cat([q["grad_weight"] for q in parts]).double()
    ref = flce_oracle(p["hidden"], p["weight"], p["targets"])
    assert int(fin["n_valid"].item()) == ref["n_valid"]
    assert all(int(s["n_valid"].item()) == ref["n_valid"] for s in stats)
    assert loss_rel(float(fin["loss"].item()), ref["loss"]) <= LOSS_RTOL
    rl = fin["row_loss"].cpu().double().numpy()
    assert np.max(np.abs(rl - ref["row_loss"])) <= LOSS_RTOL * max(1.0, np.abs(ref["row_loss"]).max())
    assert frob_rel(gh.cpu().numpy(), ref["grad_hidden"]) <= GRAD_FROB_RTOL
    assert frob_rel(gw.cpu().numpy(), ref["grad_weight"]) <= GRAD_FROB_RTOL
    ign_rows = torch.from_numpy(p["targets"] == -100).to(dev)
    if bool(ign_rows.any()):
        assert float(gh[ign_rows].abs().max().item()) == 0.0
