"""flce_fwd_bwd captured in a CUDA graph.

A call only enqueues kernels on the caller's stream. It does not allocate or
synchronise, and the tile counters and split flags are reset by its first
kernel. A captured call therefore replays correctly after new inputs are
copied into the captured buffers. The result must match an eager call on those
inputs bit for bit, because the kernels reduce in a fixed order, and it must
match the fp64 oracle within the tolerances.
"""
import numpy as np
import pytest

from linear_cross_entropy_ce_gb300 import workloads as wl
from oracle import flce_oracle
from tests.helpers import LOSS_RTOL, GRAD_FROB_RTOL, to_device, frob_rel, loss_rel, gh_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_cross_entropy_ce_gb300 import flce
    try:
        flce.library()
    except RuntimeError:
        import __graft_entry__
        __graft_entry__.build()
    return flce, torch, torch.device("cuda:0")


@pytest.mark.parametrize("N,H,V,ign,chunk", [(1000, 512, 16000, 0.05, 256), (700, 256, 64000, 0.1, 128)])
def test_graph_replay_matches_eager_and_oracle(env, N, H, V, ign, chunk):
    flce, torch, dev = env
    p1 = wl.random_problem(N, H, V, seed=31, ignore_frac=ign)
    p2 = wl.random_problem(N, H, V, seed=32, ignore_frac=ign)
    h, w, t = to_device(p1, dev)
    ws = flce.new_workspace(flce.workspace_bytes(N, H, V, chunk_rows=chunk), dev)
    out = {}
    flce.fwd_bwd(h, w, t, workspace=ws, out=out, row_loss=True)   # first call sets up the device state
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        flce.fwd_bwd(h, w, t, workspace=ws, out=out, row_loss=True)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        flce.fwd_bwd(h, w, t, workspace=ws, out=out, row_loss=True)

    for p in (p2, p1):   # replay on new inputs, then on the first ones again
        h2, w2, t2 = to_device(p, dev)
        h.copy_(h2)
        w.copy_(w2)
        t.copy_(t2)
        g.replay()
        torch.cuda.synchronize()
        assert flce.query_status(ws) == flce.FLCE_OK
        eager = flce.fwd_bwd(h2, w2, t2, chunk_rows=chunk, row_loss=True)
        for k in ("loss", "n_valid", "row_loss", "grad_hidden", "grad_weight"):
            assert torch.equal(out[k], eager[k]), k
        ref = flce_oracle(p["hidden"], p["weight"], p["targets"])
        assert int(out["n_valid"].item()) == ref["n_valid"]
        assert loss_rel(float(out["loss"].item()), ref["loss"]) <= LOSS_RTOL
        assert frob_rel(gh_np(out["grad_hidden"]), ref["grad_hidden"]) <= GRAD_FROB_RTOL
        assert frob_rel(out["grad_weight"].cpu().double().numpy(), ref["grad_weight"]) <= GRAD_FROB_RTOL
