"""flce_fwd_bwd_noalloc: the entry point for callers that cannot allocate
device memory (inside a graph capture or an allocator hook, or under a
memory budget fixed in advance).  Its scratch is a static device array in the
library, so it must give the same results as flce_fwd_bwd with a
caller-allocated workspace, call after call on the same shared array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

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
        lib = flce.library()
    except RuntimeError:
        import __graft_entry__
        __graft_entry__.build()
        lib = flce.library()
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    lib.flce_fwd_bwd_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i32, u32, vp, vp, vp, vp, vp, vp]
    lib.flce_fwd_bwd_noalloc.restype = ctypes.c_int
    return lib, flce, torch, torch.device("cuda:0")


def _noalloc(lib, torch, dev, h, w, t, N, H, V):
    out = {"loss": torch.full((1,), float("nan"), device=dev),
           "n_valid": torch.full((1,), -1, dtype=torch.int32, device=dev),
           "row_loss": torch.full((N,), float("nan"), device=dev),
           "grad_hidden": torch.full((N, H), float("nan"), dtype=torch.bfloat16, device=dev),
           "grad_weight": torch.full((V, H), float("nan"), dtype=torch.float32, device=dev)}
    p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    st = lib.flce_fwd_bwd_noalloc(p(h), p(w), p(t), N, H, V, -100, 0, p(out["loss"]), p(out["n_valid"]),
                                  p(out["row_loss"]), p(out["grad_hidden"]), p(out["grad_weight"]),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


@pytest.mark.parametrize("shape", [(1000, 200, 1000, 0.1, 21), (2048, 512, 16000, 0.05, 22)])
def test_noalloc_matches_workspace_entry(env, shape):
    lib, flce, torch, dev = env
    N, H, V, ign, seed = shape
    p = wl.random_problem(N, H, V, seed=seed, ignore_frac=ign)
    h, w, t = to_device(p, dev)
    ref = flce.fwd_bwd(h, w, t, row_loss=True)
    assert flce.query_status(ref["workspace"]) == flce.FLCE_OK
    orc = flce_oracle(p["hidden"], p["weight"], p["targets"])   # the fp64 definition, independent of both paths
    for _ in range(2):    # two calls in a row on the same static scratch
        st, out = _noalloc(lib, torch, dev, h, w, t, N, H, V)
        assert st == flce.FLCE_OK
        torch.cuda.synchronize()
        assert int(out["n_valid"].item()) == int(ref["n_valid"].item()) == orc["n_valid"]
        loss = float(out["loss"].item())
        assert loss_rel(loss, float(ref["loss"].item())) <= LOSS_RTOL
        assert loss_rel(loss, orc["loss"]) <= LOSS_RTOL
        rl, rr = out["row_loss"].cpu().double().numpy(), ref["row_loss"].cpu().double().numpy()
        assert np.max(np.abs(rl - rr)) <= LOSS_RTOL * max(1.0, np.abs(rr).max())
        assert np.max(np.abs(rl - orc["row_loss"])) <= LOSS_RTOL * max(1.0, np.abs(orc["row_loss"]).max())
        gh, gw = gh_np(out["grad_hidden"]), out["grad_weight"].cpu().double().numpy()
        assert frob_rel(gh, gh_np(ref["grad_hidden"])) <= GRAD_FROB_RTOL
        assert frob_rel(gw, ref["grad_weight"].cpu().double().numpy()) <= GRAD_FROB_RTOL
        assert frob_rel(gh, orc["grad_hidden"]) <= GRAD_FROB_RTOL
        assert frob_rel(gw, orc["grad_weight"]) <= GRAD_FROB_RTOL


def test_noalloc_rejects_sizes_beyond_its_scratch(env):
    lib, flce, torch, dev = env
    # one 128-token chunk of a 300000-word vocabulary needs ~77 MB of logits:
    # too big.  Every buffer is real and of the full size, so that the call
    # stays in bounds whatever it does before its size check.
    N, H, V = 256, 64, 300000
    h = torch.zeros((N, H), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((V, H), dtype=torch.bfloat16, device=dev)
    t = torch.zeros(N, dtype=torch.int32, device=dev)
    loss = torch.zeros(1, device=dev)
    nv = torch.zeros(1, dtype=torch.int32, device=dev)
    gh = torch.zeros((N, H), dtype=torch.bfloat16, device=dev)
    gw = torch.zeros((V, H), dtype=torch.float32, device=dev)
    p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    st = lib.flce_fwd_bwd_noalloc(p(h), p(w), p(t), N, H, V, -100, 0, p(loss), p(nv), None, p(gh), p(gw),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == flce.FLCE_EWORKSPACE
    torch.cuda.synchronize()
    assert int(nv.item()) == 0 and not gh.any().item()   # nothing was enqueued
