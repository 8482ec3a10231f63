"""GPU parity: libflce through its C ABI against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation): loss relative error <= 2e-3,
grad_hidden / grad_weight relative Frobenius error <= 1e-2, n_valid exact,
grad_hidden rows of ignored tokens exactly +0.0.

Small problems are compared element by element; they span several 128-row
and 256-column tiles, force several token chunks, and leave ragged tails in
N, H and V.  The full-size workloads run in the launch configuration the
benchmark uses and are checked on sampled rows the oracle computes one by
one, plus properties that hold at any size.
"""
import json
import math
import os

import numpy as np
import pytest

from linear_cross_entropy_ce_gb300 import workloads as wl
from oracle import flce_oracle, oracle_rows, lse_all_rows, grad_weight_rows, decode_bf16
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


def _flce():
    from linear_cross_entropy_ce_gb300 import flce
    return flce


def report(case, **errors):
    """Append the measured errors of a parity case to $FLCE_PARITY_REPORT (JSON lines), if set."""
    path = os.environ.get("FLCE_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": case, **{k: float(v) for k, v in errors.items()}}) + "\n")


def check_full(p, dev, chunk_rows=None, reduction="mean", case=None):
    flce = _flce()
    h, w, t = to_device(p, dev)
    out = flce.fwd_bwd(h, w, t, reduction=reduction, chunk_rows=chunk_rows, row_loss=True)
    assert flce.query_status(out["workspace"]) == flce.FLCE_OK
    ref = flce_oracle(p["hidden"], p["weight"], p["targets"], reduction=reduction)
    nv = int(out["n_valid"].item())
    assert nv == ref["n_valid"]
    loss = float(out["loss"].item())
    if ref["loss"] != 0:
        assert loss_rel(loss, ref["loss"]) <= LOSS_RTOL, (loss, ref["loss"])
    else:
        assert abs(loss) <= 1e-6
    gh = gh_np(out["grad_hidden"])
    gw = out["grad_weight"].cpu().double().numpy()
    assert np.all(np.isfinite(gh)) and np.all(np.isfinite(gw))
    e_gh, e_gw = frob_rel(gh, ref["grad_hidden"]), frob_rel(gw, ref["grad_weight"])
    assert e_gh <= GRAD_FROB_RTOL
    assert e_gw <= GRAD_FROB_RTOL
    if case:
        report(case, loss=loss_rel(loss, ref["loss"]) if ref["loss"] else abs(loss), grad_hidden=e_gh,
               grad_weight=e_gw)
    ign = p["targets"] == -100
    if ign.any():
        import torch
        bits = out["grad_hidden"].view(torch.int16)[torch.from_numpy(ign).to(dev)]
        assert int(bits.abs().max().item()) == 0          # exactly +0.0
    rl = out["row_loss"].cpu().double().numpy()
    assert np.all(rl[ign] == 0.0)
    assert np.max(np.abs(rl - ref["row_loss"])) <= LOSS_RTOL * max(1.0, np.abs(ref["row_loss"]).max())
    return out, ref


# --------------------------------------------------------------------------
# element-by-element cases
# --------------------------------------------------------------------------

def test_tiny_workload(dev):
    check_full(wl.make_inputs(wl.WORKLOADS["tiny"]), dev, case="tiny")


@pytest.mark.parametrize("N,H,V,ign,chunk,seed", [
    (1000, 200, 1000, 0.1, 128, 1),    # 8 chunks, ragged H tile and V tail
    (300, 64, 512, 0.0, 128, 2),       # 3 chunks, last one 44 rows
    (130, 64, 7, 0.0, 128, 3),         # V narrower than one TMA box
    (1, 8, 300, 0.0, None, 4),         # one token, smallest H
    (257, 8, 5000, 0.3, 128, 5),       # H = 8: one K block, mostly padding
    (256, 1024, 2000, 0.05, None, 6),  # 16 K blocks, one chunk
    (640, 256, 3001, 0.5, 256, 7),     # half the tokens ignored, odd V
    (64, 8192, 300, 0.0, None, 20),    # wide hidden size: 128 K blocks, 32 grad_hidden column tiles
    (20000, 64, 50, 0.3, None, 21),    # many tokens, a tiny vocabulary: 20 compaction tiles, V inside one tile
    (2600, 136, 20000, 0.1, 1536, 22), # two chunks of 6 and 5 row blocks x 79 vocabulary tiles, ragged H and V
    (1200, 512, 16000, 0.05, 768, 23), # the full-model H and V in 768-row chunks, a 432-row last chunk
])
def test_ragged_shapes(dev, N, H, V, ign, chunk, seed):
    check_full(wl.random_problem(N, H, V, seed=seed, ignore_frac=ign), dev, chunk_rows=chunk)


def test_vocab_of_one(dev):
    out, ref = check_full(wl.random_problem(40, 16, 1, seed=8), dev)
    assert float(out["loss"].item()) == 0.0


def test_all_ignored(dev):
    flce = _flce()
    p = wl.random_problem(64, 32, 100, seed=9)
    p["targets"][:] = -100
    h, w, t = to_device(p, dev)
    out = flce.fwd_bwd(h, w, t, row_loss=True)
    assert flce.query_status(out["workspace"]) == flce.FLCE_OK
    assert int(out["n_valid"].item()) == 0 and float(out["loss"].item()) == 0.0
    assert out["grad_hidden"].float().abs().max().item() == 0.0
    assert out["grad_weight"].abs().max().item() == 0.0


def test_reduction_sum(dev):
    check_full(wl.random_problem(500, 128, 700, seed=10, ignore_frac=0.2), dev, chunk_rows=128,
               reduction="sum")


def test_forward_only_matches(dev):
    flce = _flce()
    p = wl.random_problem(700, 192, 1500, seed=11, ignore_frac=0.1)
    h, w, t = to_device(p, dev)
    out = flce.loss(h, w, t, row_loss=True)
    assert flce.query_status(out["workspace"]) == flce.FLCE_OK
    ref = flce_oracle(p["hidden"], p["weight"], p["targets"], want_grads=False)
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert loss_rel(float(out["loss"].item()), ref["loss"]) <= LOSS_RTOL
    fb = flce.fwd_bwd(h, w, t)
    assert abs(float(out["loss"].item()) - float(fb["loss"].item())) <= 1e-6 * abs(ref["loss"])


def test_deterministic(dev):
    flce = _flce()
    p = wl.random_problem(1000, 200, 1000, seed=12, ignore_frac=0.1)
    h, w, t = to_device(p, dev)
    a = flce.fwd_bwd(h, w, t, chunk_rows=128, row_loss=True)
    b = flce.fwd_bwd(h, w, t, chunk_rows=128, row_loss=True)
    import torch
    for k in ("loss", "n_valid", "row_loss", "grad_hidden", "grad_weight"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("N,H,V,chunk", [
    (2048, 512, 20000, None),   # default 5% plan: 128-row chunks, the grad_hidden GEMM split over the vocabulary
    (1536, 1024, 12000, 768),   # two 768-row chunks, unsplit grad_hidden GEMM, many short grad_weight tiles
])
def test_repeated_calls_bitwise(dev, N, H, V, chunk):
    # The tile scheduler is dynamic (CTA pairs claim tiles from a counter and
    # hand them to the peer CTA), so every call runs a different interleaving;
    # the results must not change by a bit, and every call must end with an
    # OK status.
    flce = _flce()
    import torch
    p = wl.random_problem(N, H, V, seed=31, ignore_frac=0.1)
    h, w, t = to_device(p, dev)
    ref = flce.fwd_bwd(h, w, t, chunk_rows=chunk)
    assert flce.query_status(ref["workspace"]) == flce.FLCE_OK
    ref = {k: v.clone() for k, v in ref.items() if k != "workspace" and isinstance(v, torch.Tensor)}
    out = None
    for _ in range(20):
        out = flce.fwd_bwd(h, w, t, chunk_rows=chunk, out=out)
        assert flce.query_status(out["workspace"]) == flce.FLCE_OK
        for k in ("loss", "n_valid", "grad_hidden", "grad_weight"):
            assert torch.equal(out[k], ref[k]), k


def test_ignored_rows_do_not_matter(dev):
    flce = _flce()
    import torch
    p = wl.random_problem(600, 128, 900, seed=13, ignore_frac=0.25)
    h, w, t = to_device(p, dev)
    a = flce.fwd_bwd(h, w, t, chunk_rows=128)
    ign = torch.from_numpy(p["targets"] == -100).to(dev)
    h2 = h.clone()
    h2[ign] = 100.0
    b = flce.fwd_bwd(h2, w, t, chunk_rows=128)
    assert torch.equal(a["loss"], b["loss"]) and torch.equal(a["grad_weight"], b["grad_weight"])
    assert torch.equal(a["grad_hidden"], b["grad_hidden"])


def test_component_workload_full(dev):
    # B=4, S=1024, H=512, V=16000 with 5% ignored, default (5%) plan
    check_full(wl.make_inputs(wl.WORKLOADS["component"]), dev, case="component")


# --------------------------------------------------------------------------
# device-side errors: recorded in the status word, the context stays usable
# --------------------------------------------------------------------------

def test_bad_target_status(dev):
    flce = _flce()
    p = wl.random_problem(100, 32, 50, seed=14)
    p["targets"][17] = 50
    h, w, t = to_device(p, dev)
    out = flce.fwd_bwd(h, w, t)
    assert flce.query_status(out["workspace"]) == flce.FLCE_EBADTARGET
    assert math.isnan(float(out["loss"].item()))        # a failed call reports a NaN loss
    p["targets"][17] = -7
    h, w, t = to_device(p, dev)
    out = flce.fwd_bwd(h, w, t)
    assert flce.query_status(out["workspace"]) == flce.FLCE_EBADTARGET
    assert math.isnan(float(out["loss"].item()))
    p["targets"][17] = 3                                 # the same workspace, a good call: status cleared
    h, w, t = to_device(p, dev)
    out = flce.fwd_bwd(h, w, t, workspace=out["workspace"])
    assert flce.query_status(out["workspace"]) == flce.FLCE_OK
    assert math.isfinite(float(out["loss"].item()))


def test_timeout_path_returns(dev):
    flce = _flce()
    import torch
    ws = torch.empty(4096, dtype=torch.uint8, device=dev)
    assert flce.selftest_timeout(ws, 20_000_000) == flce.FLCE_OK      # 20 ms
    assert flce.query_status(ws) == flce.FLCE_ETIMEOUT
    check_full(wl.random_problem(64, 32, 100, seed=15), dev)          # context still healthy


W_TMEM_FULL = 10   # wait site: an epilogue waiting for its accumulator (flce_query_stall)


def test_gemm_pipeline_timeout(dev):
    # The tcgen05 GEMM's own failure path: the armed launch (the first logits
    # launch of the call) withholds the accumulator-ready signal of the first
    # tile of every CTA pair, the epilogues' bounded waits run out after 50 ms,
    # and every CTA aborts (drains its copies, waits for its MMAs, frees TMEM).
    flce = _flce()
    p = wl.random_problem(300, 64, 512, seed=16)
    h, w, t = to_device(p, dev)
    flce.debug_arm_stall(50_000_000)
    out = flce.fwd_bwd(h, w, t)
    assert flce.query_status(out["workspace"]) == flce.FLCE_ETIMEOUT
    st = flce.query_stall(out["workspace"])
    assert st["site"] == W_TMEM_FULL and st["count"] >= 1, st
    assert math.isnan(float(out["loss"].item()))
    # the same workspace and context: the next call is normal
    out = flce.fwd_bwd(h, w, t, workspace=out["workspace"])
    assert flce.query_status(out["workspace"]) == flce.FLCE_OK
    assert flce.query_stall(out["workspace"])["site"] == 0
    check_full(p, dev)


def test_grad_weight_bf16(dev):
    # FLCE_GW_BF16: the same fp32 accumulation, rounded once to bf16 at the end
    flce = _flce()
    import torch
    p = wl.random_problem(1000, 200, 1000, seed=17, ignore_frac=0.1)
    h, w, t = to_device(p, dev)
    a = flce.fwd_bwd(h, w, t, chunk_rows=128)
    b = flce.fwd_bwd(h, w, t, chunk_rows=128, grad_weight_dtype=torch.bfloat16)
    assert flce.query_status(b["workspace"]) == flce.FLCE_OK
    assert b["grad_weight"].dtype == torch.bfloat16
    assert torch.equal(b["grad_weight"], a["grad_weight"].to(torch.bfloat16))
    assert torch.equal(a["grad_hidden"], b["grad_hidden"]) and torch.equal(a["loss"], b["loss"])
    ref = flce_oracle(p["hidden"], p["weight"], p["targets"])
    e = frob_rel(b["grad_weight"].double().cpu().numpy(), ref["grad_weight"])
    assert e <= GRAD_FROB_RTOL
    report("grad_weight_bf16", grad_weight=e)


# --------------------------------------------------------------------------
# full-size workloads, default plan (the benchmark's launch configuration)
# --------------------------------------------------------------------------

def _vocab_rows(p, V, n_min=32):
    """Vocabulary rows of grad_weight to compare with the oracle: the first and
    last rows, both sides of 128-column part and 256-row tile boundaries, the
    last (possibly partial) 256-row tile, the 8 most frequent targets, and
    seeded random rows up to n_min."""
    t = p["targets"]
    freq = np.bincount(t[t != -100], minlength=V)
    rows = {0, 1, V - 2, V - 1}
    for b in (128, 256, 384, 512, (V // 2) // 128 * 128):
        rows.update(v for v in (b - 1, b) if 0 <= v < V)
    last_tile = (V - 1) // 256 * 256
    rows.update(range(max(last_tile, V - 8), V))      # every row of a partial last tile (V=256007: 7 rows)
    rows.update(int(v) for v in np.argsort(-freq, kind="stable")[:8])
    rng = np.random.default_rng(V)
    while len(rows) < n_min:
        rows.add(int(rng.integers(0, V)))
    return np.array(sorted(rows))


def _sampled(name, dev, n_rows=24, reduce=None):
    """One call of the default plan (the benchmark's launch configuration) at a
    full-size workload, compared with the fp64 oracle on:
      * the total loss (every valid row's log-sum-exp from the oracle),
      * >= 32 rows of grad_weight (every valid row contributes to each),
      * grad_hidden and the per-row loss on the first and last valid row of
        every token chunk plus seeded random rows and two ignored rows,
    plus two properties that hold at any size."""
    flce = _flce()
    import torch
    w_ = wl.WORKLOADS[name] if reduce is None else wl.WORKLOADS[name].with_shape(**reduce)
    p = wl.make_inputs(w_)
    h, w, t = to_device(p, dev)
    N, H, V = w_.N, w_.H, w_.V
    C = flce.plan(N, H, V, flce.workspace_bytes(N, H, V))["chunk_rows"]
    out = flce.fwd_bwd(h, w, t, row_loss=True)
    assert flce.query_status(out["workspace"]) == flce.FLCE_OK
    nv = int(out["n_valid"].item())
    assert nv == int((p["targets"] != -100).sum())
    rng = np.random.default_rng(123)
    valid = np.nonzero(p["targets"] != -100)[0]
    ign = np.nonzero(p["targets"] == -100)[0]
    edges = [valid[c0] for c0 in range(0, valid.size, C)] + \
            [valid[min(c0 + C, valid.size) - 1] for c0 in range(0, valid.size, C)]
    rows = np.unique(np.concatenate([rng.choice(valid, size=min(n_rows, valid.size), replace=False),
                                     ign[:2], np.array(edges, dtype=np.int64)]))
    W64 = decode_bf16(p["weight"])
    ref = oracle_rows(p["hidden"][rows], p["weight"], p["targets"][rows], nv, weight_f64=W64)
    rl = out["row_loss"][torch.from_numpy(rows).to(dev)].cpu().double().numpy()
    e_rl = np.max(np.abs(rl - ref["row_loss"])) / np.abs(ref["row_loss"]).max()
    assert e_rl <= LOSS_RTOL
    gh = gh_np(out["grad_hidden"][torch.from_numpy(rows).to(dev)])
    e_gh = frob_rel(gh, ref["grad_hidden"])
    assert e_gh <= GRAD_FROB_RTOL
    for i, r in enumerate(rows):
        if p["targets"][r] != -100:
            assert frob_rel(gh[i], ref["grad_hidden"][i]) <= 3 * GRAD_FROB_RTOL, r
        else:
            assert not gh[i].any()
    gw = out["grad_weight"]
    # softmax rows sum to one, so the columns of grad_weight sum to zero
    col = gw.double().sum(dim=0)
    assert (col.norm() / gw.double().norm()).item() <= GRAD_FROB_RTOL
    # <dX, X> = <dW, W> = sum_nv dz_nv z_nv  (both are d/da of L(aX, W) = L(X, aW) at a = 1)
    a = (out["grad_hidden"].double() * h.double()).sum().item()
    b = (gw.double() * w.double()).sum().item()
    assert abs(a - b) <= GRAD_FROB_RTOL * max(abs(a), abs(b)), (a, b)
    # total loss and grad_weight rows against the oracle (needs every row's lse)
    lse = lse_all_rows(p["hidden"], p["weight"], p["targets"], weight_f64=W64)
    vr = _vocab_rows(p, V)
    assert vr.size >= 32
    ew = grad_weight_rows(p["hidden"], p["weight"], p["targets"], lse, vr, weight_f64=W64)
    got = gw[torch.from_numpy(vr).to(dev)].cpu().double().numpy()
    e_gw = frob_rel(got, ew)
    assert e_gw <= GRAD_FROB_RTOL
    X64 = decode_bf16(p["hidden"][valid])
    zt = (X64 * W64[p["targets"][valid]]).sum(axis=1)
    ref_loss = float((lse[valid] - zt).sum()) / nv
    e_loss = loss_rel(float(out["loss"].item()), ref_loss)
    assert e_loss <= LOSS_RTOL
    report(name, loss=e_loss, row_loss=e_rl, grad_hidden_rows=e_gh, grad_weight_rows=e_gw,
           n_grad_hidden_rows=rows.size, n_grad_weight_rows=vr.size, chunk_rows=C)
    return out


def test_full_model_workload(dev):
    _sampled("full_model", dev)


def test_llama3_head_workload(dev):
    _sampled("llama3_8b_head", dev)


def test_large_vocab_workload(dev):
    _sampled("large_vocab", dev)


def test_large_vocab_tail_workload(dev):
    _sampled("large_vocab_tail", dev)


@pytest.mark.parametrize("name,N", [("llama3_8b_head", 300), ("large_vocab_tail", 600)])
def test_full_vocab_reduced_tokens(dev, name, N):
    # full H and V of the big workloads, fewer tokens so the oracle runs whole;
    # 128-row chunks exercise the fp32 grad_weight accumulation at full V
    check_full(wl.make_inputs(wl.WORKLOADS[name].with_shape(N=N)), dev, chunk_rows=128, case=f"{name}_N{N}")


def test_concurrent_calls_on_two_streams(dev):
    # Calls are reentrant: two problems enqueued on two streams at once, each
    # with its own workspace and outputs, give bitwise the results of the same
    # calls made one after the other (the tile counters and split flags live
    # in each call's workspace; no kernel waits on another launch).
    flce = _flce()
    import torch
    pa = wl.random_problem(1000, 256, 3000, seed=18, ignore_frac=0.1)
    pb = wl.random_problem(700, 128, 5000, seed=19, ignore_frac=0.2)
    ha, wa, ta = to_device(pa, dev)
    hb, wb, tb = to_device(pb, dev)
    ref_a = flce.fwd_bwd(ha, wa, ta, chunk_rows=256, row_loss=True)
    ref_b = flce.fwd_bwd(hb, wb, tb, chunk_rows=128, row_loss=True)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    for _ in range(3):
        with torch.cuda.stream(s1):
            a = flce.fwd_bwd(ha, wa, ta, chunk_rows=256, row_loss=True, stream=s1)
        with torch.cuda.stream(s2):
            b = flce.fwd_bwd(hb, wb, tb, chunk_rows=128, row_loss=True, stream=s2)
        torch.cuda.synchronize()
        assert flce.query_status(a["workspace"]) == flce.FLCE_OK and flce.query_status(b["workspace"]) == flce.FLCE_OK
        for k in ("loss", "n_valid", "row_loss", "grad_hidden", "grad_weight"):
            assert torch.equal(a[k], ref_a[k]), k
            assert torch.equal(b[k], ref_b[k]), k
