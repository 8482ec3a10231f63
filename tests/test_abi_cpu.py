"""C-ABI checks that need no GPU: the library loads, exports every entry
point that include/flce.h declares, plans workspaces within the memory
budget, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")


@pytest.fixture(scope="module")
def lib():
    from linear_cross_entropy_ce_gb300 import flce
    try:
        return flce.library()
    except RuntimeError:
        import __graft_entry__
        __graft_entry__.build()
        return flce.library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert "flce_fwd_bwd" in names and "flce_loss" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in flce.h but not exported"


def test_version_and_strings(lib):
    from linear_cross_entropy_ce_gb300 import flce
    assert flce.version() == "0.1.0"
    for s in range(7):
        assert len(lib.flce_status_string(s)) > 0


WORKLOADS = {"component": (4096, 512, 16000), "full_model": (65536, 512, 16000),
             "llama3_8b_head": (16384, 4096, 128256), "large_vocab": (8192, 2048, 256000),
             "large_vocab_tail": (8192, 2048, 256007)}


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_default_workspace_within_five_percent(lib, name):
    from linear_cross_entropy_ce_gb300 import flce
    N, H, V = WORKLOADS[name]
    nb = flce.workspace_bytes(N, H, V)
    assert nb <= 0.05 * N * V * 2
    p = flce.plan(N, H, V, nb)
    assert p["workspace_bytes"] <= nb
    assert p["chunk_rows"] % 128 == 0 and p["chunk_rows"] >= 128
    assert p["max_chunks"] * p["chunk_rows"] >= N
    assert p["logits_row_stride"] >= V and p["logits_row_stride"] % 64 == 0
    assert p["vocab_tiles"] == -(-V // 256)


# Default plans at the benchmark workloads (76 CTA pairs assumed when no GPU is
# visible): chunk rows and grad_hidden vocabulary splits.  The Llama-3-8B head
# has no room for the split accumulator inside 5% of its logits; the component
# shape cannot spread its split units through the few grad_weight units, so
# the split count balances unit length against the ordered chain of splits.
PLANS = {"component": (128, 4), "full_model": (2944, 2), "llama3_8b_head": (768, 1), "large_vocab": (384, 16),
         "large_vocab_tail": (384, 16)}


@pytest.mark.parametrize("name", sorted(PLANS))
def test_default_plans(lib, name):
    from linear_cross_entropy_ce_gb300 import flce
    N, H, V = WORKLOADS[name]
    p = flce.plan(N, H, V, flce.workspace_bytes(N, H, V))
    assert (p["chunk_rows"], p["dx_splits"]) == PLANS[name]


def test_plan_monotone_and_minimum(lib):
    from linear_cross_entropy_ce_gb300 import flce
    N, H, V = 1000, 64, 3000
    small = flce.workspace_bytes(N, H, V, chunk_rows=128)
    big = flce.workspace_bytes(N, H, V, chunk_rows=1024)
    assert big > small
    assert flce.plan(N, H, V, small)["chunk_rows"] == 128
    assert flce.plan(N, H, V, big)["chunk_rows"] == 1024
    with pytest.raises(flce.FlceError) as e:
        flce.plan(N, H, V, 4096)
    assert e.value.status == flce.FLCE_EWORKSPACE
    # forward-only needs no logits buffer: the same bytes hold a larger chunk
    f = flce.workspace_bytes(N, H, V)
    assert flce.plan(N, H, V, f, forward_only=True)["chunk_rows"] >= flce.plan(N, H, V, f)["chunk_rows"]


def test_bad_arguments_rejected_on_host(lib):
    from linear_cross_entropy_ce_gb300 import flce
    vp = ctypes.c_void_p
    good = vp(1 << 20)
    args = dict(h=good, w=good, t=good, N=16, H=64, V=32, ii=-100, fl=0, loss=good, nv=good, rl=None,
                gh=good, gw=good, ws=good, wsb=1 << 20, st=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.flce_fwd_bwd(a["h"], a["w"], a["t"], a["N"], a["H"], a["V"], a["ii"], a["fl"], a["loss"],
                                a["nv"], a["rl"], a["gh"], a["gw"], a["ws"], a["wsb"], a["st"])
    assert call(h=None) == flce.FLCE_EINVAL
    assert call(gw=None) == flce.FLCE_EINVAL
    assert call(ws=None) == flce.FLCE_EINVAL
    assert call(N=0) == flce.FLCE_EINVAL
    assert call(V=0) == flce.FLCE_EINVAL
    assert call(fl=4) == flce.FLCE_EINVAL
    assert call(H=60) == flce.FLCE_EUNSUPPORTED
    assert call(h=vp((1 << 20) + 8)) == flce.FLCE_EUNSUPPORTED
    assert call(w=vp((1 << 20) + 2)) == flce.FLCE_EUNSUPPORTED
    assert call(gh=vp((1 << 20) + 4)) == flce.FLCE_EUNSUPPORTED
    assert lib.flce_workspace_bytes(0, 64, 32, 0) == 0
    assert lib.flce_workspace_bytes(16, 63, 32, 0) == 0
    assert lib.flce_query_status(None, None) == flce.FLCE_EINVAL
    assert lib.flce_selftest_timeout(None, 1000, None) == flce.FLCE_EINVAL


def test_bf16_grad_weight_flag_sizes_and_rules(lib):
    # FLCE_GW_BF16 adds the fp32 V x H accumulator of grad_weight to the default plan
    from linear_cross_entropy_ce_gb300 import flce
    import torch
    for N, H, V in [(1000, 64, 3000), WORKLOADS["llama3_8b_head"]]:
        base = flce.workspace_bytes(N, H, V)
        with_acc = flce.workspace_bytes(N, H, V, grad_weight_dtype=torch.bfloat16)
        assert with_acc - base >= V * H * 4
        assert flce.plan(N, H, V, with_acc, grad_weight_dtype=torch.bfloat16)["chunk_rows"] == \
            flce.plan(N, H, V, base)["chunk_rows"]
        # the fp32 plan's bytes are too few once the accumulator is needed
        with pytest.raises(flce.FlceError):
            flce.plan(N, H, V, base, grad_weight_dtype=torch.bfloat16)
    vp = ctypes.c_void_p
    g = vp(1 << 20)
    # forward-only and vocabulary-shard calls have no grad_weight to round
    assert lib.flce_loss(g, g, g, 16, 64, 32, -100, flce.FLCE_GW_BF16, g, g, None, g, 1 << 20, None) == \
        flce.FLCE_EINVAL
    assert lib.flce_loss_workspace_bytes(16, 64, 32, flce.FLCE_GW_BF16) == 0


def test_debug_and_stall_entry_points_reject_bad_arguments(lib):
    from linear_cross_entropy_ce_gb300 import flce
    assert lib.flce_debug_arm_stall(0) == flce.FLCE_EINVAL
    assert lib.flce_debug_arm_stall(20_000_000_000) == flce.FLCE_EINVAL
    info = (ctypes.c_int32 * 4)()
    assert lib.flce_query_stall(None, info, None) == flce.FLCE_EINVAL
    assert lib.flce_query_stall(ctypes.c_void_p(1 << 20), None, None) == flce.FLCE_EINVAL
