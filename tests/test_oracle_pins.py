"""Pins for the fp64 oracle: each check ties it to something other than itself.

* PyTorch's CPU ``F.cross_entropy(..., ignore_index)`` plus autograd in fp64
  (the library routine that "Alisa's book of LLMs" uses in its
  "implementing the loss" code).
* Exact symbolic differentiation (sympy) of the loss written from its
  definition, independent of the softmax-minus-onehot formula.
* Central finite differences ("Backpropagation" section, manual gradient
  checking: recompute the loss at theta +- eps).
* Closed forms: zero weight gives loss = ln V; hand-derived tiny examples
  (tests/golden/closed_form_examples.json).
* Invariants: softmax rows sum to one so the column sums of grad_weight
  vanish; log-sum-exp is shift invariant ("Numerical stability and other
  tricks"); ignored tokens contribute nothing; the mean splits linearly over
  token subsets (mean-reduction paragraph).

The last test plants plausible mistakes in the oracle (on the CPU) and checks
that at least one pin catches each of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle.flce_fp64 as ofl
from oracle import flce_oracle, flce_oracle_f64, oracle_rows, lse_all_rows, grad_weight_rows
from linear_cross_entropy_ce_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_examples.json")


def _rand_f64(N, H, V, seed, ignore=0, wstd=0.5):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H)) * wstd
    t = rng.integers(0, V, size=N).astype(np.int32)
    if ignore:
        t[rng.choice(N, size=ignore, replace=False)] = -100
    return X, W, t


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.linalg.norm((a - b).ravel())
    n = np.linalg.norm(b.ravel())
    return d / n if n > 0 else d


# --------------------------------------------------------------------------
# pin checks: each returns (ok, message) for a given oracle callable
# --------------------------------------------------------------------------

def pin_torch(orc):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    cases = [(128, 64, 512, 0, 0), (7, 5, 11, 1, 2), (16, 8, 3, 2, 5), (1, 4, 9, 3, 0),
             (33, 16, 40, 4, 10)]
    for N, H, V, seed, ign in cases:
        X, W, t = _rand_f64(N, H, V, seed, ign)
        for red in ("mean", "sum"):
            Xt = torch.tensor(X, requires_grad=True)
            Wt = torch.tensor(W, requires_grad=True)
            loss = F.cross_entropy(Xt @ Wt.T, torch.tensor(t, dtype=torch.long),
                                   ignore_index=-100, reduction=red)
            loss.backward()
            o = orc(X, W, t, -100, red)
            if abs(o["loss"] - loss.item()) > 1e-12 * max(1.0, abs(loss.item())):
                return False, f"torch loss {N},{H},{V},{red}"
            if _rel(o["grad_hidden"], Xt.grad.numpy()) > 1e-12:
                return False, f"torch grad_hidden {N},{H},{V},{red}"
            if _rel(o["grad_weight"], Wt.grad.numpy()) > 1e-12:
                return False, f"torch grad_weight {N},{H},{V},{red}"
    return True, ""


def pin_sympy(orc):
    sp = pytest.importorskip("sympy")
    N, H, V = 3, 2, 4
    t = [1, -100, 3]
    rng = np.random.default_rng(11)
    Xq = [[sp.Rational(int(v), 8) for v in row] for row in rng.integers(-16, 16, (N, H))]
    Wq = [[sp.Rational(int(v), 8) for v in row] for row in rng.integers(-16, 16, (V, H))]
    xs = sp.symbols(f"x0:{N * H}")
    ws = sp.symbols(f"w0:{V * H}")
    Xs = [[xs[n * H + h] for h in range(H)] for n in range(N)]
    Ws = [[ws[v * H + h] for h in range(H)] for v in range(V)]
    valid = [n for n in range(N) if t[n] != -100]
    terms = []
    for n in valid:
        z = [sum(Xs[n][h] * Ws[v][h] for h in range(H)) for v in range(V)]
        terms.append(sp.log(sum(sp.exp(zz) for zz in z)) - z[t[n]])
    L = sum(terms) / len(valid)
    subs = {xs[n * H + h]: Xq[n][h] for n in range(N) for h in range(H)}
    subs.update({ws[v * H + h]: Wq[v][h] for v in range(V) for h in range(H)})
    X = np.array([[float(v) for v in r] for r in Xq])
    W = np.array([[float(v) for v in r] for r in Wq])
    o = orc(X, W, np.array(t, dtype=np.int32), -100, "mean")
    if abs(float(L.subs(subs).evalf(30)) - o["loss"]) > 1e-13:
        return False, "sympy loss"
    for n in range(N):
        for h in range(H):
            g = float(sp.diff(L, xs[n * H + h]).subs(subs).evalf(30))
            if abs(g - o["grad_hidden"][n, h]) > 1e-13:
                return False, f"sympy dX[{n},{h}]"
    for v in range(V):
        for h in range(H):
            g = float(sp.diff(L, ws[v * H + h]).subs(subs).evalf(30))
            if abs(g - o["grad_weight"][v, h]) > 1e-13:
                return False, f"sympy dW[{v},{h}]"
    return True, ""


def pin_finite_differences(orc):
    N, H, V = 4, 3, 5
    X, W, t = _rand_f64(N, H, V, 5)
    t[2] = -100
    o = orc(X, W, t, -100, "mean")
    eps = 1e-6
    for which, A, G in (("X", X, o["grad_hidden"]), ("W", W, o["grad_weight"])):
        for idx in np.ndindex(A.shape):
            Ap, Am = A.copy(), A.copy()
            Ap[idx] += eps
            Am[idx] -= eps
            args_p = (Ap, W) if which == "X" else (X, Ap)
            args_m = (Am, W) if which == "X" else (X, Am)
            fd = (orc(*args_p, t, -100, "mean", False)["loss"]
                  - orc(*args_m, t, -100, "mean", False)["loss"]) / (2 * eps)
            if abs(fd - G[idx]) > 1e-7 * max(1.0, abs(G[idx])):
                return False, f"finite difference d{which}{idx}: {fd} vs {G[idx]}"
    return True, ""


def pin_zero_weight(orc):
    for (N, H, V, ign) in ((6, 3, 7, 2), (5, 4, 1000, 0), (3, 2, 1, 1)):
        X, _, t = _rand_f64(N, H, V, N + V, ign)
        W = np.zeros((V, H))
        o = orc(X, W, t, -100, "mean")
        if abs(o["loss"] - math.log(V)) > 1e-14 * max(1, math.log(V)):
            return False, "zero weight loss != ln V"
        if np.abs(o["grad_hidden"]).max() != 0.0:
            return False, "zero weight grad_hidden != 0"
        nv = int((t != -100).sum())
        expect = np.zeros((V, H))
        for v in range(V):
            for n in range(N):
                if t[n] == -100:
                    continue
                coef = 1.0 / V - (1.0 if t[n] == v else 0.0)
                for h in range(H):
                    expect[v, h] += coef * X[n, h] / nv
        if np.abs(o["grad_weight"] - expect).max() > 1e-14:
            return False, "zero weight grad_weight"
    # equal rows: softmax still uniform, grad_hidden = sum_v dz_v w = 0
    X, W, t = _rand_f64(5, 3, 6, 9)
    W[:] = W[0]
    o = orc(X, W, t, -100, "mean")
    if abs(o["loss"] - math.log(6)) > 1e-13 or np.abs(o["grad_hidden"]).max() > 1e-14:
        return False, "equal-rows weight"
    return True, ""


def pin_golden(orc):
    ex = json.load(open(GOLDEN))["examples"]
    ev = lambda s: eval(s, {"__builtins__": {}}, {"math": math})  # noqa: E731
    for e in ex:
        X = np.array(e["hidden"], dtype=np.float64)
        W = np.array(e["weight"], dtype=np.float64)
        t = np.array(e["targets"], dtype=np.int32)
        o = orc(X, W, t, -100, "mean")
        if o["n_valid"] != e["n_valid"]:
            return False, f"golden {e['name']} n_valid"
        if abs(o["loss"] - ev(e["loss"])) > 1e-14:
            return False, f"golden {e['name']} loss"
        gh = np.array([[ev(s) for s in r] for r in e["grad_hidden"]])
        gw = np.array([[ev(s) for s in r] for r in e["grad_weight"]])
        if np.abs(o["grad_hidden"] - gh).max() > 1e-14:
            return False, f"golden {e['name']} grad_hidden"
        if np.abs(o["grad_weight"] - gw).max() > 1e-14:
            return False, f"golden {e['name']} grad_weight"
    return True, ""


def pin_column_sums(orc):
    for seed in range(3):
        X, W, t = _rand_f64(20, 6, 13, seed, 4)
        gw = orc(X, W, t, -100, "mean")["grad_weight"]
        if np.abs(gw.sum(axis=0)).max() > 1e-14 * max(1.0, np.abs(gw).max()):
            return False, "grad_weight column sums do not vanish"
        if np.abs(gw).max() == 0:
            return False, "grad_weight identically zero"
    return True, ""


def pin_shift_and_scale(orc):
    X, W, t = _rand_f64(8, 4, 9, 21, 2)
    base = orc(X, W, t, -100, "mean")
    for c in (1e3, -1e4):
        Xa = np.concatenate([X, np.ones((8, 1))], axis=1)
        Wa = np.concatenate([W, np.full((9, 1), c)], axis=1)
        o = orc(Xa, Wa, t, -100, "mean")
        if not np.isfinite(o["loss"]) or abs(o["loss"] - base["loss"]) > 1e-9:
            return False, f"shift by {c} changed the loss"
        if _rel(o["grad_hidden"][:, :4], base["grad_hidden"]) > 1e-9:
            return False, f"shift by {c} changed grad_hidden"
        if _rel(o["grad_weight"][:, :4], base["grad_weight"]) > 1e-9:
            return False, f"shift by {c} changed grad_weight"
    o = orc(X, W * 3000.0, t, -100, "mean")
    for k in ("loss", "grad_hidden", "grad_weight"):
        if not np.all(np.isfinite(o[k])):
            return False, f"non-finite {k} at large logits"
    return True, ""


def pin_ignored_rows(orc):
    X, W, t = _rand_f64(12, 5, 7, 31, 4)
    o = orc(X, W, t, -100, "mean")
    ign = t == -100
    X2 = X.copy()
    X2[ign] = 1e6
    o2 = orc(X2, W, t, -100, "mean")
    if abs(o["loss"] - o2["loss"]) != 0.0 or not np.array_equal(o["grad_weight"], o2["grad_weight"]):
        return False, "ignored rows changed the result"
    if np.abs(o2["grad_hidden"][ign]).max() != 0.0 or not np.array_equal(
            o["grad_hidden"][~ign], o2["grad_hidden"][~ign]):
        return False, "ignored rows of grad_hidden"
    # dropping ignored rows altogether gives the same answer
    o3 = orc(X[~ign], W, t[~ign], -100, "mean")
    if abs(o3["loss"] - o["loss"]) > 1e-15 or _rel(o3["grad_weight"], o["grad_weight"]) > 1e-15:
        return False, "dropping ignored rows changed the result"
    if o["n_valid"] != int((~ign).sum()):
        return False, "n_valid"
    return True, ""


def pin_mean_linearity(orc):
    X, W, t = _rand_f64(30, 4, 6, 41, 7)
    full = orc(X, W, t, -100, "mean")
    parts = [slice(0, 9), slice(9, 10), slice(10, 30)]
    S = 0.0
    n = 0
    gw = np.zeros_like(W)
    gh = []
    for p in parts:
        o = orc(X[p], W, t[p], -100, "sum")
        S += o["loss"]
        n += o["n_valid"]
        gw += o["grad_weight"]
        gh.append(o["grad_hidden"])
    if abs(S / n - full["loss"]) > 1e-14:
        return False, "mean != sum of part sums / sum of counts"
    if _rel(gw / n, full["grad_weight"]) > 1e-14:
        return False, "grad_weight not linear over splits"
    if _rel(np.concatenate(gh) / n, full["grad_hidden"]) > 1e-14:
        return False, "grad_hidden not linear over splits"
    return True, ""


def pin_special_cases(orc):
    X, W, t = _rand_f64(4, 3, 1, 51)
    o = orc(X, W, t, -100, "mean")
    if o["loss"] != 0.0 or np.abs(o["grad_hidden"]).max() != 0 or np.abs(o["grad_weight"]).max() != 0:
        return False, "V = 1 must give zero loss and grads"
    # one dominant target logit: loss = log(1 + (V-1) e^-50)
    X = np.array([[1.0, 0.0]])
    W = np.zeros((5, 2))
    W[3, 0] = 50.0
    o = orc(X, W, np.array([3], dtype=np.int32), -100, "mean")
    if abs(o["loss"] - math.log1p(4 * math.exp(-50))) > 1e-13:
        return False, "dominant target"
    if np.abs(o["grad_hidden"]).max() > 1e-20 or np.abs(o["grad_weight"]).max() > 1e-20:
        return False, "dominant target: gradients must vanish"
    # all tokens ignored: the reading is loss 0 and zero grads
    X, W, t = _rand_f64(3, 2, 4, 52)
    t[:] = -100
    o = orc(X, W, t, -100, "mean")
    if o["n_valid"] != 0 or o["loss"] != 0.0 or np.abs(o["grad_weight"]).max() != 0:
        return False, "n_valid = 0"
    return True, ""


PINS = [pin_torch, pin_sympy, pin_finite_differences, pin_zero_weight, pin_golden,
        pin_column_sums, pin_shift_and_scale, pin_ignored_rows, pin_mean_linearity,
        pin_special_cases]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    ok, msg = pin(flce_oracle_f64)
    assert ok, msg


# --------------------------------------------------------------------------
# the bf16 entry point, the row-restricted forms, errors
# --------------------------------------------------------------------------

def test_bf16_decode_exact():
    vals = np.array([0.0, -0.0, 1.0, -2.5, 3.140625, 1e-30, 65280.0, 2.0 ** -133],
                    dtype=np.float32)
    bits = wl.f32_to_bf16_bits(vals)
    dec = ofl.decode_bf16(bits)
    for v, d in zip(vals, dec):
        # every value above is exactly representable in bf16 except 1e-30
        if v != np.float32(1e-30):
            assert d == float(v)
    # rounding is to nearest even: 1 + 2^-8 is a tie between 1 and 1 + 2^-7
    assert ofl.decode_bf16(wl.f32_to_bf16_bits(np.array([1 + 2 ** -8], np.float32)))[0] == 1.0
    assert ofl.decode_bf16(wl.f32_to_bf16_bits(np.array([1 + 3 * 2 ** -8], np.float32)))[0] == 1 + 2 ** -6


def test_bf16_entry_matches_f64_core():
    p = wl.make_inputs(wl.WORKLOADS["tiny"])
    a = flce_oracle(p["hidden"], p["weight"], p["targets"])
    b = flce_oracle_f64(ofl.decode_bf16(p["hidden"]), ofl.decode_bf16(p["weight"]), p["targets"])
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["grad_weight"], b["grad_weight"])
    assert abs(a["loss"] - math.log(512)) < 0.5      # near-uniform softmax at std 0.02


def test_row_forms_match_full():
    p = wl.random_problem(50, 16, 37, seed=3, ignore_frac=0.2)
    full = flce_oracle(p["hidden"], p["weight"], p["targets"])
    rows = np.array([0, 3, 7, 8, 49])
    r = oracle_rows(p["hidden"][rows], p["weight"], p["targets"][rows], full["n_valid"])
    np.testing.assert_allclose(r["row_loss"], full["row_loss"][rows], rtol=1e-13, atol=0)
    np.testing.assert_allclose(r["grad_hidden"], full["grad_hidden"][rows], rtol=1e-12, atol=1e-18)
    lse = lse_all_rows(p["hidden"], p["weight"], p["targets"], rows_per_block=7)
    np.testing.assert_array_equal(np.isnan(lse), np.isnan(full["lse"]))
    ok = ~np.isnan(lse)
    np.testing.assert_allclose(lse[ok], full["lse"][ok], rtol=1e-13)
    vr = np.array([0, 5, 36])
    gw = grad_weight_rows(p["hidden"], p["weight"], p["targets"], lse, vr)
    np.testing.assert_allclose(gw, full["grad_weight"][vr], rtol=1e-11, atol=1e-17)


def test_bad_target_raises():
    X, W, t = _rand_f64(4, 2, 5, 1)
    t[1] = 5
    with pytest.raises(ofl.BadTarget):
        flce_oracle_f64(X, W, t)
    t[1] = -1
    with pytest.raises(ofl.BadTarget):
        flce_oracle_f64(X, W, t)
    t[1] = -100
    flce_oracle_f64(X, W, t)


def test_workload_recipes():
    w = wl.WORKLOADS
    assert (w["llama3_8b_head"].n_ignored, w["llama3_8b_head"].n_valid) == (327, 16057)
    assert (w["large_vocab"].n_ignored, w["component"].n_ignored, w["full_model"].n_ignored) == (4096, 204, 3276)
    p = wl.make_inputs(w["component"])
    assert int((p["targets"] == -100).sum()) == 204
    v = p["targets"][p["targets"] != -100]
    assert v.min() >= 0 and v.max() < 16000
    q = wl.make_inputs(w["component"])
    assert np.array_equal(p["hidden"], q["hidden"]) and np.array_equal(p["targets"], q["targets"])
    # Zipf targets: the most frequent token takes about 1/H_{V,1.1} of the mass
    z = wl.zipf_ranks(np.random.default_rng(0), 200000, 16000, 1.1)
    Hs = np.sum(np.arange(1, 16001, dtype=np.float64) ** -1.1)
    assert abs(np.mean(z == 0) - 1 / Hs) < 0.01


def test_rms_rows_recipe():
    w = wl.WORKLOADS["llama3_8b_head"].with_shape(N=64, H=256, V=300)
    p = wl.make_inputs(w)
    x = wl.bf16_bits_to_f32(p["hidden"]).astype(np.float64)
    rms = np.sqrt(np.mean(x * x, axis=1))
    assert np.all(np.abs(rms - 1) < 0.01)


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# --------------------------------------------------------------------------

def _mut_no_onehot(Z, lse, tv, scale):
    return np.exp(Z - lse[:, None]) * scale


def _mut_sign(Z, lse, tv, scale):
    P = np.exp(Z - lse[:, None])
    P[np.arange(Z.shape[0]), tv] -= 1.0
    return -P * scale


def _mut_lse_no_shift(Z):
    return np.log(np.exp(Z).sum(axis=1))


def _mut_lse_drop_max(Z):
    m = Z.max(axis=1)
    return np.log(np.exp(Z - m[:, None]).sum(axis=1))


def _mut_loss_sign(Z, lse, tv):
    return lse + Z[np.arange(Z.shape[0]), tv]


def _mut_target_offbyone(Z, lse, tv):
    return lse - Z[np.arange(Z.shape[0]), (tv + 1) % Z.shape[1]]


def _mut_scale_count_all(n_valid, reduction):
    return 1.0 / (n_valid + 1) if reduction == "mean" else 1.0


def _mut_gw_wrong_rows(dZ, Xv):
    return dZ.T @ Xv[::-1]


def _mut_gh_transposed_w(dZ, W):
    return dZ[:, ::-1] @ W


MUTATIONS = [
    ("dlogits", _mut_no_onehot), ("dlogits", _mut_sign),
    ("logsumexp_rows", _mut_lse_no_shift), ("logsumexp_rows", _mut_lse_drop_max),
    ("row_losses", _mut_loss_sign), ("row_losses", _mut_target_offbyone),
    ("grad_scale", _mut_scale_count_all), ("grad_weight_full", _mut_gw_wrong_rows),
    ("grad_hidden_rows", _mut_gh_transposed_w),
]


@pytest.mark.parametrize("name,fn", MUTATIONS, ids=[f.__name__ for _, f in MUTATIONS])
def test_pins_catch_planted_mistake(monkeypatch, name, fn):
    monkeypatch.setattr(ofl, name, fn)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                ok, msg = pin(ofl.flce_oracle_f64)
        except (FloatingPointError, ValueError, IndexError, AssertionError) as e:
            ok, msg = False, repr(e)
        if not ok:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake in {name}"
