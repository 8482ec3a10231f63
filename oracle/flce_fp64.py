"""fp64 CPU oracle for the fused linear cross-entropy (LM head).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code with
the CUDA path (the two meet only through the seeded input generator, which
holds no loss arithmetic).

What it computes is the plain definition, step by step, in fp64 with numpy
(a matmul is the only library primitive used as a step):

  inputs   X [N,H] bf16, W [V,H] bf16 (PyTorch ``Linear`` layout, forward is
           X @ W.T), targets t [N] int32, ignore_index ii.
  1. decode bf16 exactly to fp64 (bf16 is a subset of fp64).
  2. valid rows: t_n != ii; every other target must lie in [0, V);
     n_valid = number of valid rows.
  3. logits z_nv = sum_h X_nh W_vh for valid rows.
  4. lse_n = m_n + log(sum_v exp(z_nv - m_n)), m_n = max_v z_nv
     (max-shifted log-sum-exp; "Alisa's book of LLMs", section "Numerical
     stability and other tricks", logsumexp paragraph).
  5. per-row loss l_n = lse_n - z_{n,t_n} (cross-entropy with a one-hot
     target is the negative log-likelihood of the target; same page,
     "cross-entropy loss" paragraph), loss = sum_n l_n / n_valid over valid
     rows (masked mean, same page, "implementing the loss" code:
     masked sum divided by the mask count).
  6. dz_nv = (softmax(z_n)_v - [v == t_n]) / n_valid for valid rows, zero
     for ignored rows ("gradient of softmax + CE loss" section: p minus the
     one-hot target; the 1/n factor from the linearity of the mean,
     "Backpropagation" section, mean-reduction paragraph).
  7. grad_hidden = dz @ W   (per-sample activation: rows stack; "Neural net
     basics", linear-layer backprop in PyTorch layout).
  8. grad_weight = dz.T @ X (shared parameter: the batch dimension is
     contracted; same paragraph).

Readings where the pages are silent (kept identical on the GPU side):
  * n_valid == 0: loss 0, grads 0 (the masked mean would be 0/0).
  * reduction "sum": loss = sum_n l_n and grads without the 1/n_valid factor.
  * a target outside [0, V) that is not ii raises ``BadTarget``.

Pins (tests/test_oracle_pins.py) tie this code to things other than itself:
PyTorch's own CPU cross_entropy + autograd in fp64, exact symbolic
differentiation with sympy, central finite differences, the zero-weight
closed form loss = ln V, hand-derived tiny examples (tests/golden), the
vanishing column sums of grad_weight, shift invariance of log-sum-exp, the
invariance under ignored rows, and mean linearity over token splits.
"""
from __future__ import annotations

import numpy as np


class BadTarget(ValueError):
    """A target outside [0, V) that is not the ignore index."""


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """Step 1: exact bf16 -> fp64 (a bf16 is the top half of an fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def valid_rows(targets: np.ndarray, V: int, ignore_index: int) -> np.ndarray:
    """Step 2: boolean mask of rows that take part in the loss."""
    t = np.asarray(targets, dtype=np.int64)
    valid = t != ignore_index
    bad = valid & ((t < 0) | (t >= V))
    if bad.any():
        raise BadTarget(f"{int(bad.sum())} target(s) outside [0, {V})")
    return valid


def logits(Xv: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Step 3: z = X @ W.T (fp64)."""
    return Xv @ W.T


def logsumexp_rows(Z: np.ndarray) -> np.ndarray:
    """Step 4: max-shifted log-sum-exp of each row."""
    m = Z.max(axis=1)
    return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))


def row_losses(Z: np.ndarray, lse: np.ndarray, tv: np.ndarray) -> np.ndarray:
    """Step 5: l_n = lse_n - z_{n, t_n}."""
    return lse - Z[np.arange(Z.shape[0]), tv]


def dlogits(Z: np.ndarray, lse: np.ndarray, tv: np.ndarray, scale: float) -> np.ndarray:
    """Step 6: (softmax - onehot) * scale, scale = 1/n_valid for the mean."""
    P = np.exp(Z - lse[:, None])
    P[np.arange(Z.shape[0]), tv] -= 1.0
    return P * scale


def grad_hidden_rows(dZ: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Step 7: grad_hidden = dz @ W (rows of a per-sample activation stack)."""
    return dZ @ W


def grad_weight_full(dZ: np.ndarray, Xv: np.ndarray) -> np.ndarray:
    """Step 8: grad_weight = dz.T @ X (the batch dimension is contracted)."""
    return dZ.T @ Xv


def grad_scale(n_valid: int, reduction: str) -> float:
    if reduction == "sum":
        return 1.0
    if reduction != "mean":
        raise ValueError(reduction)
    return 0.0 if n_valid == 0 else 1.0 / n_valid


def flce_oracle(hidden_bits, weight_bits, targets, ignore_index: int = -100,
                reduction: str = "mean", want_grads: bool = True) -> dict:
    """Full forward+backward of the fused linear cross-entropy, in fp64.

    Returns ``loss`` (float), ``n_valid`` (int), ``row_loss`` [N] (0 on
    ignored rows), ``lse`` [N] (nan on ignored rows) and, if ``want_grads``,
    ``grad_hidden`` [N,H] and ``grad_weight`` [V,H] (fp64).
    """
    return flce_oracle_f64(decode_bf16(hidden_bits), decode_bf16(weight_bits),
                           targets, ignore_index, reduction, want_grads)


def flce_oracle_f64(X: np.ndarray, W: np.ndarray, targets, ignore_index: int = -100,
                    reduction: str = "mean", want_grads: bool = True) -> dict:
    """Steps 2-8 on fp64 inputs (used directly by the finite-difference and
    symbolic pins, which perturb X and W continuously)."""
    N, H = X.shape
    V = W.shape[0]
    valid = valid_rows(targets, V, ignore_index)
    n_valid = int(valid.sum())
    tv = np.asarray(targets, dtype=np.int64)[valid]
    Xv = X[valid]

    Z = logits(Xv, W)
    lse = logsumexp_rows(Z)
    rl = row_losses(Z, lse, tv)
    total = float(rl.sum())
    if reduction == "mean":
        loss = 0.0 if n_valid == 0 else total / n_valid
    elif reduction == "sum":
        loss = total
    else:
        raise ValueError(reduction)

    out = {"loss": loss, "n_valid": n_valid,
           "row_loss": np.zeros(N), "lse": np.full(N, np.nan)}
    out["row_loss"][valid] = rl
    out["lse"][valid] = lse
    if want_grads:
        dZ = dlogits(Z, lse, tv, grad_scale(n_valid, reduction))
        gX = np.zeros((N, H))
        gX[valid] = grad_hidden_rows(dZ, W)
        out["grad_hidden"] = gX
        out["grad_weight"] = grad_weight_full(dZ, Xv)
    return out


# ---------------------------------------------------------------------------
# Row-restricted forms for problems too large to evaluate whole.  Rows are
# independent given W, so each function below is the definition above applied
# to a subset of rows; only grad_weight needs every row's log-sum-exp.
# ---------------------------------------------------------------------------

def oracle_rows(hidden_rows_bits, weight_bits, target_rows, n_valid: int,
                ignore_index: int = -100, reduction: str = "mean",
                weight_f64: np.ndarray | None = None) -> dict:
    """lse, per-row loss and grad_hidden rows for the given rows.

    ``n_valid`` is the count over the whole problem (it sets the 1/n scale).
    Ignored rows get loss 0, lse nan and a zero grad_hidden row.
    """
    X = decode_bf16(hidden_rows_bits)
    W = decode_bf16(weight_bits) if weight_f64 is None else weight_f64
    V = W.shape[0]
    valid = valid_rows(target_rows, V, ignore_index)
    tv = np.asarray(target_rows, dtype=np.int64)[valid]
    Z = logits(X[valid], W)
    lse = logsumexp_rows(Z)
    rl = row_losses(Z, lse, tv)
    dZ = dlogits(Z, lse, tv, grad_scale(n_valid, reduction))
    gX = np.zeros(X.shape)
    gX[valid] = grad_hidden_rows(dZ, W)
    R = X.shape[0]
    out_lse = np.full(R, np.nan)
    out_lse[valid] = lse
    out_rl = np.zeros(R)
    out_rl[valid] = rl
    return {"lse": out_lse, "row_loss": out_rl, "grad_hidden": gX}


def lse_all_rows(hidden_bits, weight_bits, targets, ignore_index: int = -100,
                 rows_per_block: int = 512, weight_f64: np.ndarray | None = None):
    """Step 4 for every row (nan on ignored rows), evaluated a block of rows
    at a time so that no N x V array is held."""
    W = decode_bf16(weight_bits) if weight_f64 is None else weight_f64
    t = np.asarray(targets, dtype=np.int64)
    valid = valid_rows(t, W.shape[0], ignore_index)
    N = t.shape[0]
    lse = np.full(N, np.nan)
    idx = np.nonzero(valid)[0]
    for i0 in range(0, idx.size, rows_per_block):
        rows = idx[i0:i0 + rows_per_block]
        Z = logits(decode_bf16(hidden_bits[rows]), W)
        lse[rows] = logsumexp_rows(Z)
    return lse


def grad_weight_rows(hidden_bits, weight_bits, targets, lse, vocab_rows,
                     ignore_index: int = -100, reduction: str = "mean",
                     weight_f64: np.ndarray | None = None) -> np.ndarray:
    """Rows ``vocab_rows`` of grad_weight = dz.T @ X, given every row's lse."""
    X = decode_bf16(hidden_bits)
    W = decode_bf16(weight_bits) if weight_f64 is None else weight_f64
    t = np.asarray(targets, dtype=np.int64)
    valid = valid_rows(t, W.shape[0], ignore_index)
    n_valid = int(valid.sum())
    vr = np.asarray(vocab_rows, dtype=np.int64)
    Xv = X[valid]
    Zs = Xv @ W[vr].T                               # z_nv for the chosen v
    P = np.exp(Zs - lse[valid][:, None])
    P -= (t[valid][:, None] == vr[None, :])
    dZs = P * grad_scale(n_valid, reduction)
    return dZs.T @ Xv


# ---------------------------------------------------------------------------
# Final RMSNorm fused in front of the LM head ("Alisa's book of LLMs",
# transformer section: final norm, then the unembedding; RMSNorm divides every
# element of the hidden state by its RMS, then multiplies by a learned
# per-dimension gain).  Reading taken: eps inside the square root,
# rms_n = sqrt(mean_h(h_nh^2) + eps).
# ---------------------------------------------------------------------------

def rmsnorm_rows(Hs: np.ndarray, gain: np.ndarray, eps: float):
    """x = (h / rms(h)) * gain, with xhat = h / rms(h) and r = 1 / rms(h)."""
    r = 1.0 / np.sqrt(np.mean(Hs * Hs, axis=1) + eps)
    xhat = Hs * r[:, None]
    return xhat * gain[None, :], xhat, r


def rmsnorm_backward(dX: np.ndarray, xhat: np.ndarray, r: np.ndarray, gain: np.ndarray):
    """Chain rule through x = xhat * gain, xhat = h * r, r = (mean(h^2)+eps)^-1/2:
    dgain = sum_n dX_n * xhat_n;  dh_n = r_n (gain * dX_n - xhat_n * mean(gain * dX_n * xhat_n))."""
    dgain = (dX * xhat).sum(axis=0)
    gdx = dX * gain[None, :]
    dh = r[:, None] * (gdx - xhat * np.mean(gdx * xhat, axis=1, keepdims=True))
    return dh, dgain


def rmsnorm_flce_oracle_f64(Hs: np.ndarray, gain: np.ndarray, W: np.ndarray, targets, eps: float = 1e-6,
                            ignore_index: int = -100, reduction: str = "mean") -> dict:
    """loss of the LM head on the normalised hidden states, and the gradients
    with respect to the un-normalised hidden states, the gain and the weight."""
    X, xhat, r = rmsnorm_rows(Hs, gain, eps)
    o = flce_oracle_f64(X, W, targets, ignore_index, reduction)
    dh, dgain = rmsnorm_backward(o["grad_hidden"], xhat, r, gain)
    return {"loss": o["loss"], "n_valid": o["n_valid"], "row_loss": o["row_loss"], "normed": X,
            "grad_hidden": dh, "grad_gain": dgain, "grad_weight": o["grad_weight"]}


def rmsnorm_flce_oracle(hidden_bits, gain_bits, weight_bits, targets, eps: float = 1e-6,
                        ignore_index: int = -100, reduction: str = "mean") -> dict:
    return rmsnorm_flce_oracle_f64(decode_bf16(hidden_bits), decode_bf16(gain_bits), decode_bf16(weight_bits),
                                   targets, eps, ignore_index, reduction)
