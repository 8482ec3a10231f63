"""Seeded synthetic inputs for the fused linear cross-entropy (LM head).

This module only draws inputs. It holds none of the loss arithmetic, so both
the fp64 oracle (``oracle/``) and the CUDA path can be fed from it without
sharing any computation.

Every array is produced from ``numpy.random.default_rng(PCG64(seed))`` in a
fixed draw order: hidden, weight, vocabulary permutation (Zipf targets only),
targets, ignored positions.  Values are drawn in fp32 and rounded to bf16
with round-to-nearest-even; bf16 tensors are returned as their raw ``uint16``
bit patterns so that both sides decode exactly the same numbers.

Workload shapes follow the pages on the fused linear cross-entropy:

* "efficient-llm-anatomy" README, "Results" section: model config H=512,
  V=16000, per-component table measured at B=4, S=1024, full-model table at
  B=16, S=4096 (bf16).
* A Llama-3-8B-shaped LM head (H=4096, V=128256) and a large-vocabulary
  stress case, the two shapes used for throughput.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    """One seeded synthetic problem: N tokens, hidden size H, vocabulary V."""

    name: str
    N: int
    H: int
    V: int
    seed: int
    weight_std: float = 0.02
    targets: str = "uniform"          # "uniform" | "zipf"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0          # exactly floor(ignore_frac * N) ignored
    rms_norm_rows: bool = False       # hidden rows scaled to unit RMS (fp32)
    ignore_index: int = IGNORE_INDEX

    @property
    def n_ignored(self) -> int:
        return int(np.floor(self.ignore_frac * self.N))

    @property
    def n_valid(self) -> int:
        return self.N - self.n_ignored

    def with_shape(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    # tiny case the oracle finishes instantly
    "tiny": Workload("tiny", N=128, H=64, V=512, seed=0),
    # per-component shape of the pages (B=4, S=1024, H=512, V=16000)
    "component": Workload("component", N=4096, H=512, V=16000, seed=1,
                          ignore_frac=0.05),
    # full-model shape of the pages (B=16, S=4096)
    "full_model": Workload("full_model", N=65536, H=512, V=16000, seed=2,
                           targets="zipf", ignore_frac=0.05),
    # Llama-3-8B-shaped LM head
    "llama3_8b_head": Workload("llama3_8b_head", N=16384, H=4096, V=128256,
                               seed=3, targets="zipf", ignore_frac=0.02,
                               rms_norm_rows=True),
    # large-vocabulary stress, peaky softmax, half the tokens ignored
    "large_vocab": Workload("large_vocab", N=8192, H=2048, V=256000, seed=4,
                            weight_std=0.05, ignore_frac=0.5),
    # same recipe with a vocabulary that is not a multiple of any tile
    "large_vocab_tail": Workload("large_vocab_tail", N=8192, H=2048, V=256007,
                                 seed=4, weight_std=0.05, ignore_frac=0.5),
}

ORDER = ["tiny", "component", "full_model", "llama3_8b_head", "large_vocab"]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (used by generators/tests)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float,
                 rms_rows: bool = False, block_rows: int = 8192) -> np.ndarray:
    """N(0, std^2) in fp32, optionally unit-RMS rows, rounded to bf16 bits.

    Drawn in row blocks to bound host memory; the stream of random numbers is
    the same as one big draw because standard_normal consumes it in order.
    """
    rows, cols = shape
    out = np.empty(shape, dtype=np.uint16)
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        x = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if rms_rows:
            ms = np.mean(x * x, axis=1, dtype=np.float32, keepdims=True)
            x /= np.sqrt(ms + np.float32(1e-6))
        out[r0:r1] = f32_to_bf16_bits(x)
    return out


def zipf_ranks(rng: np.random.Generator, n: int, V: int, s: float) -> np.ndarray:
    """Truncated Zipf over ranks 1..V, P(r) proportional to r^-s (inverse CDF)."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    r = np.searchsorted(cdf, u, side="right")
    return np.minimum(r, V - 1).astype(np.int64)      # 0-based rank


def make_inputs(w: Workload, hidden: bool = True, weight: bool = True) -> dict:
    """Draw (hidden, weight, targets) for workload ``w``.

    Returns a dict with ``hidden`` (uint16 [N,H] bf16 bits), ``weight``
    (uint16 [V,H] bf16 bits), ``targets`` (int32 [N]) and the workload.
    ``hidden=False``/``weight=False`` still consume the same random stream
    (so targets are identical) but skip keeping the array.
    """
    rng = np.random.default_rng(np.random.PCG64(w.seed))
    X = _normal_bf16(rng, (w.N, w.H), 1.0, rms_rows=w.rms_norm_rows)
    W = _normal_bf16(rng, (w.V, w.H), w.weight_std)
    if w.targets == "zipf":
        perm = rng.permutation(w.V)
        t = perm[zipf_ranks(rng, w.N, w.V, w.zipf_s)]
    elif w.targets == "uniform":
        t = rng.integers(0, w.V, size=w.N)
    else:
        raise ValueError(w.targets)
    t = t.astype(np.int32)
    k = w.n_ignored
    if k:
        pos = rng.choice(w.N, size=k, replace=False)
        t[pos] = np.int32(w.ignore_index)
    return {"hidden": X if hidden else None, "weight": W if weight else None,
            "targets": t, "workload": w}


def random_problem(N: int, H: int, V: int, seed: int, weight_std: float = 0.05,
                   ignore_frac: float = 0.0, ignore_index: int = IGNORE_INDEX,
                   hidden_std: float = 1.0) -> dict:
    """Small seeded problem of any shape (edge-case and parity tests)."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    X = _normal_bf16(rng, (N, H), hidden_std)
    W = _normal_bf16(rng, (V, H), weight_std)
    t = rng.integers(0, V, size=N).astype(np.int32)
    k = int(np.floor(ignore_frac * N))
    if k:
        t[rng.choice(N, size=k, replace=False)] = np.int32(ignore_index)
    return {"hidden": X, "weight": W, "targets": t,
            "workload": Workload("random", N=N, H=H, V=V, seed=seed,
                                 weight_std=weight_std, ignore_frac=ignore_frac,
                                 ignore_index=ignore_index)}


def describe(w: Workload) -> str:
    return (f"{w.name}: N={w.N} H={w.H} V={w.V} weight~N(0,{w.weight_std}) "
            f"targets={w.targets} ignore={w.n_ignored} seed={w.seed}"
            + (" rms-rows" if w.rms_norm_rows else ""))
