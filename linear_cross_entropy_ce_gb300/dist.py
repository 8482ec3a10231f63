"""Host-side helpers for running the fused linear cross-entropy on several
ranks (one process per GPU, torch.distributed).

The path itself has no exchange: rows are independent given W, so each rank
processes its own tokens.  Two uses:

* replicas (what ``bench.py --gpus N`` runs): every rank an independent batch,
  timed with a barrier on both sides and the max over ranks;
* a data-parallel step over one global batch split by tokens: each rank calls
  ``flce_fwd_bwd`` with ``FLCE_REDUCE_SUM`` on its shard, then one exchange
  (sum of the loss sums, the valid counts and grad_weight) and a 1/n_valid
  rescale give the global mean -- the linearity of the mean ("Alisa's book of
  LLMs", Backpropagation section) applied across ranks, as data parallelism
  all-reduces gradients.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_rows(n_rows: int, rank: int, world: int) -> slice:
    """Contiguous block of token rows owned by `rank` (sizes differ by <= 1)."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    return slice(n_rows * rank // world, n_rows * (rank + 1) // world)


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of the synthetic batch of a benchmark replica."""
    return base_seed + 1000 * rank


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank scalar (step time); identity without a process group."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def exchange_sums(loss_sum: float, n_valid: int, grad_weight: torch.Tensor):
    """All-reduce the unscaled outputs of a token shard and rescale in place.

    Returns (mean loss, global n_valid, scale); grad_weight becomes the global
    mean gradient.  grad_hidden rows stay local: scale them by the returned
    factor.
    """
    t = torch.tensor([float(loss_sum), float(n_valid)], dtype=torch.float64, device=grad_weight.device)
    dist.all_reduce(t)
    dist.all_reduce(grad_weight)
    n = int(round(t[1].item()))
    scale = 1.0 / n if n else 0.0
    grad_weight.mul_(scale)
    return (t[0].item() * scale, n, scale)


def vocab_merge(row_max: torch.Tensor, row_sumexp: torch.Tensor, row_target_logit: torch.Tensor, rescale):
    """The exchange of the vocabulary-parallel LM head, in place.

    Each rank holds per-token (max, sum of exp(z - max), target logit) over
    its vocabulary shard.  After the call every rank holds the global max, the
    sum of exp(z - global max) over the whole vocabulary and the target logit
    (the online-softmax merge of "Alisa's book of LLMs" applied across ranks).
    ``rescale(local_max, global_max, sumexp)`` multiplies sumexp by
    exp(local_max - global_max) in place (``flce.vocab_rescale`` on the GPU).
    """
    local_max = row_max.clone()
    dist.all_reduce(row_max, op=dist.ReduceOp.MAX)
    rescale(local_max, row_max, row_sumexp)
    dist.all_reduce(row_sumexp)
    dist.all_reduce(row_target_logit)
