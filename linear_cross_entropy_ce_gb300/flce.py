"""ctypes binding of libflce (argument marshalling only).

Every step of the fused linear cross-entropy runs in the CUDA kernels of
``libflce.so``; this module only checks tensor types, allocates outputs and
the workspace through PyTorch's caching allocator, and passes raw device
pointers and the current CUDA stream to the C ABI declared in
``include/flce.h``.  There is no fallback: if the library is missing or the
call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libflce.so")

FLCE_OK, FLCE_EINVAL, FLCE_EUNSUPPORTED, FLCE_EWORKSPACE, FLCE_EBADTARGET, FLCE_ETIMEOUT, FLCE_ECUDA = range(7)
STATUS_NAMES = {0: "FLCE_OK", 1: "FLCE_EINVAL", 2: "FLCE_EUNSUPPORTED", 3: "FLCE_EWORKSPACE",
                4: "FLCE_EBADTARGET", 5: "FLCE_ETIMEOUT", 6: "FLCE_ECUDA"}
REDUCE = {"mean": 0, "sum": 1}
FLCE_GW_BF16 = 0x2

_lib = None


class FlceError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{what}: {name} ({_status_string(status)})" if what else name)


class PlanInfo(ctypes.Structure):
    _fields_ = [("chunk_rows", ctypes.c_int64), ("max_chunks", ctypes.c_int64),
                ("logits_row_stride", ctypes.c_int64), ("gemm_launches_per_chunk", ctypes.c_int32),
                ("dx_splits", ctypes.c_int32),
                ("vocab_tiles", ctypes.c_int32), ("workspace_bytes", ctypes.c_size_t)]


def library() -> ctypes.CDLL:
    """Load libflce.so (built in-tree by ``linear_cross_entropy_ce_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with linear_cross_entropy_ce_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    i64, u32, i32, sz, vp = ctypes.c_int64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
    lib.flce_workspace_bytes.argtypes = [i64, i64, i64, u32]
    lib.flce_workspace_bytes.restype = sz
    lib.flce_loss_workspace_bytes.argtypes = [i64, i64, i64, u32]
    lib.flce_loss_workspace_bytes.restype = sz
    lib.flce_workspace_bytes_for_chunk.argtypes = [i64, i64, i64, u32, i64]
    lib.flce_workspace_bytes_for_chunk.restype = sz
    lib.flce_plan.argtypes = [i64, i64, i64, u32, ctypes.c_int, sz, ctypes.POINTER(PlanInfo)]
    lib.flce_plan.restype = ctypes.c_int
    lib.flce_fwd_bwd.argtypes = [vp, vp, vp, i64, i64, i64, i32, u32, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_fwd_bwd.restype = ctypes.c_int
    lib.flce_loss.argtypes = [vp, vp, vp, i64, i64, i64, i32, u32, vp, vp, vp, vp, sz, vp]
    lib.flce_loss.restype = ctypes.c_int
    lib.flce_query_status.argtypes = [vp, vp]
    lib.flce_query_status.restype = ctypes.c_int
    lib.flce_selftest_timeout.argtypes = [vp, ctypes.c_uint64, vp]
    lib.flce_selftest_timeout.restype = ctypes.c_int
    lib.flce_query_stall.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
    lib.flce_query_stall.restype = ctypes.c_int
    lib.flce_debug_arm_stall.argtypes = [ctypes.c_uint64]
    lib.flce_debug_arm_stall.restype = ctypes.c_int
    lib.flce_status_string.argtypes = [ctypes.c_int]
    lib.flce_status_string.restype = ctypes.c_char_p
    lib.flce_rmsnorm_workspace_bytes.argtypes = [i64, i64, i64, u32]
    lib.flce_rmsnorm_workspace_bytes.restype = sz
    lib.flce_rmsnorm_fwd_bwd.argtypes = [vp, vp, ctypes.c_float, vp, vp, i64, i64, i64, i32, u32, vp, vp, vp, vp, vp,
                                         vp, vp, sz, vp]
    lib.flce_rmsnorm_fwd_bwd.restype = ctypes.c_int
    lib.flce_vocab_shard_workspace_bytes.argtypes = [i64, i64, i64, u32]
    lib.flce_vocab_shard_workspace_bytes.restype = sz
    lib.flce_vocab_shard_stats.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_vocab_shard_stats.restype = ctypes.c_int
    lib.flce_vocab_rescale.argtypes = [vp, vp, vp, i64, vp]
    lib.flce_vocab_rescale.restype = ctypes.c_int
    lib.flce_vocab_finish.argtypes = [vp, vp, vp, vp, i64, i32, u32, vp, vp, vp, vp, vp]
    lib.flce_vocab_finish.restype = ctypes.c_int
    lib.flce_vocab_shard_bwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, u32, vp, vp, vp, vp, sz, vp]
    lib.flce_vocab_shard_bwd.restype = ctypes.c_int
    lib.flce_scale_grads.argtypes = [vp, vp, i64, i64, i64, vp, vp]
    lib.flce_scale_grads.restype = ctypes.c_int
    lib.flce_profile_begin.argtypes = []
    lib.flce_profile_begin.restype = ctypes.c_int
    lib.flce_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_int64)]
    lib.flce_profile_end.restype = ctypes.c_int
    lib.flce_version.argtypes = []
    lib.flce_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _status_string(s: int) -> str:
    try:
        return library().flce_status_string(int(s)).decode()
    except Exception:  # pragma: no cover - library not loadable
        return "?"


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_inputs(hidden, weight, targets):
    if not (hidden.is_cuda and weight.is_cuda and targets.is_cuda):
        raise ValueError("hidden, weight and targets must be CUDA tensors")
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("hidden and weight must be bfloat16")
    if targets.dtype != torch.int32:
        raise TypeError("targets must be int32")
    if hidden.dim() != 2 or weight.dim() != 2 or targets.dim() != 1:
        raise ValueError("expected hidden [N,H], weight [V,H], targets [N]")
    N, H = hidden.shape
    V, H2 = weight.shape
    if H2 != H or targets.shape[0] != N:
        raise ValueError("shape mismatch")
    for t in (hidden, weight, targets):
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    return N, H, V


def _flags(reduction: str, grad_weight_dtype=torch.float32) -> int:
    if grad_weight_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("grad_weight_dtype must be torch.float32 or torch.bfloat16")
    return REDUCE[reduction] | (FLCE_GW_BF16 if grad_weight_dtype == torch.bfloat16 else 0)


def workspace_bytes(N: int, H: int, V: int, reduction: str = "mean", chunk_rows: Optional[int] = None,
                    forward_only: bool = False, grad_weight_dtype=torch.float32) -> int:
    """Workspace of the default plan (or of a given chunk size).  With a bf16
    grad_weight it includes the fp32 V x H accumulator of grad_weight."""
    lib = library()
    f = _flags(reduction, torch.float32 if forward_only else grad_weight_dtype)
    if forward_only:
        n = lib.flce_loss_workspace_bytes(N, H, V, f)
    elif chunk_rows is not None:
        n = lib.flce_workspace_bytes_for_chunk(N, H, V, f, chunk_rows)
    else:
        n = lib.flce_workspace_bytes(N, H, V, f)
    if n == 0:
        raise FlceError(FLCE_EINVAL, "workspace size")
    return int(n)


def plan(N: int, H: int, V: int, workspace_bytes: int, forward_only: bool = False,
         reduction: str = "mean", grad_weight_dtype=torch.float32) -> dict:
    info = PlanInfo()
    s = library().flce_plan(N, H, V, _flags(reduction, grad_weight_dtype), int(forward_only), workspace_bytes,
                            ctypes.byref(info))
    if s != FLCE_OK:
        raise FlceError(s, "flce_plan")
    return {k: getattr(info, k) for k, _ in PlanInfo._fields_}


def new_workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd_bwd(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
            reduction: str = "mean", *, workspace: Optional[torch.Tensor] = None,
            chunk_rows: Optional[int] = None, row_loss: bool = False, out: Optional[dict] = None,
            stream=None, grad_weight_dtype=torch.float32) -> dict:
    """Loss, n_valid, grad_hidden (bf16 [N,H]) and grad_weight ([V,H], fp32 by
    default, or bf16 rounded once from the fp32 accumulation) in one call."""
    N, H, V = _check_inputs(hidden, weight, targets)
    dev = hidden.device
    flags = _flags(reduction, grad_weight_dtype)
    if workspace is None:
        workspace = new_workspace(workspace_bytes(N, H, V, reduction, chunk_rows,
                                                  grad_weight_dtype=grad_weight_dtype), dev)
    o = out if out is not None else {}
    if "loss" not in o:
        o["loss"] = torch.empty(1, dtype=torch.float32, device=dev)
        o["n_valid"] = torch.empty(1, dtype=torch.int32, device=dev)
        o["grad_hidden"] = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        o["grad_weight"] = torch.empty((V, H), dtype=grad_weight_dtype, device=dev)
        o["row_loss"] = torch.empty(N, dtype=torch.float32, device=dev) if row_loss else None
    if o["grad_weight"].dtype != grad_weight_dtype:
        raise TypeError("out['grad_weight'] does not have grad_weight_dtype")
    s = library().flce_fwd_bwd(_ptr(hidden), _ptr(weight), _ptr(targets), N, H, V, int(ignore_index),
                               flags, _ptr(o["loss"]), _ptr(o["n_valid"]), _ptr(o.get("row_loss")),
                               _ptr(o["grad_hidden"]), _ptr(o["grad_weight"]), _ptr(workspace),
                               workspace.numel(), _stream(stream))
    if s != FLCE_OK:
        raise FlceError(s, "flce_fwd_bwd")
    o["workspace"] = workspace
    return o


def rmsnorm_fwd_bwd(hidden: torch.Tensor, gain: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                    eps: float = 1e-6, ignore_index: int = -100, reduction: str = "mean", *,
                    workspace: Optional[torch.Tensor] = None, row_loss: bool = False, out: Optional[dict] = None,
                    stream=None, grad_weight_dtype=torch.float32) -> dict:
    """Final RMSNorm (x = h / rms(h) * gain) fused in front of the LM head loss.

    grad_hidden is the gradient with respect to the pre-norm hidden states;
    grad_gain (fp32 [H]) and grad_weight ([V,H], fp32 or bf16) as the parameters'."""
    N, H, V = _check_inputs(hidden, weight, targets)
    if gain.dtype != torch.bfloat16 or gain.shape != (H,) or not gain.is_cuda or not gain.is_contiguous():
        raise ValueError("gain must be a contiguous bf16 CUDA tensor of shape [H]")
    dev = hidden.device
    flags = _flags(reduction, grad_weight_dtype)
    if workspace is None:
        nb = library().flce_rmsnorm_workspace_bytes(N, H, V, flags)
        if nb == 0:
            raise FlceError(FLCE_EINVAL, "workspace size")
        workspace = new_workspace(nb, dev)
    o = out if out is not None else {}
    if "loss" not in o:
        o["loss"] = torch.empty(1, dtype=torch.float32, device=dev)
        o["n_valid"] = torch.empty(1, dtype=torch.int32, device=dev)
        o["grad_hidden"] = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        o["grad_gain"] = torch.empty(H, dtype=torch.float32, device=dev)
        o["grad_weight"] = torch.empty((V, H), dtype=grad_weight_dtype, device=dev)
        o["row_loss"] = torch.empty(N, dtype=torch.float32, device=dev) if row_loss else None
    if o["grad_weight"].dtype != grad_weight_dtype:
        raise TypeError("out['grad_weight'] does not have grad_weight_dtype")
    s = library().flce_rmsnorm_fwd_bwd(_ptr(hidden), _ptr(gain), float(eps), _ptr(weight), _ptr(targets), N, H, V,
                                       int(ignore_index), flags, _ptr(o["loss"]), _ptr(o["n_valid"]),
                                       _ptr(o.get("row_loss")), _ptr(o["grad_hidden"]), _ptr(o["grad_gain"]),
                                       _ptr(o["grad_weight"]), _ptr(workspace), workspace.numel(), _stream(stream))
    if s != FLCE_OK:
        raise FlceError(s, "flce_rmsnorm_fwd_bwd")
    o["workspace"] = workspace
    return o


def loss(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor, ignore_index: int = -100,
         reduction: str = "mean", *, workspace: Optional[torch.Tensor] = None, row_loss: bool = False,
         out: Optional[dict] = None, stream=None) -> dict:
    """Forward only: loss, n_valid and optionally the per-token loss."""
    N, H, V = _check_inputs(hidden, weight, targets)
    dev = hidden.device
    if workspace is None:
        workspace = new_workspace(workspace_bytes(N, H, V, reduction, forward_only=True), dev)
    o = out if out is not None else {}
    if "loss" not in o:
        o["loss"] = torch.empty(1, dtype=torch.float32, device=dev)
        o["n_valid"] = torch.empty(1, dtype=torch.int32, device=dev)
        o["row_loss"] = torch.empty(N, dtype=torch.float32, device=dev) if row_loss else None
    s = library().flce_loss(_ptr(hidden), _ptr(weight), _ptr(targets), N, H, V, int(ignore_index),
                            REDUCE[reduction], _ptr(o["loss"]), _ptr(o["n_valid"]), _ptr(o.get("row_loss")),
                            _ptr(workspace), workspace.numel(), _stream(stream))
    if s != FLCE_OK:
        raise FlceError(s, "flce_loss")
    o["workspace"] = workspace
    return o


# ---------------------------------------------------------------------------
# vocabulary-parallel LM head (see include/flce.h); the collectives between
# the calls are the caller's
# ---------------------------------------------------------------------------

def _ok(s, what):
    if s != FLCE_OK:
        raise FlceError(s, what)


def vocab_shard_stats(hidden, weight_shard, targets, v0: int, V_total: int, ignore_index: int = -100,
                      workspace=None, stream=None) -> dict:
    N, H = hidden.shape
    Vs = weight_shard.shape[0]
    dev = hidden.device
    if workspace is None:
        workspace = new_workspace(library().flce_vocab_shard_workspace_bytes(N, H, Vs, 0), dev)
    o = {k: torch.empty(N, dtype=torch.float32, device=dev) for k in ("row_max", "row_sumexp", "row_target_logit")}
    o["n_valid"] = torch.empty(1, dtype=torch.int32, device=dev)
    _ok(library().flce_vocab_shard_stats(_ptr(hidden), _ptr(weight_shard), _ptr(targets), N, H, Vs, v0, V_total,
                                         int(ignore_index), _ptr(o["row_max"]), _ptr(o["row_sumexp"]),
                                         _ptr(o["row_target_logit"]), _ptr(o["n_valid"]), _ptr(workspace),
                                         workspace.numel(), _stream(stream)), "flce_vocab_shard_stats")
    o["workspace"] = workspace
    return o


def vocab_rescale(row_max_local, row_max_global, row_sumexp, stream=None) -> None:
    _ok(library().flce_vocab_rescale(_ptr(row_max_local), _ptr(row_max_global), _ptr(row_sumexp),
                                     row_sumexp.numel(), _stream(stream)), "flce_vocab_rescale")


def vocab_finish(row_max, row_sumexp, row_target_logit, targets, ignore_index: int = -100,
                 reduction: str = "mean", stream=None) -> dict:
    N = targets.shape[0]
    dev = targets.device
    o = {"lse": torch.empty(N, dtype=torch.float32, device=dev),
         "row_loss": torch.empty(N, dtype=torch.float32, device=dev),
         "loss": torch.empty(1, dtype=torch.float32, device=dev),
         "n_valid": torch.empty(1, dtype=torch.int32, device=dev)}
    _ok(library().flce_vocab_finish(_ptr(row_max), _ptr(row_sumexp), _ptr(row_target_logit), _ptr(targets), N,
                                    int(ignore_index), REDUCE[reduction], _ptr(o["lse"]), _ptr(o["row_loss"]),
                                    _ptr(o["loss"]), _ptr(o["n_valid"]), _stream(stream)), "flce_vocab_finish")
    return o


def vocab_shard_bwd(hidden, weight_shard, targets, lse, v0: int, V_total: int, ignore_index: int = -100,
                    reduction: str = "mean", workspace=None, stream=None) -> dict:
    N, H = hidden.shape
    Vs = weight_shard.shape[0]
    dev = hidden.device
    if workspace is None:
        workspace = new_workspace(library().flce_vocab_shard_workspace_bytes(N, H, Vs, REDUCE[reduction]), dev)
    o = {"grad_hidden_partial": torch.empty((N, H), dtype=torch.float32, device=dev),
         "grad_weight": torch.empty((Vs, H), dtype=torch.float32, device=dev)}
    _ok(library().flce_vocab_shard_bwd(_ptr(hidden), _ptr(weight_shard), _ptr(targets), N, H, Vs, v0, V_total,
                                       int(ignore_index), REDUCE[reduction], _ptr(lse),
                                       _ptr(o["grad_hidden_partial"]), _ptr(o["grad_weight"]), _ptr(workspace),
                                       workspace.numel(), _stream(stream)), "flce_vocab_shard_bwd")
    o["workspace"] = workspace
    return o


def scale_grads(grad_hidden: torch.Tensor, grad_weight: torch.Tensor, scale: torch.Tensor, stream=None) -> None:
    """grad_hidden and grad_weight *= scale (a one-element fp32 CUDA tensor), in place, on the device."""
    if scale.dtype != torch.float32 or scale.numel() != 1 or not scale.is_cuda:
        raise TypeError("scale must be a one-element float32 CUDA tensor")
    N, H = grad_hidden.shape
    V = grad_weight.shape[0]
    s = library().flce_scale_grads(_ptr(grad_hidden), _ptr(grad_weight), N, H, V, _ptr(scale.contiguous()),
                                   _stream(stream))
    if s != FLCE_OK:
        raise FlceError(s, "flce_scale_grads")


class _LinearCrossEntropyFn(torch.autograd.Function):
    """Forward computes the loss and both gradients in one library call; the
    backward only scales those gradients by the incoming gradient of the loss."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, ignore_index, reduction):
        o = fwd_bwd(hidden.contiguous(), weight.contiguous(), targets.contiguous(), ignore_index, reduction)
        ctx.grads = (o["grad_hidden"], o["grad_weight"])
        ctx.n_valid = o["n_valid"]
        return o["loss"].reshape(())

    @staticmethod
    def backward(ctx, grad_loss):
        gh, gw = ctx.grads
        ctx.grads = None
        scale_grads(gh, gw, grad_loss.detach().reshape(1).to(torch.float32))
        # autograd casts grad_weight (fp32) to the weight's dtype if they differ
        return gh, gw, None, None, None


def linear_cross_entropy(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                         ignore_index: int = -100, reduction: str = "mean") -> torch.Tensor:
    """Drop-in for ``F.cross_entropy(hidden @ weight.T, targets, ignore_index=...)``
    with autograd support; the N x V logits are never materialised."""
    return _LinearCrossEntropyFn.apply(hidden, weight, targets, ignore_index, reduction)


class LinearCrossEntropy(torch.nn.Module):
    """LM head + cross-entropy as one module: ``loss = module(hidden, targets)``."""

    def __init__(self, weight: torch.Tensor, ignore_index: int = -100, reduction: str = "mean"):
        super().__init__()
        self.weight = torch.nn.Parameter(weight)
        self.ignore_index = ignore_index
        self.reduction = reduction

    def forward(self, hidden: torch.Tensor, targets: torch.Tensor) -> torch.Tensor:
        return linear_cross_entropy(hidden, self.weight, targets, self.ignore_index, self.reduction)


def query_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the device status of the last call."""
    return int(library().flce_query_status(_ptr(workspace), _stream(stream)))


def selftest_timeout(workspace: torch.Tensor, timeout_ns: int, stream=None) -> int:
    return int(library().flce_selftest_timeout(_ptr(workspace), int(timeout_ns), _stream(stream)))


def query_stall(workspace: torch.Tensor, stream=None) -> dict:
    """Where the first pipeline wait of the last call ran out of time (site 0: none)."""
    info = (ctypes.c_int32 * 4)()
    s = library().flce_query_stall(_ptr(workspace), info, _stream(stream))
    if s != FLCE_OK:
        raise FlceError(s, "flce_query_stall")
    return {"site": info[0], "cta_rank": info[1], "block": info[2], "count": info[3]}


def debug_arm_stall(timeout_ns: int) -> None:
    """Test hook: the next GEMM launch withholds one pipeline signal (see flce.h)."""
    s = library().flce_debug_arm_stall(int(timeout_ns))
    if s != FLCE_OK:
        raise FlceError(s, "flce_debug_arm_stall")


def profile_begin() -> None:
    """Record CUDA events around every GEMM launch of the following calls."""
    library().flce_profile_begin()


def profile_end() -> dict:
    """Synchronise the recorded events; per GEMM mode summed ms and launch counts."""
    ms = (ctypes.c_double * 3)()
    n = (ctypes.c_int64 * 3)()
    total = ctypes.c_int64()
    s = library().flce_profile_end(ms, n, ctypes.byref(total))
    if s != FLCE_OK:
        raise FlceError(s, "flce_profile_end")
    names = ("logits", "backward", "unused")
    return {"gemm_ms": dict(zip(names, list(ms))), "gemm_launches": dict(zip(names, list(n))),
            "kernel_launches": int(total.value)}


def version() -> str:
    return library().flce_version().decode()
