"""Shared helpers for the GPU parity tests (conversion and error metrics)."""
import numpy as np

LOSS_RTOL = 2e-3      # |loss_gpu - loss_ref| / |loss_ref|
GRAD_FROB_RTOL = 1e-2 # ||G_gpu - G_ref||_F / ||G_ref||_F  (bf16 in, fp32 accumulate)


def to_device(p, dev):
    import torch
    h = torch.from_numpy(np.ascontiguousarray(p["hidden"]).view(np.int16)).view(torch.bfloat16).to(dev)
    w = torch.from_numpy(np.ascontiguousarray(p["weight"]).view(np.int16)).view(torch.bfloat16).to(dev)
    t = torch.from_numpy(np.ascontiguousarray(p["targets"])).to(dev)
    return h, w, t


def frob_rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    d = np.linalg.norm(a - b)
    return d / nb if nb > 0 else d


def loss_rel(a, b):
    return abs(a - b) / abs(b) if b != 0 else abs(a - b)


def gh_np(t):
    return t.float().cpu().double().numpy()
