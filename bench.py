#!/usr/bin/env python
"""Benchmark of the fused linear cross-entropy forward+backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl flce|reference]

One step = one call of flce_fwd_bwd over one batch of seeded synthetic input
(all stages of the path: valid-row compaction, logits GEMM with the online
log-sum-exp epilogue, dlogits, the grad_hidden and grad_weight GEMMs, the
loss reduction).  Inputs are resident in HBM when the timed region starts;
the weight (1 GB at the default workload) is larger than L2, so no flush is
needed between steps.  Rank 0 prints one JSON line.

With torchrun (N > 1) every rank runs an independent replica on its own
batch (weak scaling): the path has no exchange step.

``--impl reference`` times the fp64 CPU oracle instead (a deliberately slow
program), each step a bounded sample of rows of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused linear-CE fwd+bwd tokens/s and % of GB300 dense BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# The sources that define and launch flce_gemm_kernel (the kernel whose DRAM
# traffic the roofline reports): the kernel, its PTX helpers and shared
# declarations, and the host code that plans and launches it.
GEMM_SOURCES = ("flce_gemm.cu", "flce_ptx.cuh", "flce_internal.h", "flce_api.cu")


def kernel_sources_sha1() -> str:
    """Hash of the GEMM kernel's sources with comments and blank space removed,
    so that DRAM counters taken on one build stay attached to it across
    comment edits and changes to the other kernels."""
    import hashlib
    import re
    h = hashlib.sha1()
    for name in GEMM_SOURCES:
        f = os.path.join(ROOT, "linear_cross_entropy_ce_gb300", "csrc", name)
        if not os.path.exists(f):
            continue
        with open(f, "r", encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = re.sub(r"\s+", " ", src).strip()
        h.update(os.path.basename(f).encode() + b"\0" + src.encode())
    return h.hexdigest()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(dev_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev_index] if vis else str(dev_index)


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------
class OracleSampler:
    """The fp64 oracle, as it stands, timed on samples of one workload.

    One sample = the full forward+backward of the oracle (steps 2-8 of
    ``oracle.flce_oracle_f64``: logits, log-sum-exp, losses, dz, grad_hidden
    and grad_weight) on the first `rows` valid tokens with the whole weight.
    The bf16 -> fp64 decode of the weight (4.2 GB of fp64 at the Llama-3-8B
    head) is done once, outside every timed sample, so that a sample measures
    the oracle's arithmetic and not a fixed decoding cost.  The benchmark's
    cpu_baseline leg and the --impl reference arm use the same sample size,
    chosen from a 64-row probe to take about `step_s` seconds."""

    def __init__(self, p, step_s=3.0):
        import numpy as np
        from oracle import decode_bf16
        self.p = p
        self.W64 = decode_bf16(p["weight"])
        self.valid = np.nonzero(p["targets"] != -100)[0]
        dt = self.time(64)
        self.rows = int(max(64, min(4096, self.valid.size, 64 * step_s / max(dt, 1e-3))))

    def time(self, rows=None):
        from oracle import decode_bf16, flce_oracle_f64
        sel = self.valid[:rows or self.rows]
        X64 = decode_bf16(self.p["hidden"][sel])
        t0 = time.perf_counter()
        flce_oracle_f64(X64, self.W64, self.p["targets"][sel])
        return time.perf_counter() - t0

    def sample_name(self):
        w = self.p["workload"]
        return (f"fp64 numpy oracle, full fwd+bwd of the first {self.rows} valid tokens of {w.name} "
                f"(H={w.H}, V={w.V}, full weight, weight decoded once outside the timing) per step")


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def cpu_baseline(p, steps=4):
    # a few steps of the sampler (about 10-15 s of CPU work in all)
    s = OracleSampler(p)
    ts = [s.time() for _ in range(steps)]
    return {"value": steps * s.rows / sum(ts), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{s.sample_name()}; {steps} steps, {sum(ts):.2f} s"}


def run_reference(args):
    import numpy as np  # noqa: F401
    from linear_cross_entropy_ce_gb300 import workloads as wl
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.workload]
    p = wl.make_inputs(w)
    s = OracleSampler(p)          # the same sample rule as the cpu_baseline leg
    for _ in range(args.warmup):
        s.time()
    times = [s.time() for _ in range(args.steps)]
    ms = 1000.0 * sum(times) / len(times)
    n = s.rows
    value = n / (ms / 1000.0)
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "N": w.N, "H": w.H, "V": w.V, "sample_rows_per_step": n},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": s.sample_name()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# widened forms of the path (one GPU, one JSON line each; not the contract line)
# ---------------------------------------------------------------------------
def run_variant(args) -> int:
    """Time one widened form of the path at the chosen workload:

    loss            the forward-only loss (flce_loss: 2*n_valid*H*V flops)
    rmsnorm         the final RMSNorm fused in front (flce_rmsnorm_fwd_bwd)
    autograd        LinearCrossEntropy forward + backward with grad_output 2.5
                    (the library call plus the flce_scale_grads pass)
    vocab_parallel  one rank's share of a vocabulary-parallel LM head over
                    --shards ranks: shard statistics, the lse finish (the
                    exchange between them is three N-float all-reduces, left
                    out on one GPU) and the shard backward
    """
    import numpy as np
    import torch
    from linear_cross_entropy_ce_gb300 import flce, workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flce.library()
    w = wl.WORKLOADS[args.workload]
    p = wl.make_inputs(w)
    N, H, V = w.N, w.H, w.V
    h = torch.from_numpy(p["hidden"].view(np.int16)).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(p["weight"].view(np.int16)).view(torch.bfloat16).to(dev)
    t = torch.from_numpy(p["targets"]).to(dev)
    nv = int((p["targets"] != -100).sum())
    flops = 6.0 * nv * H * V
    cfg = {"workload": w.name, "N": N, "H": H, "V": V, "n_valid": nv}

    if args.variant == "loss":
        ws = flce.new_workspace(flce.workspace_bytes(N, H, V, forward_only=True), dev)
        out = {}

        def step():
            flce.loss(h, W, t, workspace=ws, out=out)
        flops = 2.0 * nv * H * V
        cfg["workspace_bytes"] = ws.numel()
        cfg["flops_note"] = "2*n_valid*H*V (logits only)"
    elif args.variant == "rmsnorm":
        gain = (1.0 + 0.1 * torch.randn(H, generator=torch.Generator().manual_seed(5))).to(torch.bfloat16).to(dev)
        ws = flce.new_workspace(flce.library().flce_rmsnorm_workspace_bytes(N, H, V, 0), dev)
        out = {}

        def step():
            flce.rmsnorm_fwd_bwd(h, gain, W, t, workspace=ws, out=out)
        cfg["workspace_bytes"] = ws.numel()
    elif args.variant == "autograd":
        hp = h.clone().requires_grad_(True)
        Wp = W.clone().requires_grad_(True)
        g = torch.full((), 2.5, device=dev)

        def step():
            hp.grad = None
            Wp.grad = None
            loss = flce.linear_cross_entropy(hp, Wp, t)
            loss.backward(g)
    elif args.variant == "vocab_parallel":
        P = args.shards
        Vs = (V + P - 1) // P
        Wsh = W[:Vs].contiguous()
        ws_s = flce.new_workspace(flce.library().flce_vocab_shard_workspace_bytes(N, H, Vs, 0), dev)
        ws_b = flce.new_workspace(flce.library().flce_vocab_shard_workspace_bytes(N, H, Vs, 0), dev)

        def step():
            st = flce.vocab_shard_stats(h, Wsh, t, 0, V, workspace=ws_s)
            fin = flce.vocab_finish(st["row_max"], st["row_sumexp"], st["row_target_logit"], t)
            flce.vocab_shard_bwd(h, Wsh, t, fin["lse"], 0, V, workspace=ws_b)
        flops = 6.0 * nv * H * Vs
        cfg.update({"shards": P, "V_shard": Vs, "flops_note": "per-rank share 6*n_valid*H*V/P; the shard "
                    "backward recomputes the shard's logits (8*N*H*V/P actual)"})
    else:
        raise SystemExit(f"unknown variant {args.variant}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_id_for(0))
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    pk, src = peaks()
    line = {"metric": METRIC, "variant": args.variant, "value": N / (ms / 1000.0), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic", "config": cfg,
            "pct_bf16_peak": {"value": 100.0 * flops / (ms / 1000.0) / 1e12 / float(pk["bf16_tflops"]),
                              "basis": f"{src} bf16 burst peak"},
            "clocks": clk}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama3_8b_head")
    ap.add_argument("--impl", default="flce", choices=["flce", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--tokens", type=int, default=None, help="override N (small profiling cases)")
    ap.add_argument("--chunk-rows", type=int, default=None, help="override the default 5%% plan")
    ap.add_argument("--workspace-bytes", type=int, default=None,
                    help="workspace size to plan for (small profiling cases that keep a full-size plan)")
    ap.add_argument("--variant", default=None, choices=["loss", "rmsnorm", "autograd", "vocab_parallel"],
                    help="time a widened form of the path instead (one GPU; not the contract line)")
    ap.add_argument("--shards", type=int, default=2, help="vocabulary shards for --variant vocab_parallel")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "flce":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.variant:
        return run_variant(args)

    import numpy as np
    import torch
    import torch.distributed as dist
    from linear_cross_entropy_ce_gb300 import flce, workloads as wl
    from linear_cross_entropy_ce_gb300 import dist as fdist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # device memory before the library is loaded (the context exists already)
    torch.zeros(1, device=dev)
    torch.cuda.synchronize()
    free_before_lib = torch.cuda.mem_get_info(dev)[0]
    flce.library()
    free_after_lib = torch.cuda.mem_get_info(dev)[0]

    base = wl.WORKLOADS[args.workload]
    if args.tokens:
        base = base.with_shape(N=args.tokens)
    w = base.with_shape(seed=fdist.replica_seed(base.seed, rank))
    p = wl.make_inputs(w)
    N, H, V = w.N, w.H, w.V
    h = torch.from_numpy(p["hidden"].view(np.int16)).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(p["weight"].view(np.int16)).view(torch.bfloat16).to(dev)
    t = torch.from_numpy(p["targets"]).to(dev)
    nv = int((p["targets"] != -100).sum())
    ws_bytes = args.workspace_bytes or flce.workspace_bytes(N, H, V, chunk_rows=args.chunk_rows)
    plan = flce.plan(N, H, V, ws_bytes)
    ws = flce.new_workspace(ws_bytes, dev)
    out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
           "n_valid": torch.empty(1, dtype=torch.int32, device=dev),
           "grad_hidden": torch.empty((N, H), dtype=torch.bfloat16, device=dev),
           "grad_weight": torch.empty((V, H), dtype=torch.float32, device=dev), "row_loss": None}
    stream = torch.cuda.current_stream()

    # every step writes its loss into its own slot, so that a failed step
    # (its loss is NaN) is seen after the timed loop
    loss_slots = torch.full((max(args.steps, args.warmup),), float("nan"), dtype=torch.float32, device=dev)

    def step(i):
        out["loss"] = loss_slots[i:i + 1]
        flce.fwd_bwd(h, W, t, workspace=ws, out=out, stream=stream)

    def check_steps(what, losses):
        st_ = flce.query_status(ws)
        if st_ != flce.FLCE_OK:
            raise RuntimeError(f"{what}: device status {flce.STATUS_NAMES[st_]}")
        if not bool(torch.isfinite(losses).all()):
            raise RuntimeError(f"{what}: a step reported a NaN loss (device-side failure)")

    # measured extra device memory: what the library's first calls take
    # beyond the caller's buffers (module load, static data), and what the
    # caching allocator hands out during a call (nothing: the caller owns every buffer)
    torch.cuda.synchronize()
    free_before_call = torch.cuda.mem_get_info(dev)[0]
    reserved_before_call = torch.cuda.memory_reserved(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    alloc_before_call = torch.cuda.memory_allocated(dev)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    free_after_call = torch.cuda.mem_get_info(dev)[0]
    lib_bytes = (free_before_lib - free_after_lib) + (free_before_call - free_after_call) \
        - (torch.cuda.memory_reserved(dev) - reserved_before_call)
    torch_peak_bytes = torch.cuda.max_memory_allocated(dev) - alloc_before_call
    check_steps("warm-up", loss_slots[:args.warmup])

    clocks = ClockSampler(gpu_id_for(local))
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    flce.profile_begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    prof = flce.profile_end()
    clk = clocks.stop()
    check_steps("timed steps", loss_slots[:args.steps])
    ms = fdist.max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)

    # end to end through the public API: pinned host inputs in, loss out, every
    # step.  As a data loader would, step i+1's inputs are copied on a second
    # stream while step i computes (two device input buffers); every copy lies
    # inside the timed region.
    e2e = None
    if not args.no_e2e:
        h_host = torch.from_numpy(p["hidden"].view(np.int16)).view(torch.bfloat16).pin_memory()
        t_host = torch.from_numpy(p["targets"]).pin_memory()
        loss_host = torch.full((args.steps + 2, 2), float("nan"), dtype=torch.float32).pin_memory()
        h_dev = [torch.empty_like(h), torch.empty_like(h)]
        t_dev = [torch.empty_like(t), torch.empty_like(t)]
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        consumed = [torch.cuda.Event(), torch.cuda.Event()]
        out["loss"] = loss_slots[0:1]

        def copy_in(b):
            with torch.cuda.stream(copy_stream):
                h_dev[b].copy_(h_host, non_blocking=True)
                t_dev[b].copy_(t_host, non_blocking=True)
            copied[b].record(copy_stream)

        def e2e_run(n, first_slot, start_event=None):
            if start_event is not None:
                copy_stream.wait_event(start_event)
            copy_in(0)
            for i in range(n):
                b = i % 2
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(consumed[(i + 1) % 2])   # step i-1 is done with that buffer
                    copy_in((i + 1) % 2)
                stream.wait_event(copied[b])
                flce.fwd_bwd(h_dev[b], W, t_dev[b], workspace=ws, out=out, stream=stream)
                consumed[b].record(stream)
                loss_host[first_slot + i, 0:1].copy_(out["loss"], non_blocking=True)
                loss_host[first_slot + i, 1:2].copy_(out["n_valid"].view(torch.float32), non_blocking=True)
        e2e_run(2, args.steps)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        e2e_run(args.steps, 0, start_event=a0)
        a1.record(stream)
        torch.cuda.synchronize()
        check_steps("e2e steps", loss_host[:, 0])
        e2e_ms = fdist.max_over_ranks(a0.elapsed_time(a1) / args.steps, dev)
        e2e = {"value": world * N / (e2e_ms / 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": N * H * 2 + N * 4, "d2h_bytes_per_step": 8,
               "ms_per_step": e2e_ms,
               "note": "hidden and targets copied from pinned host memory each step (the next step's copy on a "
                       "second stream, overlapping the current step), loss and n_valid read back; the weight "
                       "stays resident"}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    pk, src = peaks()
    flops_alg = 6.0 * nv * H * V
    gemm_ms = sum(prof["gemm_ms"].values())
    gemm_n = sum(prof["gemm_launches"].values())
    achieved = flops_alg * args.steps / (gemm_ms / 1000.0) / 1e12 if gemm_ms > 0 else None
    peak_s = float(pk["bf16_tflops_sustained"])
    peak_b = float(pk["bf16_tflops"])
    step_tflops = flops_alg / (ms / 1000.0) / 1e12
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            tj = json.load(open(tpath))
            # only valid for the kernel sources the counters were taken on
            if tj.get("workload") == w.name and tj.get("kernel_sources_sha1") == kernel_sources_sha1() \
                    and not args.tokens and not args.chunk_rows and not args.workspace_bytes:
                traffic = tj.get("dram_bytes_per_launch")
        except Exception:
            traffic = None
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak_s, "unit": "TFLOP/s",
            "frac": (achieved / peak_s) if achieved else None, "traffic": traffic,
            "kernel": "flce_gemm_kernel (tcgen05, all three GEMM modes)",
            "peak_source": f"{src} bf16_tflops_sustained (kernel timed inside a long step)",
            "flops_per_launch": flops_alg / max(1, gemm_n / args.steps),
            "avg_launch_ms": gemm_ms / max(1, gemm_n),
            "per_mode_ms_per_step": {k: v / args.steps for k, v in prof["gemm_ms"].items()}}
    if traffic is not None:
        # DRAM bytes the GEMM launches of one step move (ncu counters x launches) and their rate
        per_step = traffic * gemm_n / args.steps
        roof["dram_bytes_per_step"] = per_step
        roof["dram_gbs_during_gemm"] = per_step / (gemm_ms / args.steps / 1000.0) / 1e9
        roof["dram_frac_of_peak"] = roof["dram_gbs_during_gemm"] / float(pk["hbm_gbs"])
    line = {
        "metric": METRIC, "value": world * N / (ms / 1000.0), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "N": N, "H": H, "V": V, "n_valid": nv, "chunk_rows": plan["chunk_rows"],
                   "workspace_bytes": ws_bytes, "extra_mem_frac_of_NV2": ws_bytes / (N * V * 2),
                   "extra_mem_measured": {
                       "workspace_bytes": ws_bytes, "library_device_bytes": lib_bytes,
                       "torch_alloc_peak_bytes": torch_peak_bytes,
                       "frac_of_NV2": (ws_bytes + max(0, lib_bytes) + torch_peak_bytes) / (N * V * 2),
                       "how": "library_device_bytes: cudaMemGetInfo free-memory drop across loading libflce.so and "
                              "its warm-up calls, minus what the caching allocator reserved meanwhile (module code "
                              "and static device data); torch_alloc_peak_bytes: max_memory_allocated during the "
                              "calls minus allocated before them"},
                   "l2": "inputs larger than L2 (weight alone exceeds 129 MB), no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_bf16_peak": {"value": 100.0 * step_tflops / peak_b, "tflops_alg": step_tflops,
                          "basis": f"6*n_valid*H*V per step over step time, vs {src} bf16 burst peak {peak_b}",
                          "vs_sustained": 100.0 * step_tflops / peak_s},
        "roofline": roof,
        "gpu_launches": prof["kernel_launches"],
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
