"""Fused linear cross-entropy (LM head) for GB300 (sm_103a).

The compute path is ``libflce.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/flce.h``); ``linear_cross_entropy_ce_gb300.flce`` is the
thin ctypes binding.  ``workloads`` draws the seeded synthetic inputs.
"""
