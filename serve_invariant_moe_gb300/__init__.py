"""Batch-invariant MoE layer + logprob/KL head for one GB300 GPU (sm_103a).

The compute path is the C-ABI library ``libinvmoe.so`` (include/invmoe.h),
built in-tree by ``serve_invariant_moe_gb300.build``; ``binding`` marshals torch
tensors to it and ``api`` offers the prefill/decode entry points.  Importing
this package does not load the library; the first call does, and raises if it
is missing.
"""
__all__ = ["api", "binding", "build", "synth"]
