"""Shared helpers for the GPU parity tests (tolerances, oracle glue)."""
import numpy as np
import torch

from oracle import moe as omoe

# Tolerance on MoE outputs: relative error of each output element measured
# against its token's output scale, |got - ref| / max_i |ref[t, i]| (a normwise
# relative error per token):  max over all elements <= 1e-2, mean <= 1e-3.
# An element-wise ratio is not used: the hidden activation h is quantised to
# bf16 on both sides, and where the kernel's fp32 value and the oracle's fp64
# value sit on opposite sides of a bf16 rounding boundary the one-ulp flip moves
# an output element by ~1e-4 of the row scale, which is an unbounded ratio for
# an element that happens to be near zero.
MOE_MAX_REL = 1e-2
MOE_MEAN_REL = 1e-3
# Logprob tolerance (absolute).
LOGP_ABS = 1e-3


def rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-30)
    return np.abs(got - ref) / scale


def elem_rel_err(got: np.ndarray, ref: np.ndarray, floor: float = 1e-3) -> np.ndarray:
    """Element-wise relative error with an absolute floor: |got - ref| / max(|ref|, floor * max_i |ref[t, i]|).
    Used where both sides start from the same bf16 operands (the stage under test is fed the kernel's
    own input), so no bf16 rounding of an intermediate can flip between them."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    row = np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-30)
    return np.abs(got - ref) / np.maximum(np.abs(ref), floor * row)


def assert_elem_close(got, ref, what, max_rel=MOE_MAX_REL, mean_rel=MOE_MEAN_REL):
    r = elem_rel_err(got, ref)
    assert r.max() <= max_rel and r.mean() <= mean_rel, (
        f"{what}: element-wise (floored) max rel {r.max():.3e} (<= {max_rel}), mean {r.mean():.3e} (<= {mean_rel})")
    return r


def assert_moe_close(got, ref, what="out"):
    r = rel_err(got, ref)
    e = elem_rel_err(got, ref)
    assert r.max() <= MOE_MAX_REL and r.mean() <= MOE_MEAN_REL, (
        f"{what}: max rel {r.max():.3e} (<= {MOE_MAX_REL}), mean rel {r.mean():.3e} (<= {MOE_MEAN_REL}); "
        f"element-wise (floored) max {e.max():.3e}, mean {e.mean():.3e}")
    return r


def f64(t):
    return omoe.to_f64(t)


def dot_bound(a64: np.ndarray, b64: np.ndarray, K: int) -> np.ndarray:
    """Error bound for an fp32-accumulated dot product of K bf16 products:
    |fl(sum) - sum| <= c * K * 2^-24 * sum |a||b| (c = 2 for slack on the
    tensor core's internal accumulation order)."""
    return 2.0 * K * 2.0 ** -24 * (np.abs(a64) @ np.abs(b64).T) + 1e-30


def check_topk(gpu_idx, gpu_logits_f32, ref_logits64, k, bound):
    """Exact index match except where the oracle's own ranking gap at a decided
    position is under the fp32 error bound; there, the oracle's top-k re-run on
    the GPU's float32 logits must match exactly.  Returns the number of tokens
    that needed the fp32 re-run."""
    gpu_idx = np.asarray(gpu_idx)
    ref_idx = omoe.topk_lowest_index(ref_logits64, k)
    mism = np.nonzero((gpu_idx != ref_idx).any(axis=1))[0]
    # every token: the oracle top-k on the GPU's own fp32 logits must match exactly
    same_prec = omoe.topk_lowest_index(np.asarray(gpu_logits_f32, np.float64), k)
    assert np.array_equal(gpu_idx, same_prec), "top-k disagrees with the oracle on the kernel's own logits"
    for t in mism:
        srt = np.sort(ref_logits64[t])[::-1]
        gaps = np.abs(np.diff(srt[: k + 1]))
        assert gaps.min() <= 2 * bound[t].max(), f"token {t}: index mismatch with gap {gaps.min()} > bound"
    return len(mism)


def sync():
    torch.cuda.synchronize()
