"""Module substitution: each stage of the MoE layer checked on its own, fed the GPU's own input.

"Reinforcement Learning: Why Numerical Alignment and MoE Routing Matter So Much", section
"混合专家模型更难对齐": a train/serve mismatch was localised by swapping one module (the MoE
block) for a reference implementation.  Here the same idea runs stage by stage: the oracle's
gate/up stage gets the kernel's permuted rows xp, the oracle's down projection gets the
kernel's hidden activation h, the oracle's combine gets the kernel's per-slot outputs Y and
gates.  No bf16 rounding of an intermediate can then flip between the two sides, so each
stage is held element by element, to a bound derived from its fp32 arithmetic, instead of
the end-to-end row-normalised tolerance.

At full size (the Zipf-skewed Qwen-like layer and the GLM-scale layer) the experts are chosen
for the tile paths that only run at size: an expert with more than 256 rows (a second row
chunk), one whose last 128-row tile holds 65..127 rows, one whose last tile holds at most 64
rows (the M = 64 tail), and the busiest expert.  Every row routed to them is compared.
"""
import dataclasses

import numpy as np
import pytest
import torch

from helpers import assert_elem_close, assert_moe_close, dot_bound, elem_rel_err, f64
from oracle import moe as omoe
from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24          # unit roundoff of fp32


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def _pick_experts(counts):
    """Experts exercising the full-size tile paths, by their row count n_e (0 if none qualifies)."""
    picks = {}
    order = np.argsort(-counts, kind="stable")
    picks["busiest"] = int(order[0])
    over = [e for e in order if counts[e] > 256]
    if over:
        picks["second_row_chunk"] = int(over[len(over) // 2])
    tail_mid = [e for e in order if 65 <= counts[e] % 128 <= 127]
    if tail_mid:
        picks["last_tile_65_127"] = int(tail_mid[0])
    tail_small = [e for e in order if 1 <= counts[e] % 128 <= 64 and counts[e] > 128]
    if tail_small:
        picks["last_tile_m64"] = int(tail_small[0])
    return picks


def _check_expert_stages(e, res, w13_e, w2_e, F, what):
    """Gate/up stage on the kernel's xp rows, then the down projection on the kernel's h rows."""
    plan = res["plan_np"]
    off, n = plan["offsets"][e], plan["counts"][e]
    xp = f64(res["xp"][off:off + n].cpu())
    h_gpu = f64(res["h"][off:off + n].cpu())
    y_gpu = res["y"][off:off + n].double().cpu().numpy()
    w13 = f64(w13_e.cpu())
    w2 = f64(w2_e.cpu())
    # stage 1: h = bf16(silu(x Wg^T) * (x Wu^T)) on the kernel's own xp rows
    h_ref = omoe.swiglu_hidden(xp, w13, F, round_h=True)
    exact = (h_gpu == h_ref).mean()
    assert exact >= 0.99, f"{what}: expert {e}: only {exact:.4f} of h elements bit-equal to the oracle's"
    # every element within its error bound: half a bf16 ulp for the final rounding, plus the fp32
    # error of the gate and up dot products (H terms each) carried through h = silu(g) * u
    # (|silu'| <= 1.1), plus a few fp32 ulps for silu and the product
    H = xp.shape[1]
    h64 = omoe.swiglu_hidden(xp, w13, F, round_h=False)
    u64 = xp @ w13[F:2 * F].T
    sg = h64 / np.where(u64 == 0, 1.0, u64)          # silu(g), where u != 0
    dg = dot_bound(xp, w13[:F], H)
    du = dot_bound(xp, w13[F:2 * F], H)
    tol = (0.5 * _bf16_ulp(np.maximum(np.abs(h64), np.abs(h_gpu))) * 1.0001
           + 1.1 * np.abs(u64) * dg + np.abs(sg) * du + 8 * U32 * np.abs(h64))
    assert (np.abs(h_gpu - h64) <= tol + 1e-30).all(), f"{what}: expert {e}: an h element is outside its bound"
    assert_elem_close(h_gpu, h_ref, f"{what}: expert {e} h")
    # stage 2: y = h W2^T on the kernel's own h, fp32 accumulation over F terms
    y_ref = omoe.down_projection(h_gpu, w2)
    bound = dot_bound(h_gpu, w2, F)
    assert (np.abs(y_gpu - y_ref) <= bound).all(), f"{what}: expert {e}: Y outside the fp32 dot-product bound"
    r = assert_elem_close(y_gpu, y_ref, f"{what}: expert {e} Y")
    return float(exact), float(r.max())


def _check_combine(res, T, k, H, what, chunk=512):
    """The oracle's combine on the kernel's own Y rows, gates and shared-expert rows, every token."""
    slot_row = res["plan_np"]["slot_row"]
    worst = 0.0
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        rows = torch.from_numpy(slot_row[t0:t1].ravel()).long().to(res["y"].device)
        y = res["y"][rows].double().cpu().numpy().reshape(t1 - t0, k, H)
        g = res["topk_w"][t0:t1].double().cpu().numpy()
        ys = None if res.get("y_shared") is None else res["y_shared"][t0:t1].double().cpu().numpy()
        ref = omoe.combine(y, g, ys)
        out = res["out"][t0:t1].double().cpu().numpy()
        # k products and k sums (plus the shared expert), each rounded once in fp32
        mag = np.einsum("tj,tjh->th", np.abs(g), np.abs(y)) + (0.0 if ys is None else np.abs(ys))
        bound = 2.0 * (k + 2) * U32 * mag + 1e-30
        assert (np.abs(out - ref) <= bound).all(), f"{what}: combine outside its fp32 bound (tokens {t0}..{t1})"
        worst = max(worst, float(elem_rel_err(out, ref).max()))
    assert worst <= 1e-2, f"{what}: combine element-wise max rel {worst:.3e}"
    return worst


def _plan_np(plan, T, E, k):
    p = plan.cpu().numpy()
    S = T * k
    return dict(counts=p[:E], offsets=p[E:2 * E + 1], row_token=p[2 * E + 1:2 * E + 1 + S],
                slot_row=p[2 * E + 1 + S:2 * E + 1 + 2 * S].reshape(T, k))


def _run_layer(cfg, expert_device):
    from serve_invariant_moe_gb300 import api
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, expert_device)
    ws13, ws2 = synth.shared_expert_weights(cfg, expert_device)
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), cfg.k,
                                        None if ws13 is None else ws13.cuda(), None if ws2 is None else ws2.cuda()))
    res = layer.prefill(x.cuda(), return_all=True)
    torch.cuda.synchronize()
    res["plan_np"] = _plan_np(res["plan"], cfg.T, cfg.E, cfg.k)
    return x, w13, w2, ws13, ws2, res


SMALL = [
    dataclasses.replace(synth.TINY, name="ragged_skew", T=700, H=256, E=8, k=3, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=1.2, seed=31),
    dataclasses.replace(synth.TINY, name="ragged_shared", T=190, H=384, E=12, k=4, F=384, F_shared=256,
                        dup_router_rows=False, seed=13),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_stages_small_layers_every_expert(cfg):
    x, w13, w2, ws13, ws2, res = _run_layer(cfg, "cpu")
    counts = res["plan_np"]["counts"]
    for e in range(cfg.E):
        if counts[e]:
            _check_expert_stages(e, res, w13[e], w2[e], cfg.F, cfg.name)
    _check_combine(res, cfg.T, cfg.k, cfg.H, cfg.name)
    if ws13 is not None:
        # the shared expert's hidden rows stay inside the call, so its output is held to the
        # end-to-end (row-normalised) tolerance
        ref = omoe.swiglu_expert(f64(x), f64(ws13), f64(ws2), cfg.F_shared)
        assert_moe_close(res["y_shared"].double().cpu().numpy(), ref, f"{cfg.name}: shared expert")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen_moe_like", "qwen_moe_like_empty", "glm_scale_moe"])
def test_stages_full_size_tile_paths(name):
    cfg = synth.CONFIGS[name]
    x, w13, w2, ws13, ws2, res = _run_layer(cfg, "cuda")
    counts = res["plan_np"]["counts"]
    picks = _pick_experts(counts)
    # each tile path this workload has must be covered
    assert "busiest" in picks and "second_row_chunk" in picks
    assert "last_tile_65_127" in picks or not any(65 <= c % 128 <= 127 for c in counts)
    assert "last_tile_m64" in picks or not any(1 <= c % 128 <= 64 and c > 128 for c in counts)
    if name.startswith("qwen_moe_like"):
        assert counts[picks["busiest"]] > 1200      # the ~1500-row expert of the Zipf head
    if cfg.zipf_starve:
        assert (counts == 0).sum() == cfg.zipf_starve   # empty experts at full size
    for kind, e in picks.items():
        _check_expert_stages(e, res, w13[e], w2[e], cfg.F, f"{name} {kind} (n={counts[e]})")
    _check_combine(res, cfg.T, cfg.k, cfg.H, name)
