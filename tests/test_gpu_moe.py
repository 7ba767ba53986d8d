"""MoE layer on the GPU (through the C ABI) against the float64 CPU oracle.

Covers the router logits, the top-k indices (bit-exact, ties to the lower
index), the gates, the dispatch plan, the permuted activations, the grouped
SwiGLU experts and the fixed-order combine, on the tiny tied layer, on ragged
layers with empty experts and a ragged token count, and on the full-size
Qwen-MoE-like and GLM-scale layers on sampled tokens."""
import dataclasses

import numpy as np
import pytest
import torch

from helpers import assert_moe_close, check_topk, dot_bound, f64
from oracle import moe as omoe
from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _layer(cfg, dev="cuda", expert_device="cpu"):
    from serve_invariant_moe_gb300 import api
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, expert_device)
    ws13, ws2 = synth.shared_expert_weights(cfg, expert_device)
    layer = api.MoELayer(api.MoEWeights(wr.to(dev), w13.to(dev), w2.to(dev), cfg.k,
                                        None if ws13 is None else ws13.to(dev),
                                        None if ws2 is None else ws2.to(dev)))
    return x, wr, w13, w2, ws13, ws2, layer


def _check_route(res, x, wr, cfg):
    T, k, E, H = x.shape[0], cfg.k, cfg.E, cfg.H
    x64, wr64 = f64(x), f64(wr)
    ref_L = omoe.router_logits(x64, wr64)
    L = res["logits"].cpu().numpy()
    bound = dot_bound(x64, wr64, H)
    assert (np.abs(L - ref_L) <= bound).all(), "router logits outside the fp32 error bound"
    idx = res["topk_idx"].cpu().numpy()
    n_near = check_topk(idx, L, ref_L, k, bound)
    # gates: the oracle's softmax over the selected logits, evaluated on the kernel's own logits
    g_ref = omoe.topk_gates(L.astype(np.float64), idx)
    g = res["topk_w"].cpu().numpy()
    assert np.allclose(g, g_ref, rtol=4e-6, atol=1e-7)
    # plan: the oracle's counting sort of the kernel's own indices, bit-exact
    counts, offsets, row_token, slot_row = omoe.dispatch_plan(idx, E)
    plan = res["plan"].cpu().numpy()
    S = T * k
    assert np.array_equal(plan[:E], counts)
    assert np.array_equal(plan[E:2 * E + 1], offsets)
    assert np.array_equal(plan[2 * E + 1:2 * E + 1 + S], row_token)
    assert np.array_equal(plan[2 * E + 1 + S:2 * E + 1 + 2 * S], slot_row.ravel())
    # permuted activations are exact copies
    xp = res["xp"][:S].cpu()
    assert torch.equal(xp.view(torch.int16), x[torch.from_numpy(row_token)].view(torch.int16))
    return n_near


def test_tiny_layer_with_exact_ties():
    cfg = synth.TINY
    x, wr, w13, w2, _, _, layer = _layer(cfg)
    res = layer.prefill(x.cuda(), return_all=True)
    torch.cuda.synchronize()
    _check_route(res, x, wr, cfg)
    idx = res["topk_idx"].cpu().numpy()
    assert np.all(idx[:, 1] == idx[:, 0] + 1) and np.all(idx[:, 0] % 2 == 0)
    assert torch.equal(res["logits"][:, 0::2], res["logits"][:, 1::2])
    assert torch.all(res["topk_w"] == 0.5)
    ref = omoe.moe_forward(f64(x), f64(wr), f64(w13), f64(w2), cfg.k, cfg.F)
    assert_moe_close(res["out"].cpu().numpy(), ref["out"])
    # expert outputs per slot (before the combine)
    y = res["y"].cpu().numpy()[res["plan"].cpu().numpy()[2 * cfg.E + 1 + cfg.T * cfg.k:].reshape(cfg.T, cfg.k)]
    assert_moe_close(y.reshape(cfg.T * cfg.k, -1), ref["y"].reshape(cfg.T * cfg.k, -1), "y")


RAGGED = [
    # T not a multiple of 128; experts with 0 tokens; a few experts above 256 tokens
    dataclasses.replace(synth.TINY, name="ragged_a", T=333, H=256, E=16, k=3, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=1.5, seed=11),
    dataclasses.replace(synth.TINY, name="ragged_b", T=1, H=512, E=8, k=8, F=128,
                        dup_router_rows=False, seed=12),
    dataclasses.replace(synth.TINY, name="ragged_shared", T=190, H=384, E=12, k=4, F=384, F_shared=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=0.8, seed=13),
]


@pytest.mark.parametrize("cfg", RAGGED, ids=lambda c: c.name)
def test_ragged_layers(cfg):
    x, wr, w13, w2, ws13, ws2, layer = _layer(cfg)
    res = layer.prefill(x.cuda(), return_all=True)
    torch.cuda.synchronize()
    _check_route(res, x, wr, cfg)
    counts = res["plan"][:cfg.E].cpu().numpy()
    ref = omoe.moe_forward(f64(x), f64(wr), f64(w13), f64(w2), cfg.k, cfg.F,
                           None if ws13 is None else f64(ws13), None if ws2 is None else f64(ws2), cfg.F_shared)
    assert_moe_close(res["out"].cpu().numpy(), ref["out"])
    if cfg.name == "ragged_a":
        assert (counts == 0).any() and counts.max() > 256


def test_all_experts_k_equals_e_matches_sparse_rows_bitwise():
    """Route every token to every expert (k = E): each (token, expert) row of Y
    must equal, bit for bit, the same row computed in a sparse k=2 run -- the
    rows land at different tile positions in the two runs."""
    from serve_invariant_moe_gb300 import api
    cfg = dataclasses.replace(synth.TINY, name="dense_vs_sparse", T=200, H=256, E=8, k=2, F=256,
                              dup_router_rows=False, seed=21)
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg)
    dense = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), cfg.E)).prefill(x.cuda(), return_all=True)
    sparse = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), 2)).prefill(x.cuda(), return_all=True)
    torch.cuda.synchronize()
    E, T = cfg.E, cfg.T
    d_idx = dense["topk_idx"].cpu().numpy()
    d_slot = dense["plan"].cpu().numpy()[2 * E + 1 + T * E:].reshape(T, E)
    s_idx = sparse["topk_idx"].cpu().numpy()
    s_slot = sparse["plan"].cpu().numpy()[2 * E + 1 + T * 2:].reshape(T, 2)
    dy, sy = dense["y"].cpu(), sparse["y"].cpu()
    dh, sh = dense["h"].cpu(), sparse["h"].cpu()
    for t in range(T):
        for j in range(2):
            e = s_idx[t, j]
            jd = int(np.nonzero(d_idx[t] == e)[0][0])
            assert torch.equal(dy[d_slot[t, jd]], sy[s_slot[t, j]]), (t, e)
            assert torch.equal(dh[d_slot[t, jd]].view(torch.int16), sh[s_slot[t, j]].view(torch.int16))
    # and the dense run agrees with the brute-force oracle
    ref = omoe.dense_all_experts_then_mask(f64(x), f64(wr), f64(w13), f64(w2), E, cfg.F)
    assert_moe_close(dense["out"].cpu().numpy(), ref)


def _sampled_oracle(x, wr, w13_dev, w2_dev, cfg, tokens, idx_gpu, L_gpu, ws13=None, ws2=None):
    """Oracle output for a few tokens, pulling only the experts they use."""
    xs = f64(x[tokens])
    L = omoe.router_logits(xs, f64(wr))
    idx = omoe.topk_lowest_index(L, cfg.k)
    gates = omoe.topk_gates(L, idx)
    cache = {}

    def ew(e):
        if e not in cache:
            cache[e] = (f64(w13_dev[e].cpu()), f64(w2_dev[e].cpu()))
        return cache[e]
    y = omoe.expert_outputs(xs, idx, None, None, cfg.F, expert_weights=ew)
    ys = None
    if ws13 is not None:
        ys = omoe.swiglu_expert(xs, f64(ws13.cpu()), f64(ws2.cpu()), cfg.F_shared)
    return dict(L=L, idx=idx, out=omoe.combine(y, gates, ys))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen_moe_like", "qwen_moe_like_empty", "glm_scale_moe"])
def test_full_size_layer_sampled_tokens(name):
    from serve_invariant_moe_gb300 import api
    cfg = synth.CONFIGS[name]
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    ws13, ws2 = synth.shared_expert_weights(cfg, "cuda")
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13, w2, cfg.k, ws13, ws2))
    res = layer.prefill(x.cuda(), return_all=True)
    torch.cuda.synchronize()
    counts = res["plan"][:cfg.E].cpu().numpy()
    assert counts.sum() == cfg.T * cfg.k
    if cfg.zipf_starve:
        assert (counts == 0).sum() == cfg.zipf_starve and 1200 <= counts.max() <= 1800
    # whole-batch properties: logits in bound, top-k exact on the kernel's logits, plan bit-exact
    _check_route(res, x, wr, cfg)
    g = torch.Generator().manual_seed(5)
    tokens = torch.randperm(cfg.T, generator=g)[:6].tolist() + [0, cfg.T - 1]
    ref = _sampled_oracle(x, wr, w13, w2, cfg, tokens, res["topk_idx"], res["logits"], ws13, ws2)
    assert np.array_equal(res["topk_idx"].cpu().numpy()[tokens], ref["idx"])
    assert_moe_close(res["out"].cpu().numpy()[tokens], ref["out"])
    assert torch.isfinite(res["out"]).all()
