"""Edge cases through the C ABI: empty inputs, the largest top-k, NaN activations,
k = 1, every token on one expert, and repeated tokens in one batch."""
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


def test_empty_batch_through_every_entry_point():
    from serve_invariant_moe_gb300 import _lib, binding
    lib = _lib.lib()
    H, E, k, F, V = 256, 8, 2, 256, 512
    ws = binding.new_workspace(binding.workspace_size(0, H, E, k, F, 128, V))
    plan = torch.full((binding.plan_len(0, E, k),), -7, dtype=torch.int32, device="cuda")
    stream = binding._stream()
    assert lib.moe_route_topk(None, None, 0, H, E, k, None, None, None, binding._p(plan), None,
                              binding._p(ws), ws.numel(), stream) == 0
    torch.cuda.synchronize()
    assert torch.all(plan[: 2 * E + 1] == 0)          # counts and offsets of an empty batch
    assert lib.moe_grouped_ffn(None, binding._p(plan), None, None, 0, H, E, k, F, None, None, None, None, None, 0,
                               None, binding._p(ws), ws.numel(), stream) == 0
    assert lib.moe_combine(None, None, binding._p(plan), None, 0, H, E, k, None, None, stream) == 0
    assert lib.lm_logprob_kl(None, None, None, None, 0, H, V, 2.0, None, None, None, None, None,
                             binding._p(ws), ws.numel(), stream) == 0
    assert lib.rl_token_loss(None, None, None, None, 0, 2.0, 0.2, 0.28, None, None, None, None, None, stream) == 0
    binding.check_status(ws)


@pytest.mark.parametrize("E,k", [(1024, 32), (1024, 1), (4, 4)])
def test_topk_extremes_match_oracle(E, k):
    from serve_invariant_moe_gb300 import binding
    T, H = 200, 128
    g = torch.Generator().manual_seed(E + k)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    wr = (torch.randn((E, H), generator=g) * 0.1).to(torch.bfloat16)
    ws = binding.new_workspace(binding.workspace_size(T, H, E, k))
    r = binding.moe_route_topk(x.cuda(), wr.cuda(), k, ws)
    binding.check_status(ws)
    L = r["logits"].cpu().numpy()
    ref = omoe.router_logits(f64(x), f64(wr))
    bound = dot_bound(f64(x), f64(wr), H)
    assert (np.abs(L - ref) <= bound).all()
    check_topk(r["topk_idx"].cpu().numpy(), L, ref, k, bound)
    g_ref = omoe.topk_gates(L.astype(np.float64), r["topk_idx"].cpu().numpy())
    assert np.allclose(r["topk_w"].cpu().numpy(), g_ref, rtol=4e-6, atol=1e-7)
    counts, offsets, row_token, slot_row = omoe.dispatch_plan(r["topk_idx"].cpu().numpy(), E)
    assert np.array_equal(r["plan"].cpu().numpy()[:E], counts)


def test_nan_token_routes_by_index_and_stays_local():
    """A NaN activation makes that token's logits NaN: NaN ranks below every number,
    so it goes to experts 0..k-1 (index order) with NaN gates; other tokens are untouched."""
    from serve_invariant_moe_gb300 import api
    cfg = dataclasses.replace(synth.TINY, name="nan", T=40, E=8, k=2, dup_router_rows=False, seed=61)
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg)
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), cfg.k))
    clean = layer.prefill(x.cuda(), return_all=True)
    clean = {k: v.clone() for k, v in clean.items() if isinstance(v, torch.Tensor)}
    xn = x.clone()
    xn[7, 3] = float("nan")
    res = layer.prefill(xn.cuda(), return_all=True)
    torch.cuda.synchronize()
    assert torch.isnan(res["logits"][7]).all()
    assert res["topk_idx"][7].tolist() == [0, 1] and torch.isnan(res["topk_w"][7]).all()
    others = [t for t in range(cfg.T) if t != 7]
    assert torch.equal(res["out"][others], clean["out"][others])
    assert torch.equal(res["topk_idx"][others], clean["topk_idx"][others])


def test_k1_and_all_tokens_on_one_expert():
    from serve_invariant_moe_gb300 import api
    cfg = dataclasses.replace(synth.TINY, name="k1", T=517, H=256, E=4, k=1, F=128, dup_router_rows=False, seed=62)
    x, wr = synth.moe_activations(cfg)
    x, wr = x.clone(), wr.clone()
    x[:, 0] = 8.0                     # a shared input feature ...
    wr[:, 0] = 0.0
    wr[2, 0] = 4.0                    # ... that only expert 2 reads: it wins every token (517-row segment)
    w13, w2 = synth.expert_weights(cfg)
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), 1))
    res = layer.prefill(x.cuda(), return_all=True)
    torch.cuda.synchronize()
    counts = res["plan"][:cfg.E].cpu().numpy()
    assert counts.tolist() == [0, 0, cfg.T, 0]
    assert torch.all(res["topk_w"] == 1.0)
    ref = omoe.moe_forward(f64(x), f64(wr), f64(w13), f64(w2), 1, cfg.F)
    assert_moe_close(res["out"].cpu().numpy(), ref["out"])


def test_repeated_tokens_in_one_batch_get_identical_rows():
    from serve_invariant_moe_gb300 import api
    cfg = dataclasses.replace(synth.TINY, name="rep", T=64, H=256, E=8, k=3, F=256, dup_router_rows=False, seed=63)
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg)
    x = torch.cat([x[:8]] * 40)        # 320 tokens: 8 distinct, each 40 times, spread over tiles
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), cfg.k))
    out = layer.prefill(x.cuda())
    torch.cuda.synchronize()
    for r in range(1, 40):
        assert torch.equal(out[8 * r:8 * r + 8], out[:8])
