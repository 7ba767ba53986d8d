"""The launch-bound decode path: the one-block routing of small batches, the one-call layer
forward and launches that overlap the previous kernel's tail must all give the bits of the
multi-kernel prefill path ("位级一致：前沿训练的差异化关键", section "端到端零 KLD": serving
prefill and generation must agree token for token)."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe as omoe
from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _layer(cfg):
    from serve_invariant_moe_gb300 import api
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg)
    ws13, ws2 = synth.shared_expert_weights(cfg)
    c = lambda t: None if t is None else t.cuda()   # noqa: E731
    return x.cuda(), api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), cfg.k, c(ws13), c(ws2)))


CFGS = [
    # small-batch routing copies the rows itself (T*k*H*2 <= 512 KB) for the smaller chunks
    dataclasses.replace(synth.TINY, name="decode_small_rows", T=600, H=256, E=64, k=8, F=256, F_shared=128,
                        dup_router_rows=False, seed=51),
    # rows too large for the one-block copy: the grid-wide permute follows the one-block routing
    dataclasses.replace(synth.TINY, name="decode_wide_rows", T=300, H=2048, E=128, k=8, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=0.5, seed=52),
    # E = 1024, k = 16 (the largest shared-memory request of the one-block routing)
    dataclasses.replace(synth.TINY, name="decode_many_experts", T=260, H=128, E=1024, k=16, F=128,
                        dup_router_rows=False, seed=53),
]


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: c.name)
def test_small_batches_match_the_large_batch_path(cfg):
    x, layer = _layer(cfg)
    ref = layer.prefill(x, return_all=True)          # T > 256: the multi-kernel routing
    ref_idx = ref["topk_idx"].cpu()
    ref_w = ref["topk_w"].cpu()
    for chunk in (1, 7, 64, 256):
        for t0 in range(0, cfg.T, chunk * 3):        # a few chunks of each size
            t1 = min(cfg.T, t0 + chunk)
            got = layer.prefill(x[t0:t1], return_all=True)
            torch.cuda.synchronize()
            assert torch.equal(got["topk_idx"].cpu(), ref_idx[t0:t1]), (chunk, t0)
            assert torch.equal(got["topk_w"].cpu().view(torch.int32), ref_w[t0:t1].view(torch.int32)), (chunk, t0)
            assert torch.equal(got["out"].view(torch.int32), ref["out"][t0:t1].view(torch.int32)), (chunk, t0)
            # the plan of the one-block routing is the oracle's counting sort of its own indices
            T, E, k = t1 - t0, cfg.E, cfg.k
            counts, offsets, row_token, slot_row = omoe.dispatch_plan(got["topk_idx"].cpu().numpy(), E)
            plan = got["plan"].cpu().numpy()
            assert np.array_equal(plan[:E], counts) and np.array_equal(plan[E:2 * E + 1], offsets)
            assert np.array_equal(plan[2 * E + 1:2 * E + 1 + T * k], row_token)
            assert np.array_equal(plan[2 * E + 1 + T * k:2 * E + 1 + 2 * T * k], slot_row.ravel())
            xp = got["xp"][:T * k].cpu()
            assert torch.equal(xp.view(torch.int16), x[t0:t1].cpu()[torch.from_numpy(row_token)].view(torch.int16))


def test_decode_fast_path_and_overlapped_launches_change_no_bit():
    from serve_invariant_moe_gb300 import _lib, binding
    cfg = CFGS[0]
    x, layer = _layer(cfg)
    lib = _lib.lib()
    outs = []
    try:
        for pdl in (1, 0, 1):
            lib.invmoe_pdl_enable(pdl)
            a = layer.decode(x[:37]).clone()
            b = layer.prefill(x[:37])
            # the three separate calls
            w = layer.w
            ws = binding.new_workspace(binding.workspace_size(37, w.H, w.E, w.k, w.F, w.F_shared, 0))
            r = binding.moe_route_topk(x[:37], w.w_router, w.k, ws)
            f = binding.moe_grouped_ffn(r["xp"], r["plan"], w.w13, w.w2, 37, w.k, ws, x_shared=x[:37],
                                        ws13=w.ws13, ws2=w.ws2)
            c = binding.moe_combine(f["y"], r["topk_w"], r["plan"], 37, w.H, w.E, w.k, y_shared=f["y_shared"])
            torch.cuda.synchronize()
            binding.check_status(ws)
            outs += [a, b, c]
    finally:
        lib.invmoe_pdl_enable(1)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


def test_decode_rejects_a_bad_token_tensor():
    cfg = CFGS[0]
    x, layer = _layer(cfg)
    layer.decode(x[:4])
    with pytest.raises(ValueError):
        layer.decode(x[:4].float())
    with pytest.raises(ValueError):
        layer.decode(x[:4, :128].contiguous())
    with pytest.raises(ValueError):
        layer.decode(x[:4].cpu())


def test_shared_expert_on_the_side_stream_changes_no_bit():
    """moe_layer_forward runs the shared expert on the library's side stream beside the routing and
    the routed experts (invmoe_shared_overlap 1, and 2 for batches up to 1024 tokens) or after them
    on the caller's stream (0): the same kernels, so the same bits, and a workspace of the size
    invmoe_workspace_size gives keeps the routing scratch and the shared expert's h apart."""
    from serve_invariant_moe_gb300 import _lib
    cfg = CFGS[0]
    x, layer = _layer(cfg)
    lib = _lib.lib()
    try:
        for T in (1, 37, cfg.T):
            outs = []
            for mode in (0, 1, 2, 0):
                assert lib.invmoe_shared_overlap(mode) == 0
                r = layer.prefill(x[:T], return_all=True)
                torch.cuda.synchronize()
                outs.append((r["out"].clone(), r["y_shared"][:T].clone()))
            for o, ys in outs[1:]:
                assert torch.equal(o.view(torch.int32), outs[0][0].view(torch.int32)), T
                assert torch.equal(ys.view(torch.int32), outs[0][1].view(torch.int32)), T
            d = layer.decode(x[:T]).clone()
            assert torch.equal(d.view(torch.int32), outs[0][0].view(torch.int32)), T
    finally:
        lib.invmoe_shared_overlap(2)
    assert lib.invmoe_shared_overlap(3) != 0
