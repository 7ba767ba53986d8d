"""Router replay (given expert choices) against the oracle and against the router's
own selection; invalid replayed indices are reported, never read out of bounds."""
import dataclasses

import numpy as np
import pytest
import torch

from helpers import assert_moe_close, f64
from oracle import moe as omoe
from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu

CFG = dataclasses.replace(synth.TINY, name="replay", T=300, H=256, E=16, k=4, F=256, dup_router_rows=False,
                          F_shared=128, seed=51)


@pytest.fixture(scope="module")
def layer():
    from serve_invariant_moe_gb300 import api, build
    build.build()
    x, wr = synth.moe_activations(CFG)
    w13, w2 = synth.expert_weights(CFG)
    ws13, ws2 = synth.shared_expert_weights(CFG)
    lay = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), CFG.k, ws13.cuda(), ws2.cuda()))
    return x, wr, w13, w2, ws13, ws2, lay


def test_replaying_own_choice_is_bit_identical(layer):
    x, _, _, _, _, _, lay = layer
    a = lay.prefill(x.cuda(), return_all=True)
    a = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in a.items()}
    b = lay.prefill(x.cuda(), return_all=True, replay_idx=a["topk_idx"].clone())
    torch.cuda.synchronize()
    for key in ("logits", "topk_w", "plan", "out"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["xp"].view(torch.int16), b["xp"].view(torch.int16))


def test_replaying_other_choices_matches_oracle(layer):
    from serve_invariant_moe_gb300 import binding
    x, wr, w13, w2, ws13, ws2, lay = layer
    g = torch.Generator().manual_seed(3)
    idx = torch.stack([torch.randperm(CFG.E, generator=g)[:CFG.k] for _ in range(CFG.T)]).to(torch.int32)
    res = lay.prefill(x.cuda(), return_all=True, replay_idx=idx.cuda())
    torch.cuda.synchronize()
    binding.check_status(lay._ws)
    L = res["logits"].double().cpu().numpy()
    gates = res["topk_w"].cpu().numpy()
    assert np.allclose(gates, omoe.topk_gates(L, idx.numpy()), rtol=4e-6, atol=1e-7)
    counts, offsets, row_token, slot_row = omoe.dispatch_plan(idx.numpy(), CFG.E)
    plan = res["plan"].cpu().numpy()
    S = CFG.T * CFG.k
    assert np.array_equal(plan[:CFG.E], counts)
    assert np.array_equal(plan[2 * CFG.E + 1:2 * CFG.E + 1 + S], row_token)
    ref = omoe.moe_forward(f64(x), f64(wr), f64(w13), f64(w2), CFG.k, CFG.F, f64(ws13), f64(ws2), CFG.F_shared,
                           replay_idx=idx.numpy())
    assert_moe_close(res["out"].cpu().numpy(), ref["out"])


def test_invalid_replay_indices_are_reported(layer):
    from serve_invariant_moe_gb300 import binding
    from serve_invariant_moe_gb300._lib import InvmoeError
    x, wr, _, _, _, _, lay = layer
    g = torch.Generator().manual_seed(4)
    idx = torch.stack([torch.randperm(CFG.E, generator=g)[:CFG.k] for _ in range(CFG.T)]).to(torch.int32)
    idx[5, 1] = CFG.E + 3          # out of range
    idx[9, 2] = -1                 # negative
    idx[17, 3] = idx[17, 0]        # repeated
    ws = binding.new_workspace(binding.workspace_size(CFG.T, CFG.H, CFG.E, CFG.k), "cuda")
    r = binding.moe_route_replay(x.cuda(), wr.cuda(), idx.cuda(), ws)
    with pytest.raises(InvmoeError) as e:
        binding.check_status(ws)
    assert e.value.code == -1
    w = r["topk_w"].cpu()
    bad = [5, 9, 17]
    assert torch.isnan(w[bad]).all()
    good = [t for t in range(CFG.T) if t not in bad]
    L = r["logits"].double().cpu().numpy()
    assert np.allclose(w[good].numpy(), omoe.topk_gates(L[good], idx[good].numpy()), rtol=4e-6, atol=1e-7)
    plan = r["plan"].cpu().numpy()
    assert plan[:CFG.E].sum() == CFG.T * CFG.k            # every slot was dispatched somewhere valid
    binding.check_status(ws)                              # cleared
