"""MoE layer backward on the GPU (through the C ABI) against the float64 oracle,
plus its determinism and batch-invariance properties ("位级一致：前沿训练的差异化关键",
section "端到端零 KLD": the trainer follows the same bit-exact standard)."""
import dataclasses

import numpy as np
import pytest
import torch

from helpers import f64, rel_err
from oracle import moe as omoe
from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu

# normwise relative error per row (bf16 operands dy, [dg | du] and the router
# gradient are rounded on both sides; elements whose fp32 and fp64 values sit
# on opposite sides of a rounding boundary differ by one bf16 ulp)
GRAD_MAX_REL = 1e-2
GRAD_MEAN_REL = 1e-3

SMALL = dataclasses.replace(synth.GLM_MOE, name="bwd_small", T=200, H=256, E=8, k=2, F=256, F_shared=128, seed=41)
RAGGED = dataclasses.replace(synth.GLM_MOE, name="bwd_ragged", T=77, H=192, E=16, k=3, F=128, F_shared=0, seed=42)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _setup(cfg, empty_expert=None):
    from serve_invariant_moe_gb300 import api
    x, wr = synth.moe_activations(cfg)
    if empty_expert is not None:
        x = x.clone(); wr = wr.clone()
        x[:, 0] = 4.0
        wr[empty_expert, 0] = -8.0             # that expert's logit is about -32 for every token
    w13, w2 = synth.expert_weights(cfg, "cpu")
    ws13, ws2 = synth.shared_expert_weights(cfg, "cpu")
    dev = "cuda"
    layer = api.MoELayer(api.MoEWeights(wr.to(dev), w13.to(dev), w2.to(dev), cfg.k,
                                        None if ws13 is None else ws13.to(dev), None if ws2 is None else ws2.to(dev)))
    g = torch.Generator().manual_seed(cfg.seed + 1000)
    dout = torch.randn((x.shape[0], cfg.H), generator=g)
    return x, wr, w13, w2, ws13, ws2, dout, layer


def _gpu_backward(layer, x, dout):
    fwd = layer.prefill(x.cuda(), return_all=True)
    b = layer.backward(x.cuda(), fwd, dout.cuda())
    torch.cuda.synchronize()
    return fwd, b


def _close(got, ref, what):
    got = np.asarray(got, np.float64).reshape(-1, np.asarray(ref).shape[-1])
    ref = np.asarray(ref, np.float64).reshape(got.shape)
    zero = np.abs(ref).max(axis=1) == 0
    assert np.all(got[zero] == 0), f"{what}: rows that must be zero are not"
    r = rel_err(got[~zero], ref[~zero])
    if r.size == 0:
        return
    assert r.max() <= GRAD_MAX_REL and r.mean() <= GRAD_MEAN_REL, (
        f"{what}: max rel {r.max():.3e} (<= {GRAD_MAX_REL}), mean rel {r.mean():.3e} (<= {GRAD_MEAN_REL})")


def _check_against_oracle(cfg, empty_expert=None):
    x, wr, w13, w2, ws13, ws2, dout, layer = _setup(cfg, empty_expert)
    fwd, b = _gpu_backward(layer, x, dout)
    Fs = cfg.F_shared
    ref = omoe.moe_backward(f64(x), f64(wr), f64(w13), f64(w2), cfg.k, cfg.F, dout.double().numpy(),
                            None if ws13 is None else f64(ws13), None if ws2 is None else f64(ws2), Fs)
    # the routing the gradients flow through is the same on both sides
    assert np.array_equal(fwd["topk_idx"].cpu().numpy(), ref["fwd"]["idx"])
    T, k = x.shape[0], cfg.k
    slot_row = fwd["plan"].cpu().numpy()[2 * cfg.E + 1 + T * k:].reshape(T, k)
    # dgate = <dout, y>: y carries the forward's bf16 rounding of h, so it is held to the same
    # per-token normwise bound as the layer output
    _close(b["dgate"].double().cpu().numpy(), ref["dgate"], "dgate")
    _close(b["dy"].double().cpu().numpy()[slot_row.ravel()], ref["dy"].reshape(T * k, -1), "dy")
    _close(b["dxp"].double().cpu().numpy()[slot_row.ravel()], ref["dxp"].reshape(T * k, -1), "dxp")
    _close(b["dx"].cpu().numpy(), ref["dx"], "dx")
    _close(b["dw_router"].cpu().numpy(), ref["dw_router"], "dw_router")
    _close(b["dw13"].cpu().numpy(), ref["dw13"], "dw13")
    _close(b["dw2"].cpu().numpy(), ref["dw2"], "dw2")
    if Fs:
        _close(b["dws13"].cpu().numpy(), ref["dws13"], "dws13")
        _close(b["dws2"].cpu().numpy(), ref["dws2"], "dws2")
    return fwd, b, ref


def test_moe_backward_matches_oracle_with_shared_expert():
    _check_against_oracle(SMALL)


def test_moe_backward_ragged_with_an_empty_expert():
    fwd, b, ref = _check_against_oracle(RAGGED, empty_expert=5)
    counts = fwd["plan"][:RAGGED.E].cpu()
    assert counts[5] == 0 and (counts % 64 != 0).any()      # an empty group and ragged K tails
    assert torch.all(b["dw13"][5] == 0) and torch.all(b["dw2"][5] == 0)


def test_moe_backward_intermediates_in_workspace():
    """[dg | du] and the recomputed h (read from the documented workspace layout) against the oracle."""
    from serve_invariant_moe_gb300 import binding
    cfg = SMALL
    x, wr, w13, w2, ws13, ws2, dout, layer = _setup(cfg)
    fwd, b = _gpu_backward(layer, x, dout)
    T, k, F, E = x.shape[0], cfg.k, cfg.F, cfg.E
    S = T * k
    ws = b["workspace"]

    def part(off, n, dtype):
        return ws[256 + off:256 + off + n * torch.tensor([], dtype=dtype).element_size()].view(dtype)

    al = lambda v: (v + 255) // 256 * 256
    off_dgu = al(S * F * 4)
    off_h = off_dgu + al(S * 2 * F * 2)
    dgu = part(off_dgu, S * 2 * F, torch.bfloat16).view(S, 2 * F)
    h = part(off_h, S * F, torch.bfloat16).view(S, F)
    # the recomputed h is bit-identical to the forward's h
    assert torch.equal(h.view(torch.int16), fwd["h"][:S].view(torch.int16))
    ref = omoe.moe_backward(f64(x), f64(wr), f64(w13), f64(w2), k, F, dout.double().numpy(), f64(ws13), f64(ws2),
                            cfg.F_shared)
    slot_row = fwd["plan"].cpu().numpy()[2 * E + 1 + S:].reshape(T, k)
    _close(dgu.double().cpu().numpy()[slot_row.ravel()], ref["dgu"].reshape(S, -1), "dgu")


def test_moe_backward_is_deterministic():
    x, wr, w13, w2, ws13, ws2, dout, layer = _setup(SMALL)
    _, a = _gpu_backward(layer, x, dout)
    for _ in range(3):
        _, b = _gpu_backward(layer, x, dout)
        for k in ("dx", "dw_router", "dw13", "dw2", "dws13", "dws2", "dgate", "dxp"):
            assert torch.equal(a[k], b[k]), k


def test_moe_backward_token_rows_are_batch_invariant():
    """The probe's dx, dgate and per-slot gradient rows are bit-identical whatever else is in the batch."""
    cfg = SMALL
    _, _, _, _, _, _, _, layer = _setup(cfg)
    g = torch.Generator().manual_seed(77)
    probe = synth.to_bf16(torch.randn((32, cfg.H), generator=g))
    pd = torch.randn((32, cfg.H), generator=g)
    ref_fwd, ref = _gpu_backward(layer, probe, pd)
    ref_dx, ref_dg = ref["dx"].clone(), ref["dgate"].clone()
    for n in (1, 7, 100, 500):
        other = synth.to_bf16(torch.randn((n, cfg.H), generator=g))
        od = torch.randn((n, cfg.H), generator=g)
        off = n // 2
        xb = torch.cat([other[:off], probe, other[off:]])
        db = torch.cat([od[:off], pd, od[off:]])
        _, b = _gpu_backward(layer, xb, db)
        assert torch.equal(b["dx"][off:off + 32], ref_dx), n
        assert torch.equal(b["dgate"][off:off + 32], ref_dg), n


@pytest.mark.slow
def test_glm_scale_moe_backward_sampled():
    """T = 8192, H = 6144, E = 256, k = 8, F = 2048 + shared: sampled dx rows against the oracle (dx of a
    token depends on that token only); sampled weight-gradient rows against a float64 sum over the
    expert's rows of the kernel's own operands (a property of the K-grouped reduction at any size);
    repeat-call bit equality."""
    from serve_invariant_moe_gb300 import api, binding
    cfg = synth.GLM_MOE
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    ws13, ws2 = synth.shared_expert_weights(cfg, "cuda")
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13, w2, cfg.k, ws13, ws2))
    g = torch.Generator().manual_seed(5)
    dout = torch.randn((cfg.T, cfg.H), generator=g)
    fwd, b = _gpu_backward(layer, x, dout)
    binding.check_status(b["workspace"])
    sample = [0, 1, 4095, 8191]
    expert = lambda e: (f64(w13[e].cpu()), f64(w2[e].cpu()))
    ref = omoe.moe_backward(f64(x[sample]), f64(wr), None, None, cfg.k, cfg.F, dout[sample].double().numpy(),
                            f64(ws13.cpu()), f64(ws2.cpu()), cfg.F_shared, expert_weights=expert)
    assert np.array_equal(fwd["topk_idx"][sample].cpu().numpy(), ref["fwd"]["idx"])
    _close(b["dx"][sample].cpu().numpy(), ref["dx"], "dx")
    _close(b["dgate"][sample].cpu().numpy(), ref["dgate"], "dgate")
    # weight-gradient rows of two busy experts: sum over the expert's rows of the kernel's own operands
    S = cfg.T * cfg.k
    counts = fwd["plan"][:cfg.E].cpu().numpy()
    offsets = fwd["plan"][cfg.E:2 * cfg.E + 1].cpu().numpy()
    ws = b["workspace"]
    al = lambda v: (v + 255) // 256 * 256
    off_dgu = al(S * cfg.F * 4)
    off_h = off_dgu + al(S * 2 * cfg.F * 2)
    dgu = ws[256 + off_dgu:256 + off_dgu + S * 2 * cfg.F * 2].view(torch.bfloat16).view(S, 2 * cfg.F)
    h = ws[256 + off_h:256 + off_h + S * cfg.F * 2].view(torch.bfloat16).view(S, cfg.F)
    for e in (int(np.argmax(counts)), int(np.argmin(counts))):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        rows = [0, 777, cfg.H - 1]
        dy_e = f64(b["dy"][r0:r1].cpu())
        ref_dw2 = dy_e[:, rows].T @ f64(h[r0:r1].cpu())
        _close(b["dw2"][e][rows].cpu().numpy(), ref_dw2, "dw2 rows")
        rows13 = [0, cfg.F + 5, 2 * cfg.F - 1]
        ref_dw13 = f64(dgu[r0:r1].cpu())[:, rows13].T @ f64(fwd["xp"][r0:r1].cpu())
        _close(b["dw13"][e][rows13].cpu().numpy(), ref_dw13, "dw13 rows")
    b2 = layer.backward(x.cuda(), fwd, dout.cuda())
    torch.cuda.synchronize()
    for k in ("dx", "dw_router", "dw13", "dw2", "dws13", "dws2"):
        assert torch.equal(b[k], b2[k]), k


def test_moe_backward_single_expert_k1_is_the_plain_mlp_backward():
    """E = 1, k = 1: the gate is exactly 1 and the router gets no gradient (a softmax over one logit),
    so the layer backward is the SwiGLU MLP backward of the oracle."""
    from serve_invariant_moe_gb300 import api
    cfg = dataclasses.replace(synth.GLM_MOE, name="bwd_k1", T=96, H=128, E=8, k=1, F=128, F_shared=0, seed=43)
    x, _ = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, "cpu")
    wr = torch.zeros((8, cfg.H), dtype=torch.bfloat16)
    wr[3, :] = 1.0                                            # logit of expert 3 = sum(x), far from the others
    x = (x.abs() + 0.25).to(torch.bfloat16)                  # positive rows: expert 3 wins every token
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), 1))
    g = torch.Generator().manual_seed(4)
    dout = torch.randn((cfg.T, cfg.H), generator=g)
    fwd, b = _gpu_backward(layer, x, dout)
    assert torch.all(fwd["topk_idx"] == 3) and torch.all(fwd["topk_w"] == 1.0)
    ref = omoe.swiglu_backward(f64(x), f64(w13[3]), f64(w2[3]), cfg.F, omoe.round_to_bf16(dout.double().numpy()))
    assert torch.all(b["dw_router"] == 0) and torch.all(b["dgate"].abs() >= 0)
    _close(b["dx"].cpu().numpy(), ref["dx"], "dx")
    _close(b["dw13"][3].cpu().numpy(), ref["dw13"], "dw13")
    _close(b["dw2"][3].cpu().numpy(), ref["dw2"], "dw2")
    others = [e for e in range(8) if e != 3]
    assert torch.all(b["dw13"][others] == 0) and torch.all(b["dw2"][others] == 0)


def test_moe_backward_through_replayed_routing():
    """Routing replayed from recorded indices: the backward follows the replayed experts and gates
    (oracle: the same backward with those indices given to its forward)."""
    from serve_invariant_moe_gb300 import binding
    cfg = SMALL
    x, wr, w13, w2, ws13, ws2, dout, layer = _setup(cfg)
    g = torch.Generator().manual_seed(6)
    idx = torch.stack([torch.randperm(cfg.E, generator=g)[:cfg.k] for _ in range(x.shape[0])]).to(torch.int32)
    fwd = layer.prefill(x.cuda(), return_all=True, replay_idx=idx.cuda())
    b = layer.backward(x.cuda(), fwd, dout.cuda())
    torch.cuda.synchronize()
    assert torch.equal(fwd["topk_idx"].cpu(), idx)
    ref = omoe.moe_backward(f64(x), f64(wr), f64(w13), f64(w2), cfg.k, cfg.F, dout.double().numpy(), f64(ws13),
                            f64(ws2), cfg.F_shared, replay_idx=idx.numpy())
    assert np.array_equal(ref["fwd"]["idx"], idx.numpy())
    _close(b["dgate"].double().cpu().numpy(), ref["dgate"], "dgate")
    _close(b["dx"].cpu().numpy(), ref["dx"], "dx")
    _close(b["dw_router"].cpu().numpy(), ref["dw_router"], "dw_router")
    _close(b["dw13"].cpu().numpy(), ref["dw13"], "dw13")
