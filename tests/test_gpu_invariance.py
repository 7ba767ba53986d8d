"""Batch invariance: a fixed 32-token probe request gets bit-identical outputs
whatever traffic shares its batch, through the prefill and the decode entry
points, and its logprobs agree bit for bit, so k3 between the two paths is
exactly 0 ("位级一致：前沿训练的差异化关键", section "端到端零 KLD": the engine
returns bit-identical logits whatever the batch size or concurrent load)."""
import dataclasses

import numpy as np
import pytest
import torch

from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu

SMALL = dataclasses.replace(synth.GLM_MOE, name="glm_like_small", H=512, E=32, k=8, F=256, F_shared=256, seed=31)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _layer(cfg, device_weights=True):
    from serve_invariant_moe_gb300 import api
    _, wr = synth.moe_activations(cfg, T=1)
    w13, w2 = synth.expert_weights(cfg, "cuda" if device_weights else "cpu")
    ws13, ws2 = synth.shared_expert_weights(cfg, "cuda" if device_weights else "cpu")
    return api.MoELayer(api.MoEWeights(wr.cuda(), w13.cuda(), w2.cuda(), cfg.k,
                                       None if ws13 is None else ws13.cuda(), None if ws2 is None else ws2.cuda()))


def _sweep(cfg, sizes, trials):
    layer = _layer(cfg)
    x0, off0, _ = synth.probe_and_batch(cfg, 0, 0)
    ref = layer.prefill(x0.cuda()).clone()
    n_runs = 0
    for n in sizes:
        for trial in range(trials):
            for skew in (False, True):
                x, off, lengths = synth.probe_and_batch(cfg, n, trial, skew=skew)
                out = layer.prefill(x.cuda())
                probe = out[off:off + 32]
                assert torch.equal(probe, ref), (
                    f"n_other={n} trial={trial} skew={skew}: {(probe != ref).sum().item()} values differ")
                n_runs += 1
    # decode path: the probe's tokens one per request, alongside other decode tokens
    for B in (1, 2, 7, 64):
        g = torch.Generator().manual_seed(B)
        others = synth.to_bf16(torch.randn((B - 1, cfg.H), generator=g))
        for i in range(32):
            pos = i % B
            xt = torch.cat([others[:pos], x0[i:i + 1], others[pos:]], 0)
            o = layer.decode(xt.cuda())
            assert torch.equal(o[pos], ref[i]), f"decode B={B} token {i}"
    return n_runs


def test_invariance_small_layer():
    assert _sweep(SMALL, [1, 2, 3, 7, 31, 32, 33, 127, 128, 129, 255, 257, 1000], 2) > 0


@pytest.mark.parametrize("name", ["qwen_moe_like", "qwen_moe_like_empty"])
def test_invariance_skewed_qwen_like_layer(name):
    """The Qwen-MoE-like layer with its own Zipf-skewed traffic around the probe (up to ~1500 tokens on
    one expert: several row chunks, M = 64 tail tiles, a handful of tokens on others, and in the second
    variant experts with none): the probe's bits never change, through prefill and through decode."""
    cfg = synth.CONFIGS[name]
    layer = _layer(cfg)
    x_all, _ = synth.moe_activations(cfg)                   # skewed traffic of the workload itself
    probe = synth.probe_tokens(cfg)
    ref = layer.prefill(probe.cuda()).clone()
    for n in (1, 7, 33, 129, 1000, 4000):
        off = n // 3
        x = torch.cat([x_all[:off], probe, x_all[off:n]])
        out = layer.prefill(x.cuda())
        assert torch.equal(out[off:off + 32], ref), n
    for B in (1, 5, 64):
        for i in range(0, 32, 7):
            xt = torch.cat([x_all[:B - 1], probe[i:i + 1]])
            o = layer.decode(xt.cuda())
            assert torch.equal(o[B - 1], ref[i]), (B, i)


GLM_SIZES = [1, 2, 3, 7, 31, 32, 33, 127, 128, 129, 255, 256, 257, 511, 1000, 2047, 4096]


@pytest.mark.slow
def test_invariance_glm_scale_layer():
    """The glm-scale layer: 17 batch sizes x 2 trials x (random, skewed) other traffic = 68
    batches through prefill, plus the probe through decode at several batch sizes."""
    assert _sweep(synth.GLM_MOE, GLM_SIZES, 2) == len(GLM_SIZES) * 4


def test_head_logprob_invariant_and_k3_zero():
    from serve_invariant_moe_gb300 import api
    H, V = 512, 8192
    g = torch.Generator().manual_seed(9)
    wv = (torch.randn((V, H), generator=g) * 0.02).to(torch.bfloat16).cuda()
    probe = torch.randn((32, H), generator=g).to(torch.bfloat16)
    tgt = torch.randint(0, V, (32,), generator=g, dtype=torch.int32)
    ref = api.head_logprob_kl(probe.cuda(), wv, tgt.cuda())["logp"].clone()
    for n in (1, 5, 100, 300):
        other = torch.randn((n, H), generator=g).to(torch.bfloat16)
        otgt = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
        off = n // 2
        x = torch.cat([other[:off], probe, other[off:]])
        t = torch.cat([otgt[:off], tgt, otgt[off:]])
        lp = api.head_logprob_kl(x.cuda(), wv, t.cuda())["logp"][off:off + 32]
        assert torch.equal(lp, ref), n
    # decode-style: one token at a time; then k3 against the batched path is exactly zero
    dec = torch.stack([api.head_logprob_kl(probe[i:i + 1].cuda(), wv, tgt[i:i + 1].cuda())["logp"][0]
                       for i in range(32)])
    assert torch.equal(dec, ref)
    r = api.head_logprob_kl(probe.cuda(), wv, tgt.cuda(), rollout_logp=dec)
    torch.cuda.synchronize()
    assert torch.all(r["k3"] == 0.0) and torch.all(r["mask"] == 1)
    assert r["k3"].double().mean().item() == 0.0
