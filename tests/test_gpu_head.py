"""logprob/KL head on the GPU (through the C ABI) against the float64 CPU oracle."""
import math

import numpy as np
import pytest
import torch

from helpers import LOGP_ABS, dot_bound, f64
from oracle import head as ohead
from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _run(hidden, wv, target, rollout=None, beta=2.0):
    from serve_invariant_moe_gb300 import api
    r = api.head_logprob_kl(hidden.cuda(), wv.cuda(), target.cuda(),
                            None if rollout is None else rollout.cuda(), beta, write_logits=True)
    torch.cuda.synchronize()
    return r


@pytest.mark.parametrize("T,H,V", [(64, 256, 4096), (37, 192, 1000), (1, 128, 260), (300, 256, 8196)])
def test_head_matches_oracle(T, H, V):
    g = torch.Generator().manual_seed(T + V)
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16)
    wv = (torch.randn((V, H), generator=g) * 0.02).to(torch.bfloat16)
    target = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    ref = ohead.head_forward(f64(hidden), f64(wv), target.numpy())
    # rollout logprobs: the oracle's own logprob plus seeded noise
    noise = torch.randn(T, generator=g) * 0.5
    rollout = torch.from_numpy(ref["logp"]).float() + noise
    r = _run(hidden, wv, target, rollout)
    z = r["logits"].double().cpu().numpy()
    bound = dot_bound(f64(hidden), f64(wv), H)
    assert (np.abs(z - ref["logits"]) <= bound).all()
    logp = r["logp"].double().cpu().numpy()
    assert np.abs(logp - ref["logp"]).max() <= LOGP_ABS
    assert np.abs(r["lse"].double().cpu().numpy() - ref["lse"]).max() <= LOGP_ABS
    k3_ref = ohead.k3(ref["logp"], rollout.double().numpy())
    assert np.allclose(r["k3"].double().cpu().numpy(), k3_ref, rtol=1e-2, atol=1e-5)
    # the mask decision: taken in fp32 on both sides; the oracle's own d may
    # differ from the kernel's by the logprob tolerance, so only tokens whose d
    # is clear of the boundary by more than that are compared
    d_ref = ref["logp"] - rollout.double().numpy()
    clear = np.abs(np.abs(d_ref) - math.log(2.0)) > 2 * LOGP_ABS
    m_ref = ohead.icepop_mask(ref["logp"], rollout.double().numpy(), 2.0, np.float32)
    assert np.array_equal(r["mask"].cpu().numpy()[clear], m_ref[clear])
    assert 0 < r["mask"].sum().item() < T or T < 8


def test_head_uniform_logits_give_minus_log_v():
    T, H, V = 16, 128, 4096
    hidden = torch.zeros((T, H), dtype=torch.bfloat16)
    wv = torch.randn((V, H)).to(torch.bfloat16)
    target = torch.arange(T, dtype=torch.int32) * 7
    r = _run(hidden, wv, target)
    assert np.allclose(r["logp"].cpu().numpy(), -math.log(V), atol=1e-6)


def test_identical_logprobs_give_zero_k3_and_keep_all():
    T, H, V = 50, 256, 2048
    g = torch.Generator().manual_seed(3)
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16)
    wv = (torch.randn((V, H), generator=g) * 0.02).to(torch.bfloat16)
    target = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    r1 = _run(hidden, wv, target)
    r2 = _run(hidden, wv, target, r1["logp"].cpu())
    assert torch.equal(r2["logp"], r1["logp"])
    assert torch.all(r2["k3"] == 0) and torch.all(r2["mask"] == 1)


def test_logits_buffer_is_optional_and_changes_nothing():
    T, H, V = 77, 256, 3000
    g = torch.Generator().manual_seed(5)
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16).cuda()
    wv = (torch.randn((V, H), generator=g) * 0.02).to(torch.bfloat16).cuda()
    target = torch.randint(0, V, (T,), generator=g, dtype=torch.int32).cuda()
    from serve_invariant_moe_gb300 import api
    a = api.head_logprob_kl(hidden, wv, target)
    b = api.head_logprob_kl(hidden, wv, target, write_logits=True)
    torch.cuda.synchronize()
    assert a["logits"] is None
    assert torch.equal(a["logp"], b["logp"]) and torch.equal(a["lse"], b["lse"])
    # the target logit the epilogue captured is the stored logit
    zt = b["logits"].gather(1, target.long()[:, None])[:, 0]
    assert torch.equal(b["logp"], zt - b["lse"])


def test_target_out_of_range_gives_nan():
    T, H, V = 4, 128, 512
    hidden = torch.randn((T, H)).to(torch.bfloat16)
    wv = torch.randn((V, H)).to(torch.bfloat16)
    target = torch.tensor([0, V, -1, V - 1], dtype=torch.int32)
    r = _run(hidden, wv, target)
    lp = r["logp"].cpu()
    assert torch.isfinite(lp[[0, 3]]).all() and torch.isnan(lp[[1, 2]]).all()


@pytest.mark.slow
def test_full_size_head_sampled_tokens():
    from serve_invariant_moe_gb300 import api
    cfg = synth.GLM_HEAD
    hidden, wv, target, noise, noise_wide = synth.head_inputs(cfg, "cuda")
    # 64 rows: the first row and one seeded row of each 256-row chunk, across both 4096-row bands
    g = torch.Generator().manual_seed(9)
    sample = sorted({c * 256 for c in range(cfg.T // 256)}
                    | {c * 256 + int(torch.randint(1, 256, (1,), generator=g)) for c in range(cfg.T // 256)})
    assert len(sample) == 64 and sample[-1] >= 4096
    # oracle logits for the sampled tokens, vocabulary in chunks
    hs = f64(hidden[sample])
    z_ref = np.empty((len(sample), cfg.V))
    bound = np.empty((len(sample), cfg.V))
    for v0 in range(0, cfg.V, 16384):
        v1 = min(cfg.V, v0 + 16384)
        wchunk = f64(wv[v0:v1].cpu())
        z_ref[:, v0:v1] = ohead.vocab_logits(hs, wchunk)
        bound[:, v0:v1] = dot_bound(hs, wchunk, cfg.H)
    logp_ref, lse_ref = ohead.token_logprob(z_ref, target.numpy()[sample])
    # rollout: the oracle's logprob + N(0, 0.05) on the sampled tokens, -log V + noise elsewhere
    rollout = torch.full((cfg.T,), -math.log(cfg.V)) + noise * cfg.noise_std
    rollout[sample] = torch.from_numpy(logp_ref).float() + noise[sample] * cfg.noise_std
    r = api.head_logprob_kl(hidden.cuda(), wv, target.cuda(), rollout.cuda(), 2.0, write_logits=True)
    torch.cuda.synchronize()
    z = r["logits"][sample].double().cpu().numpy()
    assert (np.abs(z - z_ref) <= bound).all()
    assert np.abs(r["logp"][sample].double().cpu().numpy() - logp_ref).max() <= LOGP_ABS
    assert np.abs(r["lse"][sample].double().cpu().numpy() - lse_ref).max() <= LOGP_ABS
    k3_ref = ohead.k3(logp_ref, rollout[sample].double().numpy())
    assert np.allclose(r["k3"][sample].double().cpu().numpy(), k3_ref, rtol=2e-2, atol=1e-5)
    assert torch.isfinite(r["logp"]).all() and (r["k3"] >= 0).all()
    # N(0, 0.05) perturbation keeps every sampled token (|d| << ln 2)
    assert torch.all(r["mask"][sample] == 1)


def test_head_very_large_vocab():
    """V = 204800 (800 LSE chunks, 25 per merge lane) with a small hidden size."""
    T, H, V = 3, 64, 204800
    g = torch.Generator().manual_seed(21)
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16)
    wv = (torch.randn((V, H), generator=g) * 0.1).to(torch.bfloat16)
    target = torch.tensor([0, 123457, V - 1], dtype=torch.int32)
    ref = ohead.head_forward(f64(hidden), f64(wv), target.numpy())
    r = _run(hidden, wv, target)
    assert np.abs(r["logp"].double().cpu().numpy() - ref["logp"]).max() <= LOGP_ABS
    assert np.abs(r["lse"].double().cpu().numpy() - ref["lse"]).max() <= LOGP_ABS
