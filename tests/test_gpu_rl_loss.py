"""IcePop-masked clipped policy loss and DIS weights on the GPU against the oracle."""
import math

import numpy as np
import pytest
import torch

from oracle import head as ohead

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


@pytest.mark.parametrize("T", [1, 777, 8192])
def test_rl_token_loss_matches_oracle(T):
    from serve_invariant_moe_gb300 import binding
    g = torch.Generator().manual_seed(T)
    lt = -torch.rand(T, generator=g) * 8
    lr = lt + torch.randn(T, generator=g) * 0.5           # rollout: perturbed (some beyond ln 2)
    lo = lt + torch.randn(T, generator=g) * 0.2           # old train policy
    adv = torch.randn(T, generator=g)
    r = binding.rl_token_loss(lt.cuda(), lr.cuda(), adv.cuda(), logp_old=lo.cuda())
    torch.cuda.synchronize()
    lt64, lr64, lo64, a64 = (v.double().numpy() for v in (lt, lr, lo, adv))
    # decisions (mask, DIS window) are compared where the ratio is clear of the boundaries
    rho = np.exp(lt64 - lr64)
    ref_loss, ref_mean = ohead.ppo_icepop_loss(lt, lo, lr, adv, 2.0, 0.2, 0.28, np.float32)
    m_ref = ohead.icepop_mask(lt, lr, 2.0, np.float32)
    clear_m = (np.abs(rho - 0.5) > 1e-5) & (np.abs(rho - 2.0) > 1e-5)
    assert np.array_equal(r["icepop_mask"].cpu().numpy()[clear_m], m_ref[clear_m])
    loss = r["loss"].double().cpu().numpy()
    assert np.allclose(loss[clear_m], ref_loss[clear_m], rtol=1e-5, atol=1e-6)
    dis = r["dis_weight"].double().cpu().numpy()
    ref_dis = ohead.dis_weight(lt64, lr64, 0.2, 0.28)
    clear_d = (np.abs(rho - 0.8) > 1e-5) & (np.abs(rho - 1.28) > 1e-5)
    assert np.allclose(dis[clear_d], ref_dis[clear_d], rtol=1e-5, atol=0)
    assert abs(r["loss_mean"].item() - loss.mean()) <= 1e-5 * (1 + abs(loss.mean()))
    assert abs(r["loss_mean"].item() - ref_mean) <= 1e-4 * (1 + abs(ref_mean)) or not clear_m.all()


def test_rl_loss_identical_policies_and_determinism():
    from serve_invariant_moe_gb300 import binding
    T = 5000
    lt = (-torch.rand(T) * 5).cuda()
    adv = torch.randn(T).cuda()
    a = binding.rl_token_loss(lt, lt.clone(), adv)          # rollout == train, old == rollout
    b = binding.rl_token_loss(lt, lt.clone(), adv)
    torch.cuda.synchronize()
    assert torch.all(a["icepop_mask"] == 1) and torch.equal(a["loss"], -adv)
    assert torch.equal(a["dis_weight"], torch.ones_like(adv))
    assert torch.equal(a["loss_mean"], b["loss_mean"])      # fixed-order mean: same bits every run
    assert math.isclose(a["loss_mean"].item(), (-adv).double().mean().item(), rel_tol=1e-5, abs_tol=1e-7)
