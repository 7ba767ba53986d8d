"""Pins for oracle.head: log-sum-exp, token logprob, k3 and the IcePop mask."""
import json
import math
import os

import numpy as np
import scipy.special
import scipy.stats
import torch

from oracle import head

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_lse_uniform_is_log_v():
    for V in (4096, 151552):
        z = np.full((2, V), 3.5)
        lse = head.logsumexp_rows(z)
        assert np.allclose(lse, 3.5 + math.log(V), rtol=0, atol=1e-12)
        logp, _ = head.token_logprob(z, np.array([0, V - 1]))
        assert np.allclose(logp, -math.log(V), rtol=0, atol=1e-12)
    # the two values the workloads use
    assert abs(-math.log(151552) - (-11.928684)) < 1e-6
    assert abs(-math.log(4096) - (-8.317766)) < 1e-6


def test_lse_matches_scipy_and_is_shift_invariant():
    rng = np.random.default_rng(0)
    z = rng.standard_normal((7, 3000)) * 4
    lse = head.logsumexp_rows(z)
    assert np.allclose(lse, scipy.special.logsumexp(z, axis=1), rtol=1e-14, atol=1e-12)
    assert np.allclose(head.logsumexp_rows(z + 123.0), lse + 123.0, rtol=0, atol=1e-10)


def test_logprob_known_values_and_target_index():
    z = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))
    for t in range(4):
        logp, lse = head.token_logprob(z, np.array([t]))
        assert abs(lse[0] - math.log(10.0)) < 1e-15
        assert abs(logp[0] - math.log((t + 1) / 10.0)) < 1e-15
    # probabilities over all targets sum to one
    rng = np.random.default_rng(1)
    z = rng.standard_normal((1, 50))
    total = sum(math.exp(head.token_logprob(z, np.array([v]))[0][0]) for v in range(50))
    assert abs(total - 1.0) < 1e-13
    # one dominant logit
    z = np.zeros((1, 1000)); z[0, 17] = 60.0
    assert abs(head.token_logprob(z, np.array([17]))[0][0]) < 1e-20


def test_vocab_logits_rows_and_columns():
    rng = np.random.default_rng(2)
    h = rng.standard_normal((3, 5))
    w = rng.standard_normal((11, 5))
    z = head.vocab_logits(h, w)
    assert z.shape == (3, 11)
    assert abs(z[2, 9] - float(np.dot(h[2], w[9]))) < 1e-13


def test_k3_zero_nonnegative_and_direction():
    lp = np.log(np.array([0.1, 0.2, 0.7]))
    assert np.array_equal(head.k3(lp, lp), np.zeros(3))          # bit-exact 0
    rng = np.random.default_rng(3)
    d = rng.standard_normal(10000) * 3
    assert np.all(head.k3(d, np.zeros_like(d)) >= 0)
    # E_{y~q}[k3(log p(y) - log q(y))] = KL(q || p) for the rollout distribution q
    for _ in range(5):
        p = rng.dirichlet(np.ones(40))
        q = rng.dirichlet(np.ones(40))
        est = float(np.sum(q * head.k3(np.log(p), np.log(q))))
        assert abs(est - scipy.stats.entropy(q, p)) < 1e-12
    # small-d expansion: k3 = d^2/2 + d^3/6 + O(d^4)
    d = np.array([1e-3, -2e-3])
    assert np.allclose(head.k3(d, 0 * d), d ** 2 / 2 + d ** 3 / 6, rtol=1e-3)


def test_icepop_mask_golden_interval():
    g = json.load(open(os.path.join(GOLDEN, "icepop_beta2.json")))
    beta = g["beta"]
    for dtype in (np.float64, np.float32):
        lo, hi = dtype(g["keep_low"]), dtype(g["keep_high"])
        rhos = np.array([lo, hi, np.nextafter(lo, dtype(0)), np.nextafter(hi, dtype(10)),
                         dtype(1.0), dtype(0.25), dtype(4.0)], dtype)
        want = np.array([1, 1, 0, 0, 1, 0, 0], np.uint8)
        # feed the ratio through d = log(rho): build logp pairs whose float
        # difference reproduces rho exactly where possible, and check the
        # comparison itself on the ratios
        keep = ((lo <= rhos) & (rhos <= hi)).astype(np.uint8)
        assert np.array_equal(keep, want)
        d = np.log(rhos.astype(np.float64)).astype(dtype)
        m = head.icepop_mask(d, np.zeros_like(d), beta, dtype)
        # exp(log(rho)) may land one ulp off rho; only the clear cases are pinned
        assert np.array_equal(m[[4, 5, 6]], want[[4, 5, 6]])
    # d = 0 (identical paths) always kept; |d| well past ln 2 always dropped
    assert head.icepop_mask(np.zeros(3), np.zeros(3))[0] == 1
    assert head.icepop_mask(np.array([0.7, -0.7]), np.zeros(2)).tolist() == [0, 0]
    assert head.icepop_mask(np.array([0.69, -0.69]), np.zeros(2)).tolist() == [1, 1]


def test_k3_golden_threshold_consistency():
    g = json.load(open(os.path.join(GOLDEN, "k3_threshold.json")))
    assert round(g["bad_path_k3"] / g["equivalence_threshold"], -2) == g["ratio_to_threshold_approx"]
    lp = np.array([-1.0, -2.0])
    assert head.k3(lp, lp).mean() == g["aligned_k3"] < g["equivalence_threshold"]


def test_ppo_icepop_loss_hand_cases():
    g = json.load(open(os.path.join(GOLDEN, "icepop_beta2.json")))
    el, eh = g["ppo_clip_eps_low"], g["ppo_clip_eps_high"]
    # identical policies: r = 1, rho = 1 -> loss = -A
    lt = np.array([-1.0, -2.0, -3.0])
    loss, mean = head.ppo_icepop_loss(lt, lt, lt, np.array([1.0, -0.5, 2.0]), 2.0, el, eh)
    assert np.array_equal(loss, np.array([-1.0, 0.5, -2.0])) and abs(mean - (-2.5 / 3)) < 1e-15
    # positive advantage: the ratio is capped at 1 + eps_h; negative: floored at 1 - eps_l
    lo = np.zeros(4)
    lt = np.log(np.array([1.5, 1.5, 0.5, 0.5]))
    A = np.array([1.0, -1.0, 1.0, -1.0])
    loss, _ = head.ppo_icepop_loss(lt, lo, lt, A, 2.0, el, eh)      # rollout == train: mask 1
    assert np.allclose(loss, [-(1 + eh), 1.5, -0.5, 1 - el], rtol=0, atol=1e-15)
    # the IcePop mask removes a token whose train/infer ratio is outside [1/2, 2]
    loss, _ = head.ppo_icepop_loss(np.zeros(2), np.zeros(2), np.log([3.0, 1.9]), np.ones(2), 2.0, el, eh)
    assert loss[0] == 0.0 and loss[1] == -1.0


def test_dis_weight_window():
    g = json.load(open(os.path.join(GOLDEN, "icepop_beta2.json")))
    el, eh = g["ppo_clip_eps_low"], g["ppo_clip_eps_high"]
    r = np.array([0.79, 0.8, 0.81, 1.0, 1.27, 1.28, 1.3])
    w = head.dis_weight(np.log(r), np.zeros_like(r), el, eh)
    # open interval (0.8, 1.28); exp(log(r)) may land an ulp away from r at the two ends
    assert w[0] == 0 and w[6] == 0 and np.allclose(w[[2, 3, 4]], r[[2, 3, 4]], rtol=1e-15)
    assert head.dis_weight(np.log([0.8 - 1e-9, 1.28 + 1e-9]), np.zeros(2), el, eh).tolist() == [0.0, 0.0]


# ---------------------------------------------------------------- backward

def _f_logp(hs, wv, target, g):
    """sum_t g_t * logp_t as a plain function of (hidden, vocab weights)."""
    logp, _ = head.token_logprob(head.vocab_logits(hs, wv), target)
    return float(np.dot(g, logp))


def test_dlogits_central_differences_and_row_sums():
    rng = np.random.default_rng(20)
    z = rng.standard_normal((4, 9)) * 2
    tgt = np.array([0, 8, 3, 3])
    g = np.array([1.0, -0.7, 0.0, 2.5])
    dz = head.dlogits(z, tgt, g)
    eps = 1e-5
    for t in range(4):
        for v in range(9):
            zp, zm = z.copy(), z.copy()
            zp[t, v] += eps; zm[t, v] -= eps
            fd = (np.dot(g, head.token_logprob(zp, tgt)[0]) - np.dot(g, head.token_logprob(zm, tgt)[0])) / (2 * eps)
            assert abs(fd - dz[t, v]) < 1e-9
    assert np.allclose(dz.sum(1), 0.0, atol=1e-15)          # softmax and one-hot both sum to one
    assert np.array_equal(dz[2], np.zeros(9))                # g = 0: the token contributes nothing
    assert dz[0, 0] > 0 and np.all(dz[0, 1:] < 0)            # g > 0 raises the target, lowers the rest


def test_dlogits_matches_torch_autograd():
    rng = np.random.default_rng(21)
    z = torch.from_numpy(rng.standard_normal((6, 40)) * 3).requires_grad_(True)
    tgt = torch.from_numpy(rng.integers(0, 40, 6))
    g = torch.from_numpy(rng.standard_normal(6))
    (torch.log_softmax(z, 1).gather(1, tgt[:, None])[:, 0] * g).sum().backward()
    assert np.allclose(head.dlogits(z.detach().numpy(), tgt.numpy(), g.numpy()), z.grad.numpy(),
                       rtol=1e-13, atol=1e-15)


def test_head_backward_central_differences():
    # every element of both gradients against a central difference of sum_t g_t logp_t;
    # a transposed operand, a dropped one-hot or a sign error fails here
    rng = np.random.default_rng(22)
    T, H, V = 3, 5, 7
    hs = rng.standard_normal((T, H))
    wv = rng.standard_normal((V, H)) * 0.5
    tgt = np.array([6, 0, 2])
    g = np.array([0.5, -1.25, 2.0])
    out = head.head_backward(hs, wv, tgt, g, round_dz=False)
    assert out["d_hidden"].shape == (T, H) and out["d_wvocab"].shape == (V, H)
    eps = 1e-6
    for name, arr, grad in (("hidden", hs, out["d_hidden"]), ("wvocab", wv, out["d_wvocab"])):
        for i in np.ndindex(arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[i] += eps; am[i] -= eps
            if name == "hidden":
                fd = (_f_logp(ap, wv, tgt, g) - _f_logp(am, wv, tgt, g)) / (2 * eps)
            else:
                fd = (_f_logp(hs, ap, tgt, g) - _f_logp(hs, am, tgt, g)) / (2 * eps)
            assert abs(fd - grad[i]) < 1e-7 * max(1.0, abs(fd)), (name, i, fd, grad[i])


def test_head_backward_bf16_rounding_of_dz():
    rng = np.random.default_rng(23)
    hs = rng.standard_normal((8, 16)); wv = rng.standard_normal((50, 16)) * 0.3
    tgt = rng.integers(0, 50, 8); g = rng.standard_normal(8)
    a = head.head_backward(hs, wv, tgt, g, round_dz=False)
    b = head.head_backward(hs, wv, tgt, g)
    # dz is rounded to bf16 (8 significant bits): relative change at most 2^-8 per element
    assert np.all(np.abs(b["dz"] - a["dz"]) <= 2.0 ** -8 * np.abs(a["dz"]))
    from oracle.numerics import round_to_bf16
    assert np.array_equal(round_to_bf16(b["dz"]), b["dz"])
    assert np.allclose(b["d_hidden"], b["dz"] @ wv, rtol=1e-14) and np.allclose(b["d_wvocab"], b["dz"].T @ hs, rtol=1e-14)


def test_ppo_icepop_grad_hand_cases():
    g = json.load(open(os.path.join(GOLDEN, "icepop_beta2.json")))
    el, eh = g["ppo_clip_eps_low"], g["ppo_clip_eps_high"]
    lo = np.zeros(6)
    r = np.array([1.0, 1.5, 0.5, 0.5, 1.5, 1.0])
    A = np.array([1.0, 1.0, 1.0, -1.0, -1.0, 0.0])
    lt = np.log(r)
    gr = head.ppo_icepop_grad(lt, lo, lt, A, 2.0, el, eh)           # mask 1 everywhere
    # inside the window: -r A / T; A > 0 above the window and A < 0 below it are clipped: 0;
    # A > 0 below and A < 0 above stay unclipped
    want = np.array([-1.0, 0.0, -0.5, 0.0, 1.5, 0.0]) / 6
    assert np.allclose(gr, want, rtol=1e-15, atol=0)
    # a token the IcePop mask drops gives no gradient
    gm = head.ppo_icepop_grad(np.zeros(2), np.zeros(2), np.log([3.0, 1.0]), np.ones(2), 2.0, el, eh)
    assert gm[0] == 0.0 and gm[1] == -0.5


def test_ppo_icepop_grad_central_differences():
    # away from the clip edges and the mask edges the loss is smooth in logp_train
    rng = np.random.default_rng(24)
    T = 400
    lo = rng.standard_normal(T) * 0.1
    lt = lo + rng.standard_normal(T) * 0.3
    lr = lt + rng.standard_normal(T) * 0.4
    A = rng.standard_normal(T)
    r = np.exp(lt - lo)
    rho = np.exp(lt - lr)
    ok = (np.abs(r - 0.8) > 1e-3) & (np.abs(r - 1.28) > 1e-3) & (np.abs(rho - 0.5) > 1e-3) & (np.abs(rho - 2) > 1e-3)
    gr = head.ppo_icepop_grad(lt, lo, lr, A)
    eps = 1e-7
    for t in np.nonzero(ok)[0][:200]:
        p, m = lt.copy(), lt.copy()
        p[t] += eps; m[t] -= eps
        # the mask is held at its value at lt (an indicator has no derivative)
        lrp, lrm = lr.copy(), lr.copy()
        lrp[t] += eps; lrm[t] -= eps
        fd = (head.ppo_icepop_loss(p, lo, lrp, A)[1] - head.ppo_icepop_loss(m, lo, lrm, A)[1]) / (2 * eps)
        assert abs(fd - gr[t]) < 1e-7, (t, fd, gr[t])
    assert (gr == 0).sum() > 10 and (gr != 0).sum() > 200     # both regimes exercised
