"""Pins for oracle.head: log-sum-exp, token logprob, k3 and the IcePop mask."""
import json
import math
import os

import numpy as np
import scipy.special
import scipy.stats

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
