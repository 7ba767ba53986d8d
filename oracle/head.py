"""Logprob / KL head oracle: plain float64 restatement (test infrastructure only).

* "GLM Post-Training Beyond SFT", section "IcePop 为什么有两层 ratio":
  rho_t = pi_train(y_t | s_t) / pi_infer(y_t | s_t) = exp(logp_train - logp_infer)
  and the trust mask m_t = 1[1/beta <= rho_t <= beta], beta = 2 (keeps
  rho in [1/2, 2], both ends included).  The rollout pseudo-code in that
  section computes the train logprob of the exact rollout token ids.
* Same page, section "动作与概率契约": sampled log-prob precision and the
  logsumexp reduction must have comparison tests.
* "Reinforcement Learning: Why Numerical Alignment and MoE Routing Matter So
  Much", section "混合专家模型更难对齐": k3 is the train/inference divergence
  metric, with 0.001 as the equivalence threshold.  The page names k3 without
  its formula; the standard k3 estimator is (r - 1) - log r with
  r = pi_train / pi_rollout on rollout-sampled tokens (so r = rho), written
  here as expm1(d) - d with d = logp_train - logp_rollout.
"""
import numpy as np


def vocab_logits(hidden: np.ndarray, w_vocab: np.ndarray) -> np.ndarray:
    """Z[t, v] = sum_h hidden[t, h] * Wv[v, h], float64."""
    return np.asarray(hidden, np.float64) @ np.asarray(w_vocab, np.float64).T


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """lse[t] = log sum_v exp(z[t, v]), float64, with the max shift."""
    z = np.asarray(z, np.float64)
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def token_logprob(z: np.ndarray, target: np.ndarray):
    """log-softmax of row t at the exact target id: z[t, target[t]] - lse[t].

    Returns (logp, lse) in float64.
    """
    z = np.asarray(z, np.float64)
    lse = logsumexp_rows(z)
    tgt = np.asarray(target, np.int64)
    logp = z[np.arange(z.shape[0]), tgt] - lse
    return logp, lse


def k3(logp_train, logp_rollout) -> np.ndarray:
    """k3 = (r - 1) - log r, r = exp(d), d = logp_train - logp_rollout; = expm1(d) - d.

    Exactly 0 when the two logprobs agree; never negative.
    """
    d = np.asarray(logp_train, np.float64) - np.asarray(logp_rollout, np.float64)
    return np.expm1(d) - d


def icepop_mask(logp_train, logp_rollout, beta: float = 2.0, dtype=np.float64) -> np.ndarray:
    """m_t = 1[1/beta <= rho_t <= beta], rho_t = exp(logp_train - logp_rollout).

    ``dtype`` is the precision in which the ratio and the comparison are
    taken.  Where two implementations must agree on this integer decision they
    take it in the same precision; the GPU kernel takes it in float32, so the
    parity tests call this with dtype=np.float32 on the kernel's own float32
    difference d.
    """
    lt = np.asarray(logp_train, dtype)
    lr = np.asarray(logp_rollout, dtype)
    d = (lt - lr).astype(dtype)
    rho = np.exp(d).astype(dtype)
    b = dtype(beta)
    lo = dtype(dtype(1.0) / b)
    return ((lo <= rho) & (rho <= b)).astype(np.uint8)


def head_forward(hidden, w_vocab, target, logp_rollout=None, beta=2.0):
    """Whole head, float64: logits -> lse -> logprob (-> k3, IcePop mask)."""
    z = vocab_logits(hidden, w_vocab)
    logp, lse = token_logprob(z, target)
    out = dict(logits=z, logp=logp, lse=lse)
    if logp_rollout is not None:
        out["k3"] = k3(logp, logp_rollout)
        out["mask"] = icepop_mask(logp, logp_rollout, beta)
    return out


def ppo_icepop_loss(logp_train, logp_old, logp_rollout, advantage, beta=2.0, eps_low=0.2, eps_high=0.28,
                    dtype=np.float64):
    """IcePop-masked clipped policy loss per token, and its mean over tokens.

    "GLM Post-Training Beyond SFT", section "GRPO 在优化什么": with the ratio
    r_t = pi_theta / pi_old the clipped objective is
    min(r_t A, clip(r_t, 1 - eps_l, 1 + eps_h) A), eps_l = 0.2, eps_h = 0.28
    (section "IcePop 为什么有两层 ratio"); the same section multiplies the trust
    mask m_t = 1[1/beta <= rho_t <= beta], rho_t = pi_train / pi_infer, into the
    token loss, which is the negated objective:
        loss_t = -m_t * min(r_t A_t, clip(r_t, 1 - eps_l, 1 + eps_h) A_t).
    The mask decision is taken in ``dtype`` (see icepop_mask).  Returns
    (loss_t [T] float64, mean loss float64).
    """
    lt = np.asarray(logp_train, np.float64)
    lo = np.asarray(logp_old, np.float64)
    A = np.asarray(advantage, np.float64)
    r = np.exp(lt - lo)
    m = icepop_mask(logp_train, logp_rollout, beta, dtype).astype(np.float64)
    obj = np.minimum(r * A, np.clip(r, 1.0 - eps_low, 1.0 + eps_high) * A)
    loss = -m * obj
    return loss, float(loss.mean()) if loss.size else 0.0


def dis_weight(logp_train, logp_rollout, eps_low=0.2, eps_high=0.28):
    """Direct double-sided importance weight ("GLM Post-Training Beyond SFT",
    section "Direct Double-Sided Importance Sampling"):
    r_t = exp(logp_theta - logp_rollout);  f(r_t) = r_t if 1 - eps_l < r_t < 1 + eps_h, else 0
    (both ends excluded; 0 means the token gives no gradient)."""
    r = np.exp(np.asarray(logp_train, np.float64) - np.asarray(logp_rollout, np.float64))
    return np.where((1.0 - eps_low < r) & (r < 1.0 + eps_high), r, 0.0)


# ----------------------------------------------------------------------------
# backward of the head (the trainer's side of the same definition)
# ----------------------------------------------------------------------------

def ppo_icepop_grad(logp_train, logp_old, logp_rollout, advantage, beta=2.0, eps_low=0.2, eps_high=0.28,
                    dtype=np.float64):
    """Derivative of the mean IcePop-masked clipped loss with respect to each logp_train.

    From ``ppo_icepop_loss``: loss_t = -m_t * min(r_t A_t, clip(r_t) A_t) with
    r_t = exp(logp_train_t - logp_old_t), mean over the T tokens.  The mask
    m_t is an indicator (piecewise constant in logp_train), so it is held fixed.
    Where the unclipped term attains the minimum (r A <= clip(r) A, which
    includes every r inside the clip window) d(r A)/d logp_train = r A; where the
    clipped term is strictly smaller it is a constant and the derivative is 0:
        g_t = -(1/T) * m_t * r_t * A_t * 1[r_t A_t <= clip(r_t) A_t].
    Returns g [T] float64.
    """
    lt = np.asarray(logp_train, np.float64)
    lo = np.asarray(logp_old, np.float64)
    A = np.asarray(advantage, np.float64)
    T = lt.shape[0]
    if T == 0:
        return np.zeros(0)
    r = np.exp(lt - lo)
    m = icepop_mask(logp_train, logp_rollout, beta, dtype).astype(np.float64)
    unclipped = r * A <= np.clip(r, 1.0 - eps_low, 1.0 + eps_high) * A
    return np.where(unclipped, -(m * r * A) / T, 0.0)


def dlogits(z, target, grad_logp):
    """dL/dz[t, v] for L = sum_t g_t * logp_t, logp_t = z[t, target_t] - lse(z_t):
        dz[t, v] = g_t * (1[v == target_t] - softmax(z_t)_v),
    float64.  A token with g_t = 0 (dropped by the IcePop mask, or clipped)
    contributes nothing."""
    z = np.asarray(z, np.float64)
    g = np.asarray(grad_logp, np.float64)
    lse = logsumexp_rows(z)
    p = np.exp(z - lse[:, None])
    onehot = np.zeros_like(z)
    onehot[np.arange(z.shape[0]), np.asarray(target, np.int64)] = 1.0
    return g[:, None] * (onehot - p)


def head_backward(hidden, w_vocab, target, grad_logp, round_dz=True):
    """Gradients of L = sum_t g_t * logp_t through the vocabulary projection, float64.

        Z = Hs Wv^T,  dZ = dlogits(Z),  dHs = dZ Wv,  dWv = dZ^T Hs.
    dZ is the bf16 operand of the two gradient products, so it is rounded to
    bf16 (nearest-even) first when round_dz, as the forward rounds h.
    Returns dict(dz, d_hidden, d_wvocab).
    """
    from .numerics import round_to_bf16
    hs = np.asarray(hidden, np.float64)
    wv = np.asarray(w_vocab, np.float64)
    dz = dlogits(vocab_logits(hs, wv), target, grad_logp)
    if round_dz:
        dz = round_to_bf16(dz)
    return dict(dz=dz, d_hidden=dz @ wv, d_wvocab=dz.T @ hs)
