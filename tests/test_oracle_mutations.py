"""Planted mistakes: each replaces one oracle function with a plausible wrong
version (on the CPU) and checks that a pin of the oracle tests catches it."""
import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

from oracle import head, moe, numerics


def _pin_topk(topk):
    pool = np.array([-1.0, 0.0, 1.0, np.nan, -np.inf])
    rng = np.random.default_rng(0)
    rows = pool[rng.integers(0, len(pool), size=(200, 6))]
    from test_oracle_moe import _brute_topk
    got = topk(rows, 3)
    for t in range(rows.shape[0]):
        assert list(got[t]) == _brute_topk(rows[t], 3)


def _pin_gates(gates_fn):
    rng = np.random.default_rng(1)
    L = rng.standard_normal((20, 8))
    idx = moe.topk_lowest_index(L, 3)
    sel = np.take_along_axis(L, idx.astype(np.int64), 1)
    assert np.allclose(gates_fn(L, idx), scipy.special.softmax(sel, axis=1), rtol=1e-13)


def _pin_swiglu(expert):
    H = F = 6
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, H)); x[:, H - 1] = 1.0
    wg = np.eye(F, H); wu = np.zeros((F, H)); wu[:, H - 1] = 1.0
    perm = np.array([1, 2, 3, 4, 5, 0])
    y = expert(x, np.concatenate([wg, wu]), np.eye(H)[perm], F)
    ref = numerics.round_to_bf16(torch.nn.functional.silu(torch.from_numpy(x)).numpy())[:, perm]
    assert np.array_equal(y, ref)


def _pin_k3(k3_fn):
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(30)); q = rng.dirichlet(np.ones(30))
    assert abs(np.sum(q * k3_fn(np.log(p), np.log(q))) - scipy.stats.entropy(q, p)) < 1e-12


def _pin_round(round_fn):
    x = np.random.default_rng(4).standard_normal(5000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(round_fn(x.astype(np.float64)), ref)


def _pin_lse(lse_fn):
    z = np.random.default_rng(5).standard_normal((5, 300)) * 30 + 1000.0   # large logits
    assert np.allclose(lse_fn(z), scipy.special.logsumexp(z, axis=1), rtol=1e-13, atol=1e-12)


def _pin_head_backward(hb):
    rng = np.random.default_rng(6)
    T, H, V = 2, 4, 5
    hs = rng.standard_normal((T, H)); wv = rng.standard_normal((V, H)) * 0.5
    tgt = np.array([4, 1]); g = np.array([0.75, -1.5])

    def f(a, b):
        logp, _ = head.token_logprob(head.vocab_logits(a, b), tgt)
        return float(np.dot(g, logp))

    out = hb(hs, wv, tgt, g, round_dz=False)
    eps = 1e-6
    for i in np.ndindex(hs.shape):
        p, m = hs.copy(), hs.copy(); p[i] += eps; m[i] -= eps
        assert abs((f(p, wv) - f(m, wv)) / (2 * eps) - out["d_hidden"][i]) < 1e-7
    for i in np.ndindex(wv.shape):
        p, m = wv.copy(), wv.copy(); p[i] += eps; m[i] -= eps
        assert abs((f(hs, p) - f(hs, m)) / (2 * eps) - out["d_wvocab"][i]) < 1e-7


def _pin_ppo_grad(gfn):
    rng = np.random.default_rng(7)
    T = 300
    lo = rng.standard_normal(T) * 0.1
    lt = lo + rng.standard_normal(T) * 0.3
    lr = lt + rng.standard_normal(T) * 0.4
    A = rng.standard_normal(T)
    r, rho = np.exp(lt - lo), np.exp(lt - lr)
    ok = (np.abs(r - 0.8) > 1e-3) & (np.abs(r - 1.28) > 1e-3) & (np.abs(rho - 0.5) > 1e-3) & (np.abs(rho - 2) > 1e-3)
    gr = gfn(lt, lo, lr, A)
    eps = 1e-7
    for t in np.nonzero(ok)[0]:
        p, m = lt.copy(), lt.copy(); p[t] += eps; m[t] -= eps
        lp, lm = lr.copy(), lr.copy(); lp[t] += eps; lm[t] -= eps
        fd = (head.ppo_icepop_loss(p, lo, lp, A)[1] - head.ppo_icepop_loss(m, lo, lm, A)[1]) / (2 * eps)
        assert abs(fd - gr[t]) < 1e-7


def _pin_moe_backward(bwd):
    rng = np.random.default_rng(8)
    T, H, E, k, F = 4, 5, 3, 2, 3
    x = rng.standard_normal((T, H)); wr = rng.standard_normal((E, H)) * 0.7
    w13 = rng.standard_normal((E, 2 * F, H)) * 0.5; w2 = rng.standard_normal((E, H, F)) * 0.5
    dout = rng.standard_normal((T, H))
    g = bwd(x, wr, w13, w2, k, F, dout, round_ops=False)

    def f(args):
        return float(np.sum(dout * moe.moe_forward(*args, k, F, round_h=False)["out"]))

    base = [x, wr, w13, w2]
    eps = 1e-6
    for a_i, name in enumerate(["dx", "dw_router", "dw13", "dw2"]):
        for i in np.ndindex(base[a_i].shape):
            ap = [a.copy() for a in base]; am = [a.copy() for a in base]
            ap[a_i][i] += eps; am[a_i][i] -= eps
            assert abs((f(ap) - f(am)) / (2 * eps) - g[name][i]) < 1e-6


def test_pins_pass_on_the_real_oracle():
    _pin_moe_backward(moe.moe_backward)
    _pin_head_backward(head.head_backward)
    _pin_ppo_grad(head.ppo_icepop_grad)
    _pin_topk(moe.topk_lowest_index)
    _pin_gates(moe.topk_gates)
    _pin_swiglu(moe.swiglu_expert)
    _pin_k3(head.k3)
    _pin_round(numerics.round_to_bf16)
    _pin_lse(head.logsumexp_rows)


def _topk_high_index_ties(L, k):            # ties to the higher index
    L = np.asarray(L, np.float64)
    E = L.shape[1]
    nan = np.isnan(L)
    idx = np.broadcast_to(-np.arange(E), L.shape)
    return np.lexsort((idx, np.where(nan, 0.0, -L), nan), axis=-1)[:, :k].astype(np.int32)


def _topk_nan_first(L, k):                  # NaN treated as the largest value
    L = np.asarray(L, np.float64)
    return moe.topk_lowest_index(np.where(np.isnan(L), np.inf, L), k)


def _gates_not_renormalised(L, idx):        # full softmax, not renormalised over the top-k
    full = scipy.special.softmax(np.asarray(L, np.float64), axis=1)
    return np.take_along_axis(full, idx.astype(np.int64), 1)


def _swiglu_swapped(x, w13, w2, F, round_h=True):   # gate and up exchanged
    return moe.swiglu_expert(x, np.concatenate([w13[F:2 * F], w13[:F]]), w2, F, round_h)


def _swiglu_down_transposed(x, w13, w2, F, round_h=True):
    return moe.swiglu_expert(x, w13, np.asarray(w2).T, F, round_h)


def _k3_reversed(lt, lr):                  # ratio taken the other way round
    return head.k3(lr, lt)


def _round_truncate(x):                    # truncation instead of round-to-nearest-even
    x = np.asarray(x, np.float64).astype(np.float32)
    b = (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    return b.astype(np.float64)


def _lse_no_shift(z):                      # forgot the max shift (overflows / underflows)
    return np.log(np.exp(np.asarray(z, np.float64)).sum(axis=1))


def _hb_sign_flipped(hs, wv, tgt, g, round_dz=True):    # softmax - onehot without the minus of g
    out = head.head_backward(hs, wv, tgt, g, round_dz)
    return {k: -v for k, v in out.items()}


def _hb_no_onehot(hs, wv, tgt, g, round_dz=True):        # dropped the one-hot term
    hs = np.asarray(hs, np.float64); wv = np.asarray(wv, np.float64)
    z = head.vocab_logits(hs, wv)
    dz = -np.asarray(g)[:, None] * np.exp(z - head.logsumexp_rows(z)[:, None])
    return dict(dz=dz, d_hidden=dz @ wv, d_wvocab=dz.T @ hs)


def _hb_unscaled(hs, wv, tgt, g, round_dz=True):         # forgot the per-token upstream gradient
    return head.head_backward(hs, wv, tgt, np.ones_like(np.asarray(g, np.float64)), round_dz)


def _ppo_grad_no_ratio(lt, lo, lr, A, *a):               # d(r A)/d logp taken as A, not r A
    r = np.exp(np.asarray(lt) - np.asarray(lo))
    g = head.ppo_icepop_grad(lt, lo, lr, A, *a)
    return g / r


def _ppo_grad_no_clip(lt, lo, lr, A, beta=2.0, *a):      # ignored the clipped branch
    r = np.exp(np.asarray(lt) - np.asarray(lo))
    m = head.icepop_mask(lt, lr, beta).astype(np.float64)
    return -(m * r * np.asarray(A)) / len(r)


def _ppo_grad_no_mask(lt, lo, lr, A, *a):                # ignored the IcePop mask
    return head.ppo_icepop_grad(lt, lo, lt, A, *a)


def _with_swiglu_backward(fake):
    """moe_backward with its per-expert SwiGLU backward replaced by ``fake``."""
    def bwd(*a, **kw):
        real = moe.swiglu_backward
        moe.swiglu_backward = fake
        try:
            return moe.moe_backward(*a, **kw)
        finally:
            moe.swiglu_backward = real
    return bwd


def _swiglu_bwd_no_silu_slope(x_rows, w13, w2, F, dy, round_ops=True):   # silu'(g) taken as sigmoid(g)
    x_rows = np.asarray(x_rows, np.float64); w13 = np.asarray(w13, np.float64)
    g = x_rows @ w13[:F].T; u = x_rows @ w13[F:2 * F].T
    s = 1.0 / (1.0 + np.exp(-g))
    h = g * s * u
    dh = np.asarray(dy) @ np.asarray(w2)
    dgu = np.concatenate([dh * u * s, dh * g * s], axis=1)
    return dict(dh=dh, dgu=dgu, h=h, dx=dgu @ w13, dw13=dgu.T @ x_rows, dw2=np.asarray(dy).T @ h)


_REAL_SWIGLU_BACKWARD = moe.swiglu_backward


def _swiglu_bwd_gate_up_swapped(x_rows, w13, w2, F, dy, round_ops=True):
    b = _REAL_SWIGLU_BACKWARD(x_rows, w13, w2, F, dy, round_ops)
    dgu = np.concatenate([b["dgu"][:, F:], b["dgu"][:, :F]], axis=1)
    w13 = np.asarray(w13, np.float64)
    return dict(b, dgu=dgu, dx=dgu @ w13, dw13=dgu.T @ np.asarray(x_rows, np.float64))


def _moe_bwd_no_jacobian_centering(x, wr, w13, w2, k, F, dout, **kw):   # ds = w * dgate
    g = moe.moe_backward(x, wr, w13, w2, k, F, dout, **kw)
    fwd = g["fwd"]
    ds = fwd["gates"] * g["dgate"]
    dlog = np.zeros_like(g["dlogits"])
    np.put_along_axis(dlog, fwd["idx"].astype(np.int64), ds, axis=1)
    dx = g["dx"] - g["dx_router"] + dlog @ np.asarray(wr)
    return dict(g, dx=dx, dw_router=dlog.T @ np.asarray(x))


def _moe_bwd_unscaled_dy(x, wr, w13, w2, k, F, dout, **kw):              # forgot the gate in dy
    E = np.asarray(w13).shape[0]
    g = moe.moe_backward(x, wr, w13, w2, k, F, dout, **kw)
    idx = g["fwd"]["idx"]
    dx = g["dx"] - g["dxp"].sum(1)
    dw13 = np.zeros_like(g["dw13"]); dw2 = np.zeros_like(g["dw2"])
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size:
            b = moe.swiglu_backward(np.asarray(x)[tok], w13[e], w2[e], F, np.asarray(dout)[tok], False)
            np.add.at(dx, tok, b["dx"]); dw13[e] = b["dw13"]; dw2[e] = b["dw2"]
    return dict(g, dx=dx, dw13=dw13, dw2=dw2)


@pytest.mark.parametrize("pin, wrong", [
    (_pin_moe_backward, _with_swiglu_backward(_swiglu_bwd_no_silu_slope)),
    (_pin_moe_backward, _with_swiglu_backward(_swiglu_bwd_gate_up_swapped)),
    (_pin_moe_backward, _moe_bwd_no_jacobian_centering),
    (_pin_moe_backward, _moe_bwd_unscaled_dy),
    (_pin_head_backward, _hb_sign_flipped),
    (_pin_head_backward, _hb_no_onehot),
    (_pin_head_backward, _hb_unscaled),
    (_pin_ppo_grad, _ppo_grad_no_ratio),
    (_pin_ppo_grad, _ppo_grad_no_clip),
    (_pin_ppo_grad, _ppo_grad_no_mask),
    (_pin_topk, _topk_high_index_ties),
    (_pin_topk, _topk_nan_first),
    (_pin_gates, _gates_not_renormalised),
    (_pin_swiglu, _swiglu_swapped),
    (_pin_swiglu, _swiglu_down_transposed),
    (_pin_k3, _k3_reversed),
    (_pin_round, _round_truncate),
    (_pin_lse, _lse_no_shift),
])
def test_planted_mistake_is_caught(pin, wrong):
    with pytest.raises(AssertionError), np.errstate(all="ignore"):
        pin(wrong)
