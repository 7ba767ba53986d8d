"""Pins for oracle.moe against brute force, closed forms and library routines."""
from fractions import Fraction
import itertools

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe
from oracle.numerics import round_to_bf16
from serve_invariant_moe_gb300 import synth


# ---------------------------------------------------------------- router logits

def test_router_logits_exact_on_integers():
    # brute force in exact rational arithmetic on a tiny integer-valued input
    rng = np.random.default_rng(3)
    x = rng.integers(-4, 5, size=(5, 7)).astype(np.float64)
    w = rng.integers(-4, 5, size=(3, 7)).astype(np.float64)
    L = moe.router_logits(x, w)
    assert L.shape == (5, 3)
    for t in range(5):
        for e in range(3):
            ref = sum(Fraction(int(x[t, h])) * Fraction(int(w[e, h])) for h in range(7))
            assert L[t, e] == float(ref)


def test_router_onehot_token_reads_one_column():
    rng = np.random.default_rng(4)
    w = rng.standard_normal((6, 9))
    x = np.eye(9)[[2, 7]]
    L = moe.router_logits(x, w)
    assert np.array_equal(L[0], w[:, 2]) and np.array_equal(L[1], w[:, 7])


# ---------------------------------------------------------------- top-k contract

def _brute_topk(row, k):
    """Rank counting: expert e beats f iff (e is not NaN and f is NaN) or
    L_e > L_f or (L_e == L_f, both or neither NaN, and e < f)."""
    E = len(row)

    def beats(e, f):
        ne, nf = np.isnan(row[e]), np.isnan(row[f])
        if ne != nf:
            return nf
        if ne and nf:
            return e < f
        if row[e] != row[f]:
            return row[e] > row[f]
        return e < f

    rank = [sum(beats(f, e) for f in range(E) if f != e) for e in range(E)]
    order = sorted(range(E), key=lambda e: rank[e])
    return order[:k]


def test_topk_brute_force_with_ties_nan_inf_signed_zero():
    rng = np.random.default_rng(5)
    pool = np.array([-2.0, -1.0, -0.0, 0.0, 1.0, 2.0, np.inf, -np.inf, np.nan])
    rows = pool[rng.integers(0, len(pool), size=(400, 8))]
    for k in (1, 2, 3, 8):
        got = moe.topk_lowest_index(rows, k)
        for t in range(rows.shape[0]):
            assert list(got[t]) == _brute_topk(rows[t], k), (rows[t], k)


def test_topk_hand_cases():
    assert list(moe.topk_lowest_index(np.zeros((1, 6)), 4)[0]) == [0, 1, 2, 3]
    assert list(moe.topk_lowest_index(np.full((1, 4), np.nan), 2)[0]) == [0, 1]
    row = np.array([[np.nan, -np.inf, 0.0, -0.0]])
    assert list(moe.topk_lowest_index(row, 4)[0]) == [2, 3, 1, 0]
    row = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    assert list(moe.topk_lowest_index(row, 3)[0]) == [1, 2, 4]
    assert moe.topk_lowest_index(row, 3).dtype == np.int32


def test_duplicated_router_rows_tie_to_lower_index():
    cfg = synth.TINY
    x, wr = synth.moe_activations(cfg)
    L = moe.router_logits(moe.to_f64(x), moe.to_f64(wr))
    assert np.array_equal(L[:, 0::2], L[:, 1::2])          # exact ties
    idx = moe.topk_lowest_index(L, cfg.k)
    # each token's top-2 is one duplicated pair, lower index first
    assert np.all(idx[:, 0] % 2 == 0) and np.all(idx[:, 1] == idx[:, 0] + 1)
    g = moe.topk_gates(L, idx)
    assert np.array_equal(g, np.full_like(g, 0.5))


# ---------------------------------------------------------------- gates

def test_gates_match_scipy_softmax():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((50, 16)) * 3
    idx = moe.topk_lowest_index(L, 4)
    g = moe.topk_gates(L, idx)
    sel = np.take_along_axis(L, idx.astype(np.int64), 1)
    assert np.allclose(g, scipy.special.softmax(sel, axis=1), rtol=1e-14, atol=0)
    assert np.allclose(g.sum(1), 1.0, rtol=0, atol=1e-15)
    # descending logits give non-increasing gates
    assert np.all(np.diff(g, axis=1) <= 0)


def test_gates_equal_logits():
    g = moe.topk_gates(np.full((3, 8), 1.25), moe.topk_lowest_index(np.full((3, 8), 1.25), 4))
    assert np.array_equal(g, np.full((3, 4), 0.25))


def test_gates_are_full_softmax_renormalised():
    rng = np.random.default_rng(7)
    L = rng.standard_normal((20, 10))
    idx = moe.topk_lowest_index(L, 3)
    full = scipy.special.softmax(L, axis=1)
    sel = np.take_along_axis(full, idx.astype(np.int64), 1)
    assert np.allclose(moe.topk_gates(L, idx), sel / sel.sum(1, keepdims=True), rtol=1e-13)


# ---------------------------------------------------------------- SwiGLU expert

def test_silu_matches_scipy():
    g = np.linspace(-30, 30, 1001)
    assert np.allclose(moe.silu(g), g * scipy.special.expit(g), rtol=1e-14, atol=1e-300)
    assert moe.silu(np.array([0.0]))[0] == 0.0


def test_swiglu_expert_structure():
    # gate = identity, up = a constant-one column, down = a permutation:
    # y = round_bf16(silu(x))[:, perm]  -- catches swapped gate/up and a
    # transposed down projection (the permutation is not an involution).
    H = F = 6
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, H))
    x[:, H - 1] = 1.0
    wg = np.eye(F, H)
    wu = np.zeros((F, H)); wu[:, H - 1] = 1.0
    perm = np.array([1, 2, 3, 4, 5, 0])
    w2 = np.eye(H)[perm]                    # (h @ w2.T)[:, i] = h[:, perm[i]]
    y = moe.swiglu_expert(x, np.concatenate([wg, wu]), w2, F)
    h = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    h = torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    # float32 step above is exact for these magnitudes only if h is a float32;
    # compare against the oracle's single-step rounding of the library silu.
    ref = round_to_bf16(torch.nn.functional.silu(torch.from_numpy(x)).numpy())[:, perm]
    assert np.array_equal(y, ref)
    assert np.allclose(y, h[:, perm], rtol=1e-2)


def test_swiglu_stages_compose_and_pin_separately():
    # the two stages the module-substitution tests feed one at a time
    rng = np.random.default_rng(18)
    H, F = 12, 8
    x = round_to_bf16(rng.standard_normal((7, H)))
    w13 = round_to_bf16(rng.standard_normal((2 * F, H)) * 0.3)
    w2 = round_to_bf16(rng.standard_normal((H, F)) * 0.3)
    h = moe.swiglu_hidden(x, w13, F)
    assert np.array_equal(moe.swiglu_expert(x, w13, w2, F), moe.down_projection(h, w2))
    # the hidden stage: silu(gate) * up, with gate and up taken from the right halves of w13
    g_t = torch.from_numpy(x) @ torch.from_numpy(w13[:F]).T
    u_t = torch.from_numpy(x) @ torch.from_numpy(w13[F:]).T
    ref_h = (torch.nn.functional.silu(g_t) * u_t).numpy()
    assert np.allclose(moe.swiglu_hidden(x, w13, F, round_h=False), ref_h, rtol=1e-13, atol=1e-13)
    assert np.array_equal(h, round_to_bf16(moe.swiglu_hidden(x, w13, F, round_h=False)))
    # the down stage: a selection matrix W2 = rows of the identity returns the chosen h columns
    sel = np.array([3, 0, 7, 1, 1, 5, 2, 6, 4, 0, 3, 7])
    assert np.array_equal(moe.down_projection(h, np.eye(F)[sel]), h[:, sel])


def _tiny_layer(T=24, H=32, E=6, k=2, F=16, seed=9):
    rng = np.random.default_rng(seed)
    x = round_to_bf16(rng.standard_normal((T, H)))
    wr = round_to_bf16(rng.standard_normal((E, H)) * 0.2)
    w13 = round_to_bf16(rng.standard_normal((E, 2 * F, H)) * 0.2)
    w2 = round_to_bf16(rng.standard_normal((E, H, F)) * 0.2)
    return x, wr, w13, w2


@pytest.mark.parametrize("k", [1, 2, 3, 6])
def test_sparse_equals_dense_all_experts_then_mask(k):
    x, wr, w13, w2 = _tiny_layer(k=k)
    sparse = moe.moe_forward(x, wr, w13, w2, k, 16)["out"]
    dense = moe.dense_all_experts_then_mask(x, wr, w13, w2, k, 16)
    assert np.allclose(sparse, dense, rtol=1e-12, atol=1e-12)


def test_single_expert_k1_is_plain_mlp():
    x, wr, w13, w2 = _tiny_layer(E=1, k=1)
    out = moe.moe_forward(x, wr, w13, w2, 1, 16)["out"]
    assert np.array_equal(out, moe.swiglu_expert(x, w13[0], w2[0], 16))


def test_shared_expert_added():
    x, wr, w13, w2 = _tiny_layer()
    rng = np.random.default_rng(10)
    ws13 = round_to_bf16(rng.standard_normal((2 * 8, 32)) * 0.2)
    ws2 = round_to_bf16(rng.standard_normal((32, 8)) * 0.2)
    a = moe.moe_forward(x, wr, w13, w2, 2, 16)["out"]
    b = moe.moe_forward(x, wr, w13, w2, 2, 16, ws13, ws2, 8)["out"]
    assert np.allclose(b - a, moe.swiglu_expert(x, ws13, ws2, 8), rtol=1e-12, atol=1e-12)


def test_dispatch_plan_invariants():
    rng = np.random.default_rng(11)
    T, E, k = 50, 7, 3
    L = rng.standard_normal((T, E))
    L[:, 5] = -1e9                      # expert 5 never chosen: an empty segment
    idx = moe.topk_lowest_index(L, k)
    counts, offsets, row_token, slot_row = moe.dispatch_plan(idx, E)
    assert counts.sum() == T * k and counts[5] == 0
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert np.array_equal(np.diff(offsets), counts)
    for e in range(E):
        seg = row_token[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)              # ascending, no repeats
        assert set(seg) == set(np.nonzero((idx == e).any(1))[0])
    for t in range(T):
        for j in range(k):
            r = slot_row[t, j]
            assert row_token[r] == t and offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]
    # the multiset of rows is a permutation
    assert sorted(slot_row.ravel()) == list(range(T * k))


def test_combine_is_gate_weighted_sum():
    rng = np.random.default_rng(12)
    y = rng.standard_normal((4, 3, 5))
    g = rng.random((4, 3))
    ys = rng.standard_normal((4, 5))
    ref = np.einsum("tj,tjh->th", g, y) + ys
    assert np.allclose(moe.combine(y, g, ys), ref, rtol=1e-14, atol=1e-14)
    # a single slot with gate 1 returns that slot's output
    assert np.array_equal(moe.combine(y[:, :1], np.ones((4, 1))), y[:, 0])


@pytest.mark.parametrize("name", ["qwen_moe_like", "qwen_moe_like_empty"])
def test_skewed_layer_has_busy_experts(name):
    cfg = synth.CONFIGS[name]
    x, wr = synth.moe_activations(cfg)
    idx = moe.topk_lowest_index(moe.router_logits(moe.to_f64(x), moe.to_f64(wr)), cfg.k)
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    assert 1200 <= counts.max() <= 1800
    assert counts.sum() == cfg.T * cfg.k
    # the starved variant: per-expert counts from 0 to about 1500
    assert (counts == 0).sum() == cfg.zipf_starve


def test_replay_of_own_choice_is_the_plain_forward():
    x, wr, w13, w2 = _tiny_layer(k=3)
    a = moe.moe_forward(x, wr, w13, w2, 3, 16)
    b = moe.moe_forward(x, wr, w13, w2, 3, 16, replay_idx=a["idx"])
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["gates"], b["gates"])
    # replaying other experts changes the output but keeps gates a distribution over them
    idx = (a["idx"] + 1) % 6
    c = moe.moe_forward(x, wr, w13, w2, 3, 16, replay_idx=idx)
    assert np.array_equal(c["idx"], idx) and np.allclose(c["gates"].sum(1), 1.0)
    dense = np.zeros_like(x)
    for e in range(6):
        ye = moe.swiglu_expert(x, w13[e], w2[e], 16)
        for j in range(3):
            dense += ((idx[:, j] == e) * c["gates"][:, j])[:, None] * ye
    assert np.allclose(c["out"], dense, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward

def _bwd_case(seed=30, T=5, H=6, E=4, k=2, F=3, Fs=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) * 0.7
    w13 = rng.standard_normal((E, 2 * F, H)) * 0.5
    w2 = rng.standard_normal((E, H, F)) * 0.5
    ws13 = rng.standard_normal((2 * Fs, H)) * 0.5
    ws2 = rng.standard_normal((H, Fs)) * 0.5
    dout = rng.standard_normal((T, H))
    return x, wr, w13, w2, ws13, ws2, dout


def test_moe_backward_central_differences():
    """Every element of every gradient against a central difference of sum(dout * out),
    with no bf16 rounding anywhere (the chain rule itself is what is pinned)."""
    x, wr, w13, w2, ws13, ws2, dout = _bwd_case()
    k, F, Fs = 2, 3, 2
    L = moe.router_logits(x, wr)
    srt = np.sort(L, axis=1)
    assert np.min(srt[:, 1:] - srt[:, :-1]) > 1e-3          # no selection flips under the perturbation
    g = moe.moe_backward(x, wr, w13, w2, k, F, dout, ws13, ws2, Fs, round_ops=False)

    def f(x_, wr_, w13_, w2_, ws13_, ws2_):
        out = moe.moe_forward(x_, wr_, w13_, w2_, k, F, ws13_, ws2_, Fs, round_h=False)["out"]
        return float(np.sum(dout * out))

    args = [x, wr, w13, w2, ws13, ws2]
    names = ["dx", "dw_router", "dw13", "dw2", "dws13", "dws2"]
    eps = 1e-6
    for a_i, name in enumerate(names):
        grad = g[name]
        assert grad.shape == args[a_i].shape, name
        for i in np.ndindex(args[a_i].shape):
            ap = [a.copy() for a in args]; am = [a.copy() for a in args]
            ap[a_i][i] += eps; am[a_i][i] -= eps
            fd = (f(*ap) - f(*am)) / (2 * eps)
            assert abs(fd - grad[i]) < 1e-6 * max(1.0, abs(fd)), (name, i, fd, grad[i])


def test_moe_backward_structure():
    x, wr, w13, w2, ws13, ws2, dout = _bwd_case(31, T=9)
    g = moe.moe_backward(x, wr, w13, w2, 2, 3, dout, ws13, ws2, 2, round_ops=False)
    fwd = g["fwd"]
    # dgate is the inner product of the upstream gradient with each slot's expert output
    assert np.allclose(g["dgate"], np.einsum("th,tjh->tj", dout, fwd["y"]), rtol=1e-14)
    # the softmax Jacobian over the selected experts: each token's router gradient sums to 0,
    # and experts not selected get exactly 0
    assert np.allclose(g["dlogits"].sum(1), 0, atol=1e-14)
    sel = np.zeros_like(g["dlogits"], bool)
    np.put_along_axis(sel, fwd["idx"].astype(np.int64), True, axis=1)
    assert np.all(g["dlogits"][~sel] == 0)
    # dx is the sum of the expert, shared and router parts
    assert np.allclose(g["dx"], g["dxp"].sum(1) + g["dx_shared"] + g["dx_router"], rtol=1e-13, atol=1e-13)
    # an expert no token chose has zero weight gradients
    x1, wr1 = x.copy(), wr.copy()
    x1[:, 0] = 5.0
    wr1[3, 0] = -100.0                                       # expert 3's logit is about -500 for every token
    g1 = moe.moe_backward(x1, wr1, w13, w2, 2, 3, dout, round_ops=False)
    assert not (g1["fwd"]["idx"] == 3).any()
    assert np.all(g1["dw13"][3] == 0) and np.all(g1["dw2"][3] == 0) and np.all(g1["dw_router"][3] == 0)


def test_moe_backward_rounded_operands_close_to_exact():
    x, wr, w13, w2, ws13, ws2, dout = _bwd_case(32, T=40, H=16, E=6, k=3, F=8, Fs=8)
    a = moe.moe_backward(x, wr, w13, w2, 3, 8, dout, ws13, ws2, 8, round_ops=False)
    b = moe.moe_backward(x, wr, w13, w2, 3, 8, dout, ws13, ws2, 8, round_ops=True)
    for name in ("dx", "dw_router", "dw13", "dw2", "dws13", "dws2"):
        scale = np.abs(a[name]).max()
        assert np.abs(a[name] - b[name]).max() <= 2e-2 * scale, name
    assert np.array_equal(round_to_bf16(b["dgu"]), b["dgu"]) and np.array_equal(round_to_bf16(b["dy"]), b["dy"])


def test_swiglu_backward_matches_torch_autograd():
    rng = np.random.default_rng(33)
    x = torch.from_numpy(rng.standard_normal((7, 5))).requires_grad_(True)
    w13 = torch.from_numpy(rng.standard_normal((8, 5))).requires_grad_(True)
    w2 = torch.from_numpy(rng.standard_normal((5, 4))).requires_grad_(True)
    dy = torch.from_numpy(rng.standard_normal((7, 5)))
    g, u = x @ w13[:4].T, x @ w13[4:].T
    ((torch.nn.functional.silu(g) * u) @ w2.T * dy).sum().backward()
    b = moe.swiglu_backward(x.detach().numpy(), w13.detach().numpy(), w2.detach().numpy(), 4, dy.numpy(),
                            round_ops=False)
    for name, t in (("dx", x), ("dw13", w13), ("dw2", w2)):
        assert np.allclose(b[name], t.grad.numpy(), rtol=1e-12, atol=1e-12), name


def test_moe_backward_replay_of_own_choice_is_the_plain_backward():
    x, wr, w13, w2, ws13, ws2, dout = _bwd_case(34, T=7)
    a = moe.moe_backward(x, wr, w13, w2, 2, 3, dout, ws13, ws2, 2, round_ops=False)
    b = moe.moe_backward(x, wr, w13, w2, 2, 3, dout, ws13, ws2, 2, round_ops=False, replay_idx=a["fwd"]["idx"])
    for name in ("dx", "dw_router", "dw13", "dw2", "dws13", "dws2"):
        assert np.array_equal(a[name], b[name]), name


def test_moe_backward_with_replayed_experts_central_differences():
    """Other experts replayed: the router gradient is the softmax Jacobian over the replayed logits."""
    x, wr, w13, w2, _, _, dout = _bwd_case(35, T=4)
    idx = np.array([[3, 0], [1, 2], [2, 3], [0, 1]], dtype=np.int32)
    g = moe.moe_backward(x, wr, w13, w2, 2, 3, dout, round_ops=False, replay_idx=idx)

    def f(x_, wr_):
        return float(np.sum(dout * moe.moe_forward(x_, wr_, w13, w2, 2, 3, round_h=False, replay_idx=idx)["out"]))

    eps = 1e-6
    for arr, name in ((x, "dx"), (wr, "dw_router")):
        for i in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[i] += eps; m[i] -= eps
            fd = (f(p, wr) - f(m, wr)) / (2 * eps) if name == "dx" else (f(x, p) - f(x, m)) / (2 * eps)
            assert abs(fd - g[name][i]) < 1e-6 * max(1.0, abs(fd)), (name, i)
