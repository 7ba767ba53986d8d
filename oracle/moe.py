"""MoE layer oracle: plain float64 restatement (test infrastructure only).

What the layer computes, from the pages:

* "位级一致：前沿训练的差异化关键", section "为什么比特级一致是一个复杂的问题":
  the router and the per-expert matmuls are reductions whose order must depend
  only on the request; a router near-tie flips which expert fires; the fix is a
  deterministic tie decision in the router and one fixed kernel choice for the
  expert matmuls whatever the per-expert token count.
* "Reinforcement Learning: Why Numerical Alignment and MoE Routing Matter So
  Much", section "混合专家模型更难对齐": the weighted sum of expert outputs must
  use the same precision and the same order on both paths.
* "GLM Post-Training Beyond SFT", section "迁移到 NPU 时": a top-k must pin ties,
  boundary ties, sort order, NaN handling and the index dtype; compare the
  index set, its order and the final log-prob.

The method does not change the mathematics of an MoE layer, only the order of
its floating-point reductions, so the oracle is the textbook definition written
out in float64 over bf16-rounded inputs.  Where the pages are silent (gate
function, intermediate precisions, NaN rank) the reading taken is stated at the
function that depends on it.
"""
import numpy as np

from .numerics import bf16_bits_to_f64, round_to_bf16


def to_f64(t) -> np.ndarray:
    """bf16 torch tensor / uint16 array / float array -> float64 numpy array (exact)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.bfloat16:
                return bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
            return t.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover - torch is always present in this repo
        pass
    a = np.asarray(t)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------
# router
# ----------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """L[t, e] = sum_h x[t, h] * Wr[e, h], in float64.

    The router is the first reduction the bit-agreement page lists as needing a
    pinned order; in exact arithmetic it is a plain matrix product.
    """
    return np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T


def topk_lowest_index(logits: np.ndarray, k: int) -> np.ndarray:
    """Per row: the k largest logits, in descending order, exact ties to the lower index.

    Contract (bit-agreement page: "deterministic tie decision in the router";
    GLM post-training page, "迁移到 NPU 时": ties, sort order and NaN handling
    must be fixed):
      * order by logit, largest first;
      * equal logits (including -0.0 == +0.0) keep ascending expert index;
      * NaN ranks below every number including -inf; NaNs keep index order.
    Returns int32 indices of shape [T, k].
    """
    L = np.asarray(logits, np.float64)
    T, E = L.shape
    if not (0 < k <= E):
        raise ValueError("need 0 < k <= E")
    nan = np.isnan(L)
    neg = np.where(nan, 0.0, -L)              # ascending -L == descending L; -(-0.0) == 0.0 ties
    idx = np.broadcast_to(np.arange(E), (T, E))
    # np.lexsort: the last key is the primary key.  Primary: NaN last.
    order = np.lexsort((idx, neg, nan), axis=-1)
    return order[:, :k].astype(np.int32)


def topk_gates(logits: np.ndarray, topk_idx: np.ndarray) -> np.ndarray:
    """Gate weights: softmax over the k selected logits (renormalised over top-k).

    The pages do not name the gate function; the workload description fixes
    "fp32 softmax gating weights renormalised over top-k".  Softmax over the
    selected logits equals the full softmax renormalised over the selected set.
    Computed here in float64 with the usual max shift.
    """
    L = np.asarray(logits, np.float64)
    sel = np.take_along_axis(L, topk_idx.astype(np.int64), axis=1)
    m = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - m)
    return ex / ex.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------
# experts
# ----------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g * sigmoid(g) = g / (1 + exp(-g)), float64."""
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_hidden(x_rows: np.ndarray, w13: np.ndarray, F: int, round_h: bool = True) -> np.ndarray:
    """The first half of one SwiGLU expert on a block of rows, float64.

    w13 is [2F, H]: rows 0..F-1 the gate projection, rows F..2F-1 the up
    projection.  g = x Wg^T, u = x Wu^T, h = silu(g) * u.  The hidden activation
    h is the bf16 input of the down projection, so it is rounded to bf16
    (nearest-even) when round_h.
    """
    x_rows = np.asarray(x_rows, np.float64)
    w13 = np.asarray(w13, np.float64)
    g = x_rows @ w13[:F].T
    u = x_rows @ w13[F:2 * F].T
    h = silu(g) * u
    return round_to_bf16(h) if round_h else h


def down_projection(h_rows: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """The second half of one SwiGLU expert: y = h W2^T with w2 [H, F], float64."""
    return np.asarray(h_rows, np.float64) @ np.asarray(w2, np.float64).T


def swiglu_expert(x_rows: np.ndarray, w13: np.ndarray, w2: np.ndarray, F: int,
                  round_h: bool = True) -> np.ndarray:
    """One SwiGLU expert on a block of rows, float64: the down projection of the
    (bf16-rounded when round_h) hidden activation,
        g = x Wg^T,  u = x Wu^T,  h = silu(g) * u,  y = h W2^T.
    The two halves are separate functions so that a test can feed either one
    the GPU path's own intermediate and compare one stage at a time.
    """
    return down_projection(swiglu_hidden(x_rows, w13, F, round_h), w2)


def expert_outputs(x, topk_idx, w13, w2, F, round_h=True, expert_weights=None):
    """y[t, j, :] = expert_{idx[t,j]}(x[t]) for every token and slot, float64.

    ``w13``/``w2`` may be float64 arrays [E, 2F, H] / [E, H, F] or a callable
    ``expert_weights(e) -> (w13_e, w2_e)`` so large configurations can feed one
    expert at a time.
    """
    x = np.asarray(x, np.float64)
    T, k = topk_idx.shape
    H = x.shape[1]
    y = np.zeros((T, k, H), np.float64)
    for e in np.unique(topk_idx):
        tok, slot = np.nonzero(topk_idx == e)
        if expert_weights is not None:
            w13_e, w2_e = expert_weights(int(e))
        else:
            w13_e, w2_e = w13[e], w2[e]
        y[tok, slot] = swiglu_expert(x[tok], w13_e, w2_e, F, round_h)
    return y


def combine(y_slots: np.ndarray, gates: np.ndarray, y_shared=None) -> np.ndarray:
    """out[t] = sum_j gates[t, j] * y[t, j] (+ shared-expert output), float64.

    The combine page finding is that precision and order of this weighted sum
    must match across paths; in float64 the order of the k terms does not
    matter at the tolerance the GPU path is held to, so the oracle takes the
    slots in rank order j = 0..k-1 and adds the shared expert last, as the GPU
    path does.
    """
    out = np.zeros(y_slots.shape[0::2], np.float64)
    for j in range(y_slots.shape[1]):
        out += gates[:, j:j + 1] * y_slots[:, j]
    if y_shared is not None:
        out += y_shared
    return out


def moe_forward(x, w_router, w13, w2, k, F, ws13=None, ws2=None, F_shared=0,
                round_h=True, expert_weights=None, logits=None, replay_idx=None):
    """Whole MoE layer, float64: router -> top-k -> gates -> experts -> combine.

    ``logits`` may be supplied (for example float32 logits produced elsewhere)
    to re-run only the selection and what follows on them.  ``replay_idx``
    [T, k] replaces the selection by recorded expert choices (router replay,
    "Reinforcement Learning: Why Numerical Alignment and MoE Routing Matter So
    Much", section "MoE 路由会放大这种不匹配"); the gates are then the softmax
    of the logits of the given experts.
    Returns a dict with logits, idx, gates, y (per slot), y_shared, out.
    """
    x = np.asarray(x, np.float64)
    if logits is None:
        logits = router_logits(x, w_router)
    idx = topk_lowest_index(logits, k) if replay_idx is None else np.asarray(replay_idx, np.int32)
    gates = topk_gates(logits, idx)
    y = expert_outputs(x, idx, w13, w2, F, round_h, expert_weights)
    ys = None
    if F_shared:
        ys = swiglu_expert(x, ws13, ws2, F_shared, round_h)
    out = combine(y, gates, ys)
    return dict(logits=logits, idx=idx, gates=gates, y=y, y_shared=ys, out=out)


def dense_all_experts_then_mask(x, w_router, w13, w2, k, F, round_h=True):
    """Brute force: run every expert on every token, then keep the top-k.

    out[t] = sum_e 1[e in topk(t)] * gate_e(t) * expert_e(x[t]).
    Independent of the permutation / dispatch bookkeeping of ``moe_forward``;
    the two must agree to float64 rounding.
    """
    x = np.asarray(x, np.float64)
    E = w13.shape[0]
    L = router_logits(x, w_router)
    idx = topk_lowest_index(L, k)
    gates = topk_gates(L, idx)
    T = x.shape[0]
    gate_full = np.zeros((T, E), np.float64)
    for j in range(k):
        gate_full[np.arange(T), idx[:, j]] = gates[:, j]
    out = np.zeros_like(x)
    for e in range(E):
        ye = swiglu_expert(x, w13[e], w2[e], F, round_h)
        out += (gate_full[:, e] != 0)[:, None] * gate_full[:, e:e + 1] * ye
    return out


# ----------------------------------------------------------------------------
# dispatch plan (permutation) -- checked as invariants, not recomputed by value
# ----------------------------------------------------------------------------

def dispatch_plan(topk_idx: np.ndarray, E: int):
    """Expert-major permutation of the (token, slot) pairs, float-free.

    Rows of expert e occupy [offsets[e], offsets[e+1]); inside an expert the
    rows follow ascending token index (a stable counting sort).  Returns
    counts[E], offsets[E+1], row_token[S], slot_row[T, k] (all int64).
    Implied by the bit-agreement page's "per-expert token count" and its call
    for one fixed expert-matmul kernel whatever that count.
    """
    idx = np.asarray(topk_idx, np.int64)
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    row_token = np.empty(T * k, np.int64)
    slot_row = np.empty((T, k), np.int64)
    fill = offsets[:-1].copy()
    for t in range(T):                      # ascending token order
        for j in range(k):
            e = idx[t, j]
            row_token[fill[e]] = t
            slot_row[t, j] = fill[e]
            fill[e] += 1
    return counts, offsets, row_token, slot_row


# ----------------------------------------------------------------------------
# backward (the trainer's side of the same definition)
# ----------------------------------------------------------------------------

def _sigmoid(g):
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def swiglu_backward(x_rows, w13, w2, F, dy, round_ops=True):
    """Backward of one SwiGLU expert on a block of rows, float64.

    Forward: g = x Wg^T, u = x Wu^T, h = silu(g) * u, y = h W2^T.  With the
    upstream gradient dy of y:
        dh = dy W2;  dg = dh * u * silu'(g);  du = dh * silu(g),
        silu'(g) = s (1 + g (1 - s)),  s = sigmoid(g);
        dx = [dg, du] W13;  dW2 = dy^T h;  dW13 = [dg, du]^T x.
    The forward's bf16 rounding of h is a quantisation of the forward
    numerics, not part of the function being differentiated: its gradient is
    taken as the identity.  When round_ops, the bf16 operands of the gradient
    products are rounded as the forward rounds h: dy is taken as given (already
    bf16), h is the forward's rounded h, and [dg, du] is rounded to bf16.
    Returns dict(dh, dgu, h, dx, dw13, dw2).
    """
    x_rows = np.asarray(x_rows, np.float64)
    w13 = np.asarray(w13, np.float64)
    w2 = np.asarray(w2, np.float64)
    dy = np.asarray(dy, np.float64)
    g = x_rows @ w13[:F].T
    u = x_rows @ w13[F:2 * F].T
    s = _sigmoid(g)
    si = silu(g)
    h = si * u
    if round_ops:
        h = round_to_bf16(h)
    dh = dy @ w2
    dg = dh * u * (s * (1.0 + g * (1.0 - s)))
    du = dh * si
    dgu = np.concatenate([dg, du], axis=1)
    if round_ops:
        dgu = round_to_bf16(dgu)
    return dict(dh=dh, dgu=dgu, h=h, dx=dgu @ w13, dw13=dgu.T @ x_rows, dw2=dy.T @ h)


def moe_backward(x, w_router, w13, w2, k, F, dout, ws13=None, ws2=None, F_shared=0, round_ops=True,
                 expert_weights=None, replay_idx=None):
    """Gradients of L = sum(dout * out) through the whole MoE layer, float64.

    Forward as ``moe_forward`` (round_h = round_ops).  Backward, per token t and
    slot j with expert e = idx[t, j], gate w_j and expert output y_j:
        dgate_j = <dout_t, y_j>;  dy_j = w_j * dout_t  (bf16 operand when round_ops)
        expert e: ``swiglu_backward`` on its rows;  dx_t += sum_j dx_j
        router: the selected logits s = L[t, idx_t] give w = softmax(s), so
            ds_j = w_j (dgate_j - sum_i w_i dgate_i),  dL[t, idx_tj] = ds_j,
            0 for the experts not selected (the selection is piecewise
            constant); dx_t += dL_t Wr;  dWr = dL^T x  (dL a bf16 operand when round_ops)
        shared expert: ``swiglu_backward`` with dy = dout (bf16 operand when round_ops).
    ``expert_weights(e) -> (w13_e, w2_e)`` may replace w13 / w2 for large
    configurations; dw13 / dw2 are then dicts over the experts the batch used.
    ``replay_idx`` [T, k] takes the recorded expert choices instead of the top-k
    (as in ``moe_forward``); the router gradient is then the softmax Jacobian over
    the replayed experts' logits.
    Returns dict(dx, dw_router, dw13, dw2, dws13, dws2, dgate, dlogits, dy, dgu, dxp, fwd).
    """
    x = np.asarray(x, np.float64)
    dout = np.asarray(dout, np.float64)
    fwd = moe_forward(x, w_router, w13, w2, k, F, ws13, ws2, F_shared, round_h=round_ops,
                      expert_weights=expert_weights, replay_idx=replay_idx)
    idx, gates, y = fwd["idx"], fwd["gates"], fwd["y"]
    T, H = x.shape
    E = np.asarray(w_router).shape[0]
    rnd = round_to_bf16 if round_ops else (lambda a: a)
    dgate = np.einsum("th,tjh->tj", dout, y)
    dy = rnd(gates[:, :, None] * dout[:, None, :])              # [T, k, H]
    dx = np.zeros((T, H))
    dxp = np.zeros((T, k, H))
    dgu = np.zeros((T, k, 2 * F))
    if expert_weights is None:
        dw13 = np.zeros(np.asarray(w13).shape)
        dw2 = np.zeros(np.asarray(w2).shape)
    else:
        dw13, dw2 = {}, {}
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        w13_e, w2_e = (w13[e], w2[e]) if expert_weights is None else expert_weights(e)
        b = swiglu_backward(x[tok], w13_e, w2_e, F, dy[tok, slot], round_ops)
        dxp[tok, slot] = b["dx"]
        dgu[tok, slot] = b["dgu"]
        dw13[e] = b["dw13"]
        dw2[e] = b["dw2"]
    for j in range(k):
        dx += dxp[:, j]
    ds = gates * (dgate - (gates * dgate).sum(axis=1, keepdims=True))
    dlog = np.zeros((T, E))
    np.put_along_axis(dlog, idx.astype(np.int64), ds, axis=1)
    dlog = rnd(dlog)
    wr = np.asarray(w_router, np.float64)
    dx_router = dlog @ wr
    dw_router = dlog.T @ x
    dws13 = dws2 = dx_shared = None
    if F_shared:
        bs = swiglu_backward(x, ws13, ws2, F_shared, rnd(dout), round_ops)
        dx_shared, dws13, dws2 = bs["dx"], bs["dw13"], bs["dw2"]
        dx = dx + dx_shared
    dx = dx + dx_router
    return dict(dx=dx, dw_router=dw_router, dw13=dw13, dw2=dw2, dws13=dws13, dws2=dws2, dgate=dgate,
                dlogits=dlog, dy=dy, dgu=dgu, dxp=dxp, dx_router=dx_router, dx_shared=dx_shared, fwd=fwd)
