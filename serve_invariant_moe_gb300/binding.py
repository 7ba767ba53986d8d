"""Python binding of the C ABI: argument marshalling only.

Each function checks dtypes/devices/contiguity, allocates missing outputs with
torch (device memory only), passes raw pointers and the current CUDA stream to
libinvmoe.so and raises on a non-zero status.  No arithmetic of the hot path
happens here: every step runs in the library's kernels.
"""
import ctypes
import math

import torch

from ._lib import check, lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _req(t, dtype, name, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    # the library launches on the current device: a pointer into another GPU's memory
    # must not reach a kernel
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current CUDA device is cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _opt(t, dtype, name, shape=None):
    """_req for an optional tensor (None passes)."""
    return None if t is None else _req(t, dtype, name, shape)


def _req_plan(plan, T, E, k):
    _req(plan, torch.int32, "plan")
    if plan.numel() < plan_len(T, E, k):
        raise ValueError("plan is too small")
    return plan


def plan_len(T, E, k) -> int:
    return int(lib().invmoe_plan_len(T, E, k))


def workspace_size(T, H, E=0, k=0, F=0, F_shared=0, V=0) -> int:
    return int(lib().invmoe_workspace_size(T, H, E, k, F, F_shared, V))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-filled device workspace (the first 256 bytes are the status word)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def check_status(workspace: torch.Tensor):
    """Synchronise the current stream and raise if a kernel's bounded wait ran out."""
    check(lib().invmoe_check(_p(workspace), _stream()))


def moe_route_topk(x, w_router, k, workspace, logits=None, topk_idx=None, topk_w=None, plan=None, xp=None):
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    _req(x, torch.bfloat16, "x")
    _req(w_router, torch.bfloat16, "w_router", (E, H))
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if logits is None else logits
    topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_w = torch.empty((T, k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    plan = torch.empty(plan_len(T, E, k), dtype=torch.int32, device=dev) if plan is None else plan
    xp = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev) if xp is None else xp
    _req(logits, torch.float32, "logits", (T, E))
    _req(topk_idx, torch.int32, "topk_idx", (T, k))
    _req(topk_w, torch.float32, "topk_w", (T, k))
    _req(plan, torch.int32, "plan")
    if plan.numel() < plan_len(T, E, k):
        raise ValueError("plan is too small")
    _req(xp, torch.bfloat16, "xp")
    if xp.numel() < T * k * H:
        raise ValueError("xp is too small")
    _req(workspace, torch.uint8, "workspace")
    check(lib().moe_route_topk(_p(x), _p(w_router), T, H, E, k, _p(logits), _p(topk_idx), _p(topk_w), _p(plan),
                               _p(xp), _p(workspace), workspace.numel(), _stream()))
    return dict(logits=logits, topk_idx=topk_idx, topk_w=topk_w, plan=plan, xp=xp)


def moe_route_replay(x, w_router, topk_idx, workspace, logits=None, topk_w=None, plan=None, xp=None):
    """Router replay: the given experts [T, k] int32, fresh gates, plan and permuted rows."""
    T, H = x.shape
    E = w_router.shape[0]
    k = topk_idx.shape[1]
    dev = x.device
    _req(x, torch.bfloat16, "x")
    _req(w_router, torch.bfloat16, "w_router", (E, H))
    _req(topk_idx, torch.int32, "topk_idx", (T, k))
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if logits is None else logits
    topk_w = torch.empty((T, k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    plan = torch.empty(plan_len(T, E, k), dtype=torch.int32, device=dev) if plan is None else plan
    xp = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev) if xp is None else xp
    _req(logits, torch.float32, "logits", (T, E))
    _req(topk_w, torch.float32, "topk_w", (T, k))
    _req(plan, torch.int32, "plan")
    _req(xp, torch.bfloat16, "xp")
    if plan.numel() < plan_len(T, E, k) or xp.numel() < T * k * H:
        raise ValueError("plan / xp too small")
    _req(workspace, torch.uint8, "workspace")
    check(lib().moe_route_replay(_p(x), _p(w_router), _p(topk_idx), T, H, E, k, _p(logits), _p(topk_w), _p(plan),
                                 _p(xp), _p(workspace), workspace.numel(), _stream()))
    return dict(logits=logits, topk_idx=topk_idx, topk_w=topk_w, plan=plan, xp=xp)


def moe_grouped_ffn(xp, plan, w13, w2, T, k, workspace, h=None, y=None,
                    x_shared=None, ws13=None, ws2=None, y_shared=None):
    E, F2, H = w13.shape
    F = F2 // 2
    dev = xp.device
    S = T * k
    _req(xp, torch.bfloat16, "xp")
    _req(plan, torch.int32, "plan")
    _req(w13, torch.bfloat16, "w13")
    _req(w2, torch.bfloat16, "w2", (E, H, F))
    h = torch.empty((S, F), dtype=torch.bfloat16, device=dev) if h is None else h
    y = torch.empty((S, H), dtype=torch.float32, device=dev) if y is None else y
    _req(h, torch.bfloat16, "h")
    _req(y, torch.float32, "y")
    if h.numel() < S * F or y.numel() < S * H:
        raise ValueError("h / y too small")
    Fs = 0
    if ws13 is not None:
        Fs = ws13.shape[0] // 2
        _req(x_shared, torch.bfloat16, "x_shared", (T, H))
        _req(ws13, torch.bfloat16, "ws13", (2 * Fs, H))
        _req(ws2, torch.bfloat16, "ws2", (H, Fs))
        y_shared = torch.empty((T, H), dtype=torch.float32, device=dev) if y_shared is None else y_shared
        _req(y_shared, torch.float32, "y_shared", (T, H))
    _req(workspace, torch.uint8, "workspace")
    check(lib().moe_grouped_ffn(_p(xp), _p(plan), _p(w13), _p(w2), T, H, E, k, F, _p(h), _p(y),
                                _p(x_shared), _p(ws13), _p(ws2), Fs, _p(y_shared), _p(workspace),
                                workspace.numel(), _stream()))
    return dict(h=h, y=y, y_shared=y_shared)


def moe_layer_forward(x, w_router, w13, w2, k, workspace, ws13=None, ws2=None, logits=None, topk_idx=None, topk_w=None,
                      plan=None, xp=None, h=None, y=None, y_shared=None, out=None, out_bf16=None):
    """The whole layer in one library call (route, grouped SwiGLU experts, combine); missing outputs
    are allocated.  Returns the same dict as the three calls."""
    T, H = x.shape
    E, F2, _ = w13.shape
    F = F2 // 2
    Fs = 0 if ws13 is None else ws13.shape[0] // 2
    S = T * k
    dev = x.device
    _req(x, torch.bfloat16, "x")
    _req(w_router, torch.bfloat16, "w_router", (E, H))
    _req(w13, torch.bfloat16, "w13", (E, 2 * F, H))
    _req(w2, torch.bfloat16, "w2", (E, H, F))

    def buf(t, shape, dtype, name, min_numel=None):
        t = torch.empty(shape, dtype=dtype, device=dev) if t is None else t
        _req(t, dtype, name)
        if t.numel() < (min_numel if min_numel is not None else math.prod(shape)):
            raise ValueError(f"{name} is too small")
        return t
    logits = buf(logits, (T, E), torch.float32, "logits")
    topk_idx = buf(topk_idx, (T, k), torch.int32, "topk_idx")
    topk_w = buf(topk_w, (T, k), torch.float32, "topk_w")
    plan = buf(plan, (plan_len(T, E, k),), torch.int32, "plan")
    xp = buf(xp, (S, H), torch.bfloat16, "xp")
    h = buf(h, (S, F), torch.bfloat16, "h")
    y = buf(y, (S, H), torch.float32, "y")
    out = buf(out, (T, H), torch.float32, "out")
    if Fs:
        _req(ws13, torch.bfloat16, "ws13", (2 * Fs, H))
        _req(ws2, torch.bfloat16, "ws2", (H, Fs))
        y_shared = buf(y_shared, (T, H), torch.float32, "y_shared")
    else:
        y_shared = None
    _opt(out_bf16, torch.bfloat16, "out_bf16", (T, H))
    _req(workspace, torch.uint8, "workspace")
    check(lib().moe_layer_forward(_p(x), _p(w_router), _p(w13), _p(w2), _p(ws13), _p(ws2), T, H, E, k, F, Fs,
                                  _p(logits), _p(topk_idx), _p(topk_w), _p(plan), _p(xp), _p(h), _p(y), _p(y_shared),
                                  _p(out), _p(out_bf16), _p(workspace), workspace.numel(), _stream()))
    return dict(out=out, logits=logits, topk_idx=topk_idx, topk_w=topk_w, plan=plan, xp=xp, h=h, y=y,
                y_shared=y_shared)


def moe_combine(y, topk_w, plan, T, H, E, k, y_shared=None, out=None, out_bf16=None):
    dev = y.device
    _req(y, torch.float32, "y")
    _req(topk_w, torch.float32, "topk_w", (T, k))
    _req(plan, torch.int32, "plan")
    if y_shared is not None:
        _req(y_shared, torch.float32, "y_shared", (T, H))
    out = torch.empty((T, H), dtype=torch.float32, device=dev) if out is None else out
    _req(out, torch.float32, "out", (T, H))
    if out_bf16 is not None:
        _req(out_bf16, torch.bfloat16, "out_bf16", (T, H))
    check(lib().moe_combine(_p(y), _p(topk_w), _p(plan), _p(y_shared), T, H, E, k, _p(out), _p(out_bf16),
                            _stream()))
    return out


def lm_logprob_kl(hidden, w_vocab, target, workspace, rollout_logp=None, beta=2.0, logits=None,
                  logp=None, lse=None, k3=None, mask=None, write_logits=False):
    """logits are written only if a buffer is passed or write_logits is set."""
    T, H = hidden.shape
    V = w_vocab.shape[0]
    dev = hidden.device
    _req(hidden, torch.bfloat16, "hidden")
    _req(w_vocab, torch.bfloat16, "w_vocab", (V, H))
    _req(target, torch.int32, "target", (T,))
    if logits is None and write_logits:
        logits = torch.empty((T, V), dtype=torch.float32, device=dev)
    if logits is not None:
        _req(logits, torch.float32, "logits", (T, V))
    logp = torch.empty(T, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(T, dtype=torch.float32, device=dev) if lse is None else lse
    if rollout_logp is not None:
        _req(rollout_logp, torch.float32, "rollout_logp", (T,))
        k3 = torch.empty(T, dtype=torch.float32, device=dev) if k3 is None else k3
        mask = torch.empty(T, dtype=torch.uint8, device=dev) if mask is None else mask
        _req(k3, torch.float32, "k3", (T,))
        _req(mask, torch.uint8, "mask", (T,))
    _req(logp, torch.float32, "logp", (T,))
    _req(lse, torch.float32, "lse", (T,))
    _req(workspace, torch.uint8, "workspace")
    check(lib().lm_logprob_kl(_p(hidden), _p(w_vocab), _p(target), _p(rollout_logp), T, H, V, float(beta),
                              _p(logits), _p(logp), _p(lse), _p(k3), _p(mask), _p(workspace), workspace.numel(),
                              _stream()))
    return dict(logits=logits, logp=logp, lse=lse, k3=k3, mask=mask)


def lm_logprob_partials(hidden, w_vocab_shard, target, V, v0, workspace, partials, tgt_logit, logits=None):
    """Pass 1 of the log-sum-exp on the vocabulary shard [v0, v0 + rows of w_vocab_shard).

    partials: fp32 [T, P, 2] (P >= the shard's chunk count), the shard's chunk j of token t at
    partials[t, j]; tgt_logit [T] fp32 receives z[t, target[t]] where the target is in the shard;
    logits (optional) is the whole [T, V] fp32 array, of which the shard's columns are written."""
    T, H = hidden.shape
    v1 = v0 + w_vocab_shard.shape[0]
    _req(hidden, torch.bfloat16, "hidden")
    _req(w_vocab_shard, torch.bfloat16, "w_vocab_shard", (v1 - v0, H))
    _req(target, torch.int32, "target", (T,))
    _req(partials, torch.float32, "partials")
    if partials.dim() != 3 or partials.shape[0] != T or partials.shape[2] != 2:
        raise ValueError(f"partials must be [T, P, 2], got {tuple(partials.shape)}")
    _req(tgt_logit, torch.float32, "tgt_logit", (T,))
    _opt(logits, torch.float32, "logits", (T, V))
    _req(workspace, torch.uint8, "workspace")
    check(lib().lm_logprob_partials(_p(hidden), _p(w_vocab_shard), _p(target), T, H, V, v0, v1, _p(logits),
                                    _p(partials), partials.shape[1], _p(tgt_logit), _p(workspace), workspace.numel(),
                                    _stream()))
    return partials


def lm_logprob_merge(partials, tgt_logit, target, V, rollout_logp=None, beta=2.0):
    """Pass 2 and the per-token outputs from partials [T, NCH, 2] with target logits [T] (one array),
    or from partials [n, T, P, 2] with target logits [n, T] (n gathered shards of P chunks each)."""
    _req(partials, torch.float32, "partials")
    if partials.dim() == 3:
        T, P = partials.shape[0], partials.shape[1]
        stride, tstride = 0, 0
        _req(tgt_logit, torch.float32, "tgt_logit", (T,))
    elif partials.dim() == 4:
        n, T, P = partials.shape[0], partials.shape[1], partials.shape[2]
        stride, tstride = T * P, T
        _req(tgt_logit, torch.float32, "tgt_logit", (n, T))
    else:
        raise ValueError("partials must be [T, NCH, 2] or [n, T, P, 2]")
    if partials.shape[-1] != 2:
        raise ValueError("partials must end in a (max, sum) pair")
    dev = partials.device
    _req(target, torch.int32, "target", (T,))
    out = dict(logp=torch.empty(T, dtype=torch.float32, device=dev),
               lse=torch.empty(T, dtype=torch.float32, device=dev), k3=None, mask=None)
    if rollout_logp is not None:
        _req(rollout_logp, torch.float32, "rollout_logp", (T,))
        out["k3"] = torch.empty(T, dtype=torch.float32, device=dev)
        out["mask"] = torch.empty(T, dtype=torch.uint8, device=dev)
    check(lib().lm_logprob_merge(_p(partials), P, P, stride, _p(tgt_logit), tstride, _p(target), _p(rollout_logp), T,
                                 V, float(beta), _p(out["logp"]), _p(out["lse"]), _p(out["k3"]), _p(out["mask"]),
                                 _stream()))
    return out


def moe_ep_regroup(recv_xp, recv_counts, workspace, xp_local=None, plan_local=None, row_src=None):
    """Received rows (source-major) -> expert-major rows, the local plan and the row map.

    recv_xp [R, H] bf16, recv_counts [n_src, E_local] int32 (device)."""
    R, H = recv_xp.shape
    n_src, E_local = recv_counts.shape
    dev = recv_xp.device
    _req(recv_xp, torch.bfloat16, "recv_xp")
    _req(recv_counts, torch.int32, "recv_counts")
    xp_local = torch.empty((R, H), dtype=torch.bfloat16, device=dev) if xp_local is None else xp_local
    plan_local = torch.empty(2 * E_local + 1, dtype=torch.int32, device=dev) if plan_local is None else plan_local
    row_src = torch.empty(max(R, 1), dtype=torch.int32, device=dev) if row_src is None else row_src
    _req(xp_local, torch.bfloat16, "xp_local", (R, H))
    _req(plan_local, torch.int32, "plan_local", (2 * E_local + 1,))
    _req(row_src, torch.int32, "row_src")
    if row_src.numel() < R:
        raise ValueError("row_src is too small")
    _req(workspace, torch.uint8, "workspace")
    check(lib().moe_ep_regroup(_p(recv_xp), _p(recv_counts), n_src, E_local, R, H, _p(xp_local), _p(plan_local),
                               _p(row_src), _p(workspace), workspace.numel(), _stream()))
    return dict(xp_local=xp_local, plan_local=plan_local, row_src=row_src)


def moe_ep_ungroup(y_local, row_src, y_send=None):
    """y_send[row_src[i]] = y_local[i]: expert outputs back in the received order."""
    R, H = y_local.shape
    _req(y_local, torch.float32, "y_local")
    _req(row_src, torch.int32, "row_src")
    y_send = torch.empty_like(y_local) if y_send is None else y_send
    _req(y_send, torch.float32, "y_send", (R, H))
    check(lib().moe_ep_ungroup(_p(y_local), _p(row_src), R, H, _p(y_send), _stream()))
    return y_send


def moe_shared_expert(x, ws13, ws2, workspace, y_shared=None):
    """The shared expert alone: y_shared [T, H] fp32 = SwiGLU(x)."""
    T, H = x.shape
    Fs = ws13.shape[0] // 2
    _req(x, torch.bfloat16, "x")
    _req(ws13, torch.bfloat16, "ws13", (2 * Fs, H))
    _req(ws2, torch.bfloat16, "ws2", (H, Fs))
    y_shared = torch.empty((T, H), dtype=torch.float32, device=x.device) if y_shared is None else y_shared
    _req(y_shared, torch.float32, "y_shared", (T, H))
    _req(workspace, torch.uint8, "workspace")
    check(lib().moe_shared_expert(_p(x), _p(ws13), _p(ws2), T, H, Fs, _p(y_shared), _p(workspace), workspace.numel(),
                                  _stream()))
    return y_shared


def rl_token_loss(logp_train, logp_rollout, advantage, logp_old=None, beta=2.0, eps_low=0.2, eps_high=0.28):
    """IcePop-masked clipped policy loss per token (+ fixed-order mean), IcePop mask, DIS weights."""
    T = logp_train.shape[0]
    dev = logp_train.device
    for name, t in (("logp_train", logp_train), ("logp_rollout", logp_rollout), ("advantage", advantage)):
        _req(t, torch.float32, name, (T,))
    if logp_old is not None:
        _req(logp_old, torch.float32, "logp_old", (T,))
    out = dict(loss=torch.empty(T, dtype=torch.float32, device=dev),
               loss_mean=torch.empty(1, dtype=torch.float32, device=dev),
               icepop_mask=torch.empty(T, dtype=torch.uint8, device=dev),
               dis_weight=torch.empty(T, dtype=torch.float32, device=dev),
               grad_logp=torch.empty(T, dtype=torch.float32, device=dev))
    check(lib().rl_token_loss(_p(logp_train), _p(logp_old), _p(logp_rollout), _p(advantage), T, float(beta),
                              float(eps_low), float(eps_high), _p(out["icepop_mask"]), _p(out["dis_weight"]),
                              _p(out["loss"]), _p(out["loss_mean"]), _p(out["grad_logp"]), _stream()))
    return out


def lm_head_backward(hidden, w_vocab, target, lse, grad_logp, workspace, dlogits=None, d_hidden=True,
                     d_wvocab=True):
    """Head backward: dlogits [T, V] bf16, d_hidden [T, H] fp32, d_wvocab [V, H] fp32.

    d_hidden / d_wvocab: a tensor to write into, True to allocate one, False to skip it."""
    T, H = hidden.shape
    V = w_vocab.shape[0]
    dev = hidden.device
    _req(hidden, torch.bfloat16, "hidden")
    _req(w_vocab, torch.bfloat16, "w_vocab", (V, H))
    _req(target, torch.int32, "target", (T,))
    _req(lse, torch.float32, "lse", (T,))
    _req(grad_logp, torch.float32, "grad_logp", (T,))
    _req(workspace, torch.uint8, "workspace")
    dlogits = torch.empty((T, V), dtype=torch.bfloat16, device=dev) if dlogits is None else dlogits
    _req(dlogits, torch.bfloat16, "dlogits", (T, V))
    if d_hidden is True:
        d_hidden = torch.empty((T, H), dtype=torch.float32, device=dev)
    if d_wvocab is True:
        d_wvocab = torch.empty((V, H), dtype=torch.float32, device=dev)
    d_hidden = None if d_hidden is False else d_hidden
    d_wvocab = None if d_wvocab is False else d_wvocab
    if d_hidden is not None:
        _req(d_hidden, torch.float32, "d_hidden", (T, H))
    if d_wvocab is not None:
        _req(d_wvocab, torch.float32, "d_wvocab", (V, H))
    check(lib().lm_head_backward(_p(hidden), _p(w_vocab), _p(target), _p(lse), _p(grad_logp), T, H, V,
                                 _p(dlogits), _p(d_hidden), _p(d_wvocab), _p(workspace), workspace.numel(),
                                 _stream()))
    return dict(dlogits=dlogits, d_hidden=d_hidden, d_wvocab=d_wvocab)


def backward_workspace_size(T, H, E, k, F, F_shared=0) -> int:
    return int(lib().invmoe_backward_workspace_size(T, H, E, k, F, F_shared))


def moe_combine_backward(dout, y, topk_w, plan, E, k, dy=None, dgate=None, dout_bf16=False):
    """dy [T*k, H] bf16 (permuted rows), dgate [T, k] fp32, optionally dout_bf16 [T, H] bf16."""
    T, H = dout.shape
    dev = dout.device
    _req(dout, torch.float32, "dout")
    _req(y, torch.float32, "y", (T * k, H))
    _req(topk_w, torch.float32, "topk_w", (T, k))
    _req_plan(plan, T, E, k)
    dy = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev) if dy is None else dy
    dgate = torch.empty((T, k), dtype=torch.float32, device=dev) if dgate is None else dgate
    db = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if dout_bf16 is True else (dout_bf16 or None)
    _req(dy, torch.bfloat16, "dy", (T * k, H))
    _req(dgate, torch.float32, "dgate", (T, k))
    _opt(db, torch.bfloat16, "dout_bf16", (T, H))
    check(lib().moe_combine_backward(_p(dout), _p(y), _p(topk_w), _p(plan), T, H, E, k, _p(dy), _p(dgate), _p(db),
                                     _stream()))
    return dict(dy=dy, dgate=dgate, dout_bf16=db)


def moe_grouped_ffn_backward(xp, plan, w13, w2, dy, T, k, workspace, dxp=None, dw13=True, dw2=True,
                             x_shared=None, ws13=None, ws2=None, dout_bf16=None, dx_shared=None, dws13=True,
                             dws2=True):
    """dxp [T*k, H] fp32, dw13 [E, 2F, H], dw2 [E, H, F] (+ shared: dx_shared, dws13, dws2), all fp32.
    A weight-gradient argument may be a tensor, True (allocate) or False (skip)."""
    E, F2, H = w13.shape
    F = F2 // 2
    dev = xp.device
    S = T * k
    Fs = 0 if ws13 is None else ws13.shape[0] // 2
    _req(xp, torch.bfloat16, "xp", (S, H))
    _req(w13, torch.bfloat16, "w13")
    _req(w2, torch.bfloat16, "w2", (E, H, F))
    _req(dy, torch.bfloat16, "dy", (S, H))
    _req_plan(plan, T, E, k)
    _req(workspace, torch.uint8, "workspace")

    def alloc(v, shape):
        if v is True:
            return torch.empty(shape, dtype=torch.float32, device=dev)
        return None if v is False or v is None else v

    dxp = torch.empty((S, H), dtype=torch.float32, device=dev) if dxp is None else dxp
    dw13, dw2 = alloc(dw13, (E, 2 * F, H)), alloc(dw2, (E, H, F))
    _req(dxp, torch.float32, "dxp", (S, H))
    _opt(dw13, torch.float32, "dw13", (E, 2 * F, H))
    _opt(dw2, torch.float32, "dw2", (E, H, F))
    if Fs:
        _req(x_shared, torch.bfloat16, "x_shared", (T, H))
        _req(ws13, torch.bfloat16, "ws13", (2 * Fs, H))
        _req(ws2, torch.bfloat16, "ws2", (H, Fs))
        _req(dout_bf16, torch.bfloat16, "dout_bf16", (T, H))
        dx_shared = torch.empty((T, H), dtype=torch.float32, device=dev) if dx_shared is None else dx_shared
        dws13, dws2 = alloc(dws13, (2 * Fs, H)), alloc(dws2, (H, Fs))
        _req(dx_shared, torch.float32, "dx_shared", (T, H))
        _opt(dws13, torch.float32, "dws13", (2 * Fs, H))
        _opt(dws2, torch.float32, "dws2", (H, Fs))
    else:
        dx_shared = dws13 = dws2 = None
    check(lib().moe_grouped_ffn_backward(_p(xp), _p(plan), _p(w13), _p(w2), _p(dy), T, H, E, k, F, _p(dxp), _p(dw13),
                                         _p(dw2), _p(x_shared), _p(ws13), _p(ws2), _p(dout_bf16), Fs, _p(dx_shared),
                                         _p(dws13), _p(dws2), _p(workspace), workspace.numel(), _stream()))
    return dict(dxp=dxp, dw13=dw13, dw2=dw2, dx_shared=dx_shared, dws13=dws13, dws2=dws2)


def moe_route_backward(x, w_router, topk_idx, topk_w, dgate, dxp, plan, workspace, dx_shared=None, dx=None,
                       dw_router=True):
    """dx [T, H] fp32 (the layer input's gradient) and dw_router [E, H] fp32."""
    T, H = x.shape
    E = w_router.shape[0]
    k = topk_idx.shape[1]
    dev = x.device
    _req(x, torch.bfloat16, "x")
    _req(w_router, torch.bfloat16, "w_router", (E, H))
    _req(topk_idx, torch.int32, "topk_idx", (T, k))
    _req(topk_w, torch.float32, "topk_w", (T, k))
    _req(dgate, torch.float32, "dgate", (T, k))
    _req(dxp, torch.float32, "dxp", (T * k, H))
    _req_plan(plan, T, E, k)
    _opt(dx_shared, torch.float32, "dx_shared", (T, H))
    _req(workspace, torch.uint8, "workspace")
    dx = torch.empty((T, H), dtype=torch.float32, device=dev) if dx is None else dx
    if dw_router is True:
        dw_router = torch.empty((E, H), dtype=torch.float32, device=dev)
    dw_router = None if dw_router is False else dw_router
    _req(dx, torch.float32, "dx", (T, H))
    _opt(dw_router, torch.float32, "dw_router", (E, H))
    check(lib().moe_route_backward(_p(x), _p(w_router), _p(topk_idx), _p(topk_w), _p(dgate), _p(dxp), _p(plan),
                                   _p(dx_shared), T, H, E, k, _p(dx), _p(dw_router), _p(workspace),
                                   workspace.numel(), _stream()))
    return dict(dx=dx, dw_router=dw_router)


def gemm_bf16(a, b, workspace, variant=0, out=None):
    """Diagnostic: the dense tcgen05 GEMM engine alone, d = a @ b^T in fp32.

    variant 5 takes b as [K, N] (d = a @ b); variant 6 takes a as [K, M] and b as
    [K, N] (d = a^T @ b)."""
    v = int(variant) & 0xff
    if v == 6:
        K, M = a.shape
    else:
        M, K = a.shape
    N = b.shape[1] if v in (5, 6) else b.shape[0]
    _req(a, torch.bfloat16, "a")
    _req(b, torch.bfloat16, "b", (K, N) if v in (5, 6) else (N, K))
    out = torch.empty((M, N), dtype=torch.float32, device=a.device) if out is None else out
    _req(out, torch.float32, "out", (M, N))
    check(lib().invmoe_gemm_bf16(_p(a), _p(b), M, N, K, _p(out), int(variant), _p(workspace), workspace.numel(),
                                 _stream()))
    return out


def debug_timeout_probe(workspace, timeout_us=20000):
    check(lib().invmoe_debug_timeout_probe(_p(workspace), workspace.numel(), int(timeout_us), _stream()))
