"""Prefill and decode entry points over the C ABI.

Both entry points run the same three library calls (moe_route_topk,
moe_grouped_ffn, moe_combine) with the same kernels and tile shapes; they differ
only on the host side.  Prefill takes any number of tokens in one call; decode
serves one token per request from buffers allocated once for a maximum batch.
Because every reduction in the library is per token with a fixed order, a
token's output bits do not depend on which entry point served it or on what
else was in its batch ("位级一致：前沿训练的差异化关键", section "端到端零 KLD":
the serving engine and the trainer must produce the same numbers whatever the
batch size or concurrent load).
"""
from dataclasses import dataclass
from typing import Optional

import torch

from . import binding


@dataclass
class MoEWeights:
    w_router: torch.Tensor            # [E, H] bf16
    w13: torch.Tensor                 # [E, 2F, H] bf16 (gate rows, then up rows)
    w2: torch.Tensor                  # [E, H, F] bf16
    k: int
    ws13: Optional[torch.Tensor] = None   # [2Fs, H] bf16 shared expert
    ws2: Optional[torch.Tensor] = None    # [H, Fs] bf16

    @property
    def E(self):
        return self.w13.shape[0]

    @property
    def H(self):
        return self.w13.shape[2]

    @property
    def F(self):
        return self.w13.shape[1] // 2

    @property
    def F_shared(self):
        return 0 if self.ws13 is None else self.ws13.shape[0] // 2


class MoELayer:
    """Batch-invariant MoE layer forward on one GPU."""

    def __init__(self, weights: MoEWeights):
        self.w = weights
        self._ws = None
        self._decode = None

    def _workspace(self, T):
        w = self.w
        need = binding.workspace_size(T, w.H, w.E, w.k, w.F, w.F_shared, 0)
        if self._ws is None or self._ws.numel() < need:
            self._ws = binding.new_workspace(need, device=w.w13.device)
        return self._ws

    def _run(self, x, ws, bufs=None, out_bf16=None, replay_idx=None):
        w = self.w
        T = x.shape[0]
        bufs = bufs or {}
        if replay_idx is None:
            # route, experts and combine in one library call
            return binding.moe_layer_forward(x, w.w_router, w.w13, w.w2, w.k, ws, ws13=w.ws13, ws2=w.ws2,
                                             logits=bufs.get("logits"), topk_idx=bufs.get("idx"), topk_w=bufs.get("w"),
                                             plan=bufs.get("plan"), xp=bufs.get("xp"), h=bufs.get("h"),
                                             y=bufs.get("y"), y_shared=bufs.get("ys"), out=bufs.get("out"),
                                             out_bf16=out_bf16)
        r = binding.moe_route_replay(x, w.w_router, replay_idx, ws, logits=bufs.get("logits"),
                                     topk_w=bufs.get("w"), plan=bufs.get("plan"), xp=bufs.get("xp"))
        f = binding.moe_grouped_ffn(r["xp"], r["plan"], w.w13, w.w2, T, w.k, ws, h=bufs.get("h"), y=bufs.get("y"),
                                    x_shared=x if w.ws13 is not None else None, ws13=w.ws13, ws2=w.ws2,
                                    y_shared=bufs.get("ys"))
        out = binding.moe_combine(f["y"], r["topk_w"], r["plan"], T, w.H, w.E, w.k, y_shared=f["y_shared"],
                                  out=bufs.get("out"), out_bf16=out_bf16)
        return dict(out=out, **r, **f)

    def prefill(self, x: torch.Tensor, out_bf16: Optional[torch.Tensor] = None, return_all=False,
                replay_idx: Optional[torch.Tensor] = None):
        """x [T, H] bf16 -> out [T, H] fp32 (optionally also a bf16 copy).  With replay_idx [T, k]
        int32 the recorded expert choices are used instead of the router's own top-k.

        A small batch (at most 1024 tokens) whose intermediates are not returned runs on the
        layer's preallocated decode buffers (only `out` is allocated per call): for such batches
        the host's allocations, not the kernels, set the call's latency."""
        T = x.shape[0]
        if not return_all and replay_idx is None and 0 < T <= 1024:
            if self._decode is None or self._decode["B"] < T:
                self.alloc_decode(max(T, 1))
            d = self._decode
            bufs = {k: d[k] for k in ("logits", "idx", "w", "plan", "xp", "h", "y", "ys")}
            return self._run(x, d["ws"], bufs, out_bf16=out_bf16)["out"]
        res = self._run(x, self._workspace(T), out_bf16=out_bf16, replay_idx=replay_idx)
        return res if return_all else res["out"]

    def backward(self, x: torch.Tensor, fwd: dict, dout: torch.Tensor, weight_grads: bool = True):
        """Backward of the layer for one batch, after ``prefill(x, return_all=True)`` returned ``fwd``.

        dout [T, H] fp32 -> dict(dx [T, H], dw_router, dw13, dw2, dws13, dws2) (fp32), computed by the
        library's combine, grouped-FFN and router backward calls (every reduction in a fixed order,
        no atomics)."""
        w = self.w
        T = x.shape[0]
        need = binding.backward_workspace_size(T, w.H, w.E, w.k, w.F, w.F_shared)
        if getattr(self, "_bws", None) is None or self._bws.numel() < need:
            self._bws = binding.new_workspace(need, device=x.device)
        ws = self._bws
        c = binding.moe_combine_backward(dout, fwd["y"], fwd["topk_w"], fwd["plan"], w.E, w.k,
                                         dout_bf16=w.ws13 is not None)
        f = binding.moe_grouped_ffn_backward(fwd["xp"], fwd["plan"], w.w13, w.w2, c["dy"], T, w.k, ws,
                                             dw13=weight_grads, dw2=weight_grads,
                                             x_shared=x if w.ws13 is not None else None, ws13=w.ws13, ws2=w.ws2,
                                             dout_bf16=c["dout_bf16"], dws13=weight_grads, dws2=weight_grads)
        r = binding.moe_route_backward(x, w.w_router, fwd["topk_idx"], fwd["topk_w"], c["dgate"], f["dxp"],
                                       fwd["plan"], ws, dx_shared=f["dx_shared"], dw_router=weight_grads)
        binding.check_status(ws)
        return dict(dx=r["dx"], dw_router=r["dw_router"], dw13=f["dw13"], dw2=f["dw2"], dws13=f["dws13"],
                    dws2=f["dws2"], dgate=c["dgate"], dy=c["dy"], dxp=f["dxp"], workspace=ws)

    def alloc_decode(self, max_batch: int):
        """Preallocate decode buffers for up to ``max_batch`` concurrent requests."""
        w = self.w
        B, dev = max_batch, w.w13.device
        S = B * w.k
        self._decode = dict(
            B=B,
            logits=torch.empty((B, w.E), dtype=torch.float32, device=dev),
            idx=torch.empty((B, w.k), dtype=torch.int32, device=dev),
            w=torch.empty((B, w.k), dtype=torch.float32, device=dev),
            plan=torch.empty(binding.plan_len(B, w.E, w.k), dtype=torch.int32, device=dev),
            xp=torch.empty((S, w.H), dtype=torch.bfloat16, device=dev),
            h=torch.empty((S, w.F), dtype=torch.bfloat16, device=dev),
            y=torch.empty((S, w.H), dtype=torch.float32, device=dev),
            ys=torch.empty((B, w.H), dtype=torch.float32, device=dev) if w.ws13 is not None else None,
            out=torch.empty((B, w.H), dtype=torch.float32, device=dev),
            ws=binding.new_workspace(binding.workspace_size(B, w.H, w.E, w.k, w.F, w.F_shared, 0), dev),
        )
        d = self._decode
        d["device"] = torch.device(dev)
        p = lambda t: None if t is None else t.data_ptr()   # noqa: E731
        # moe_layer_forward's arguments; decode() fills in x (0), B (6), out_bf16 (21) and the stream (24)
        d["args"] = [None, p(w.w_router), p(w.w13), p(w.w2), p(w.ws13), p(w.ws2), B, w.H, w.E, w.k, w.F, w.F_shared,
                     p(d["logits"]), p(d["idx"]), p(d["w"]), p(d["plan"]), p(d["xp"]), p(d["h"]), p(d["y"]),
                     p(d["ys"]), p(d["out"]), None, p(d["ws"]), d["ws"].numel(), None]
        d["fn"] = binding.lib().moe_layer_forward

    def decode(self, x_tokens: torch.Tensor, out_bf16: Optional[torch.Tensor] = None) -> torch.Tensor:
        """One token per request: x_tokens [B, H] bf16 -> [B, H] fp32 (a view of the decode buffer);
        out_bf16 [B, H] (optional) receives the bf16 copy the head reads.

        One library call (moe_layer_forward) on buffers allocated once: the argument list is built in
        alloc_decode (every buffer's batch-B view starts at the same address), so a call checks the
        token tensor, sets its pointer, the batch size and the stream, and enters the library."""
        B = x_tokens.shape[0]
        if self._decode is None or self._decode["B"] < B:
            self.alloc_decode(max(B, 1))
        d = self._decode
        w = self.w
        if (x_tokens.dtype != torch.bfloat16 or x_tokens.device != d["device"] or not x_tokens.is_contiguous()
                or x_tokens.dim() != 2 or x_tokens.shape[1] != w.H):
            raise ValueError(f"x_tokens must be a contiguous [B, {w.H}] bf16 tensor on {d['device']}")
        if out_bf16 is not None:
            binding._req(out_bf16, torch.bfloat16, "out_bf16", (B, w.H))
        args = d["args"]
        args[0] = x_tokens.data_ptr()
        args[6] = B
        args[21] = None if out_bf16 is None else out_bf16.data_ptr()
        args[24] = torch.cuda.current_stream(d["device"]).cuda_stream
        binding.check(d["fn"](*args))
        return d["out"][:B]


class InputStager:
    """Double-buffered host-to-device staging of a step's inputs on a side stream.

    ``stage(host)`` issues the copies of the next batch (pinned host tensors) into
    the buffer the step before last has finished with; ``next()`` makes the
    current stream wait for the oldest staged batch and returns its device
    buffers; ``release()`` marks that batch's buffers free once the work enqueued
    so far on the current stream is done.  Staging batch i+1 before running
    batch i overlaps its copies with batch i's kernels.
    """

    def __init__(self, like: dict):
        dev = next(iter(like.values())).device
        self.bufs = [{k: torch.empty_like(v) for k, v in like.items()} for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]
        self.fill = 0
        self.cur = 0

    def stage(self, host: dict):
        b = self.fill
        s = self.copy_stream
        if self.used[b]:
            s.wait_event(self.free[b])
        with torch.cuda.stream(s):
            for k, v in host.items():
                self.bufs[b][k].copy_(v, non_blocking=True)
            self.ready[b].record(s)
        self.fill ^= 1

    def next(self) -> dict:
        b = self.cur
        torch.cuda.current_stream().wait_event(self.ready[b])
        return self.bufs[b]

    def release(self):
        b = self.cur
        self.free[b].record(torch.cuda.current_stream())
        self.used[b] = True
        self.cur ^= 1


class DecodeGraphs:
    """Decode steps captured as CUDA graphs, one per batch-size bucket.

    Every kernel of the decode path takes its sizes and buffers at capture time,
    so a step for a bucket of B requests replays as one graph launch; batches
    smaller than a bucket are padded with zero tokens, which changes no other
    row's bits (every row is computed on its own).  The captured kernels are the
    same as the eager ones, so a replayed step gives the same bits as
    MoELayer.decode on the same tokens.
    """

    def __init__(self, layer: MoELayer, buckets=(1, 2, 4, 8, 16, 32, 64, 128)):
        self.layer = layer
        self.buckets = sorted(buckets)
        w = layer.w
        dev = w.w13.device
        layer.alloc_decode(self.buckets[-1])
        self.inp = {B: torch.zeros((B, w.H), dtype=torch.bfloat16, device=dev) for B in self.buckets}
        self.out = {}
        self.graphs = {}
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for B in self.buckets:
                layer.decode(self.inp[B])          # warm-up outside capture (kernel attributes, caches)
        torch.cuda.current_stream(dev).wait_stream(side)
        for B in self.buckets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.out[B] = layer.decode(self.inp[B])
            self.graphs[B] = g

    def __call__(self, x_tokens: torch.Tensor) -> torch.Tensor:
        """x_tokens [b, H] bf16 (b <= largest bucket) -> [b, H] fp32 (a view of the graph's output)."""
        b = x_tokens.shape[0]
        B = next(B for B in self.buckets if B >= b)
        self.inp[B][:b].copy_(x_tokens)
        if b < B:
            self.inp[B][b:].zero_()
        self.graphs[B].replay()
        return self.out[B][:b]


def moe_prefill(layer: MoELayer, x: torch.Tensor) -> torch.Tensor:
    return layer.prefill(x)


def moe_decode(layer: MoELayer, x_tokens: torch.Tensor) -> torch.Tensor:
    return layer.decode(x_tokens)


def head_logprob_kl(hidden, w_vocab, target, rollout_logp=None, beta=2.0, workspace=None, logits=None,
                    write_logits=False):
    """Token logprobs of the exact target ids, and (with rollout logprobs) k3 and the IcePop mask."""
    T, H = hidden.shape
    V = w_vocab.shape[0]
    if workspace is None:
        workspace = binding.new_workspace(binding.workspace_size(T, H, V=V), hidden.device)
    return binding.lm_logprob_kl(hidden, w_vocab, target, workspace, rollout_logp=rollout_logp, beta=beta,
                                 logits=logits, write_logits=write_logits)
