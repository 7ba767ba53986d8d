"""Expert-parallel MoE layer and vocabulary-parallel head across ranks.

Both split one model over several devices and keep the bits of the one-device
path ("位级一致：前沿训练的差异化关键", section "为什么比特级一致是一个复杂的问题":
a cross-device reduction whose algorithm changes with the size of the job breaks
agreement; "GLM Post-Training Beyond SFT", section "动作与概率契约": the
vocabulary-parallel log-sum-exp needs comparison tests).  Neither adds a
reduction across devices:

* Expert parallelism (experts [e0, e1) on each rank): every rank routes its own
  tokens with the whole router, sends each owner the slice of its
  expert-sorted rows that the owner's experts need (an all-to-all of rows),
  the owner regroups them expert-major and runs its experts, and the output
  rows go back by the reverse all-to-all.  An expert output row depends on its
  own input row only, so it has the same bits on any rank; the weighted
  combine stays on the token's own rank in the fixed slot order.
* Vocabulary parallelism (vocabulary cut at 256-column chunk boundaries): each
  rank computes the first log-sum-exp pass for its own chunks, an all-gather
  brings every rank all chunks' (max, sum) pairs and target logits, and every
  rank folds the chunks in the one-device order.

This module only moves data: its collectives (all-to-all, all-gather) copy
bytes and combine nothing, and every arithmetic step runs in the library's
kernels through ``binding``.  ``Collectives`` runs them over torch.distributed
(NCCL between GPUs, gloo on the CPU); the ``emulate_*`` functions run all
ranks' steps one after another on one device, with the exchanges done as
copies, which is how the one-GPU tests check the bits against the unsharded
calls.
"""
import math
from typing import List, Optional, Sequence, Tuple

import torch

from . import binding

LSE_CHUNK = 256   # vocabulary columns per log-sum-exp partial (the library's chunk)


# ----------------------------------------------------------------------------- partitions

def expert_ranges(E: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous expert ranges [e0, e1), the same size on every rank (E % world == 0)."""
    if world < 1 or E % world != 0:
        raise ValueError(f"{E} experts do not split evenly over {world} ranks")
    n = E // world
    return [(r * n, (r + 1) * n) for r in range(world)]


def vocab_shards(V: int, world: int) -> Tuple[int, List[Tuple[int, int]]]:
    """Chunks per shard P and each rank's vocabulary columns [v0, v1), cut at chunk boundaries.

    NCH = ceil(V / 256) chunks are dealt out P = ceil(NCH / world) at a time; the last shards
    may hold fewer (or none: v0 == v1 == V)."""
    nch = math.ceil(V / LSE_CHUNK)
    P = math.ceil(nch / world)
    out = []
    for r in range(world):
        c0, c1 = min(r * P, nch), min((r + 1) * P, nch)
        out.append((min(c0 * LSE_CHUNK, V), min(c1 * LSE_CHUNK, V)))
    return P, out


def ep_send_counts(counts: torch.Tensor, world: int) -> torch.Tensor:
    """Rows a rank sends to each owner, per local expert: its plan's expert counts [E] viewed
    as [world, E_local] (row d = the rows for rank d's experts)."""
    E = counts.numel()
    if E % world != 0:
        raise ValueError(f"{E} experts do not split evenly over {world} ranks")
    return counts.reshape(world, E // world)


# ----------------------------------------------------------------------------- collectives

class Collectives:
    """The exchange steps of the sharded paths over torch.distributed (any backend)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

    def exchange_counts(self, send_counts: torch.Tensor) -> torch.Tensor:
        """send_counts [world, E_local] (row d to rank d) -> recv_counts [world, E_local] (row s from rank s)."""
        send = send_counts.contiguous()
        recv = torch.empty_like(send)
        self.dist.all_to_all_single(recv.view(-1), send.view(-1), group=self.group)
        return recv

    def exchange_rows(self, send: torch.Tensor, send_splits: Sequence[int], recv_splits: Sequence[int]) -> torch.Tensor:
        """All-to-all of rows: the first send_splits[0] rows to rank 0, the next to rank 1, ...;
        returns the received rows, rank 0's first."""
        recv = torch.empty((int(sum(recv_splits)),) + tuple(send.shape[1:]), dtype=send.dtype, device=send.device)
        self.dist.all_to_all_single(recv, send.contiguous(), [int(v) for v in recv_splits],
                                    [int(v) for v in send_splits], group=self.group)
        return recv

    def gather(self, local: torch.Tensor) -> torch.Tensor:
        """All-gather of equal-shaped tensors into [world, *shape], rank order."""
        out = torch.empty((self.world,) + tuple(local.shape), dtype=local.dtype, device=local.device)
        parts = list(out.unbind(0))
        self.dist.all_gather(parts, local.contiguous(), group=self.group)
        return out


# ----------------------------------------------------------------------------- expert parallelism

def ep_route(w_router, k, x, workspace):
    """Step 1 on every rank: the whole router, top-k, dispatch and permute of its own tokens."""
    return binding.moe_route_topk(x, w_router, k, workspace)


def ep_experts(recv_xp, recv_counts, w13_local, w2_local, workspace):
    """Step 2 on an expert owner: the received rows (source-major) -> its experts' output rows,
    in the received order (fp32)."""
    R = recv_xp.shape[0]
    g = binding.moe_ep_regroup(recv_xp, recv_counts, workspace)
    f = binding.moe_grouped_ffn(g["xp_local"], g["plan_local"], w13_local, w2_local, R, 1, workspace)
    return binding.moe_ep_ungroup(f["y"], g["row_src"])


def ep_combine(route, y_back, x, H, E, k, ws13=None, ws2=None, workspace=None, out_bf16=None):
    """Step 3 on every rank: its own shared expert, then the fixed-order combine of its tokens."""
    T = x.shape[0]
    ys = binding.moe_shared_expert(x, ws13, ws2, workspace) if ws13 is not None else None
    return binding.moe_combine(y_back, route["topk_w"], route["plan"], T, H, E, k, y_shared=ys, out_bf16=out_bf16)


def _ep_workspace(T, H, E_all, E_local, k, F, Fs, R_max, device):
    need = max(binding.workspace_size(T, H, E_all, k, F, Fs, 0), binding.workspace_size(R_max, H, E_local, 1, F, 0, 0))
    return binding.new_workspace(need, device)


class ExpertParallelMoE:
    """One rank of an expert-parallel MoE layer: the router and shared expert replicated, the
    routed experts [e0, e1) local (w13_local [E_local, 2F, H], w2_local [E_local, H, F])."""

    def __init__(self, w_router, w13_local, w2_local, k, coll: Collectives, ws13=None, ws2=None):
        self.w_router, self.w13, self.w2, self.k = w_router, w13_local, w2_local, k
        self.ws13, self.ws2 = ws13, ws2
        self.coll = coll
        self.E = w_router.shape[0]
        self.E_local = w13_local.shape[0]
        if self.E_local * coll.world != self.E:
            raise ValueError("the local experts times the ranks must be all experts")

    def _ws(self, key, nbytes, device):
        """A zero-filled workspace of at least nbytes, kept across calls."""
        cache = self.__dict__.setdefault("_ws_cache", {})
        w = cache.get(key)
        if w is None or w.numel() < nbytes:
            w = binding.new_workspace(nbytes, device)
            cache[key] = w
        return w

    def forward(self, x: torch.Tensor, out_bf16: Optional[torch.Tensor] = None) -> torch.Tensor:
        """x [T, H] bf16 (this rank's tokens) -> out [T, H] fp32, the bits of the one-device layer."""
        T, H = x.shape
        k, E, F = self.k, self.E, self.w13.shape[1] // 2
        Fs = 0 if self.ws13 is None else self.ws13.shape[0] // 2
        ws = self._ws("route", binding.workspace_size(T, H, E, k, F, Fs, 0), x.device)
        r = ep_route(self.w_router, k, x, ws)
        send_counts = ep_send_counts(r["plan"][:E], self.coll.world)
        recv_counts = self.coll.exchange_counts(send_counts)
        send_splits = send_counts.sum(1).tolist()
        recv_splits = recv_counts.sum(1).tolist()
        recv_xp = self.coll.exchange_rows(r["xp"][:T * k], send_splits, recv_splits)
        R = recv_xp.shape[0]
        ws_e = self._ws("experts", binding.workspace_size(R, H, self.E_local, 1, F, 0, 0), x.device)
        y_send = ep_experts(recv_xp, recv_counts, self.w13, self.w2, ws_e)
        y_back = self.coll.exchange_rows(y_send, recv_splits, send_splits)
        return ep_combine(r, y_back, x, H, E, k, self.ws13, self.ws2, ws, out_bf16)


def emulate_expert_parallel(w_router, w13, w2, k, x_shards: Sequence[torch.Tensor], world: int,
                            ws13=None, ws2=None) -> List[torch.Tensor]:
    """All ranks of an expert-parallel layer run one after another on this device; the two
    all-to-alls are done as row copies.  Returns each rank's output for its own tokens."""
    E, F2, H = w13.shape
    F = F2 // 2
    Fs = 0 if ws13 is None else ws13.shape[0] // 2
    ranges = expert_ranges(E, world)
    dev = w13.device
    routes, sends, ws = [], [], []
    for r in range(world):
        T = x_shards[r].shape[0]
        ws.append(_ep_workspace(T, H, E, E // world, k, F, Fs, 0, dev))
        routes.append(ep_route(w_router, k, x_shards[r], ws[r]))
        sends.append(ep_send_counts(routes[r]["plan"][:E], world))
    # all-to-all of rows: owner d receives, from each source s in order, xp_s[offsets[e0_d] : offsets[e1_d]]
    y_send = []
    recv_splits = []
    for d, (e0, e1) in enumerate(ranges):
        recv_counts = torch.stack([sends[s][d] for s in range(world)])
        parts = []
        for s in range(world):
            off = routes[s]["plan"][E:2 * E + 1]
            a, b = int(off[e0]), int(off[e1])
            parts.append(routes[s]["xp"][a:b])
        recv_xp = torch.cat(parts).contiguous()
        recv_splits.append(recv_counts.sum(1).tolist())
        ws_e = _ep_workspace(0, H, E, E // world, k, F, 0, recv_xp.shape[0], dev)
        y_send.append(ep_experts(recv_xp, recv_counts, w13[e0:e1], w2[e0:e1], ws_e))
    # reverse all-to-all: source s gets, from each owner d in order, the rows it sent to d
    outs = []
    for s in range(world):
        T = x_shards[s].shape[0]
        parts = []
        for d in range(world):
            start = sum(recv_splits[d][:s])
            parts.append(y_send[d][start:start + recv_splits[d][s]])
        y_back = torch.cat(parts).contiguous()
        assert y_back.shape[0] == T * k
        outs.append(ep_combine(routes[s], y_back, x_shards[s], H, E, k, ws13, ws2, ws[s]))
    return outs


# ----------------------------------------------------------------------------- vocabulary parallelism

class VocabParallelHead:
    """One rank of a vocabulary-parallel head: rows [v0, v1) of the vocabulary projection local."""

    def __init__(self, w_vocab_shard: torch.Tensor, V: int, coll: Collectives):
        self.coll = coll
        self.V = V
        self.P, shards = vocab_shards(V, coll.world)
        self.v0, self.v1 = shards[coll.rank]
        if w_vocab_shard.shape[0] != self.v1 - self.v0:
            raise ValueError(f"rank {coll.rank} holds vocabulary rows [{self.v0}, {self.v1})")
        self.w = w_vocab_shard

    def forward(self, hidden, target, rollout_logp=None, beta=2.0):
        """The same hidden states and targets on every rank -> logp, lse (k3, mask) on every rank."""
        T = hidden.shape[0]
        part = torch.zeros((T, self.P, 2), dtype=torch.float32, device=hidden.device)
        tgt = torch.zeros(T, dtype=torch.float32, device=hidden.device)
        if self.v1 > self.v0:
            ws = binding.new_workspace(256, hidden.device)
            binding.lm_logprob_partials(hidden, self.w, target, self.V, self.v0, ws, part, tgt)
        return binding.lm_logprob_merge(self.coll.gather(part), self.coll.gather(tgt), target, self.V,
                                        rollout_logp, beta)


def emulate_vocab_parallel(hidden, w_vocab, target, world: int, rollout_logp=None, beta=2.0):
    """All vocabulary shards one after another on this device, each writing its block of the
    gathered arrays ([world, T, P, 2] partials, [world, T] target logits), then the merge."""
    T = hidden.shape[0]
    V = w_vocab.shape[0]
    P, shards = vocab_shards(V, world)
    part = torch.zeros((world, T, P, 2), dtype=torch.float32, device=hidden.device)
    tgt = torch.zeros((world, T), dtype=torch.float32, device=hidden.device)
    ws = binding.new_workspace(256, hidden.device)
    for r, (v0, v1) in enumerate(shards):
        if v1 > v0:
            binding.lm_logprob_partials(hidden, w_vocab[v0:v1], target, V, v0, ws, part[r], tgt[r])
    return binding.lm_logprob_merge(part, tgt, target, V, rollout_logp, beta)
