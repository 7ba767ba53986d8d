"""Expert-parallel layer and vocabulary-parallel head, all ranks emulated one after another on one
GPU (the exchanges done as copies), against the unsharded calls: every output must be bit-identical.

"位级一致：前沿训练的差异化关键", section "为什么比特级一致是一个复杂的问题" (a cross-device
reduction must not change with the size of the job) and "GLM Post-Training Beyond SFT", section
"动作与概率契约" (the vocabulary-parallel log-sum-exp needs comparison tests).  The sharded paths
move rows and partials between ranks and reduce nothing across them, so any split must give the
one-device bits; the unsharded calls are themselves held to the oracle by the other tests, and
the merge of the sharded head is checked against the oracle here too."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from helpers import LOGP_ABS, f64
from oracle import head as ohead
from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


# ----------------------------------------------------------------------------- vocabulary parallel

@pytest.mark.parametrize("T,H,V", [(300, 256, 8196), (64, 128, 4096), (5, 64, 151552)])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_vocab_parallel_head_bit_identical(T, H, V, world):
    from serve_invariant_moe_gb300 import api, sharded
    g = torch.Generator().manual_seed(T + V + world)
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16).cuda()
    wv = (torch.randn((V, H), generator=g) * 0.05).to(torch.bfloat16).cuda()
    target = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    target[0] = V - 1                       # the last (partial) chunk
    target[-1] = 0
    target = target.cuda()
    rollout = (torch.randn(T, generator=g) * 0.5 - math.log(V)).cuda()
    ref = api.head_logprob_kl(hidden, wv, target, rollout_logp=rollout)
    got = sharded.emulate_vocab_parallel(hidden, wv, target, world, rollout_logp=rollout)
    torch.cuda.synchronize()
    for key in ("logp", "lse", "k3", "mask"):
        assert torch.equal(_bits(got[key]), _bits(ref[key])), f"{key} differs with {world} shards"


def test_vocab_parallel_shard_logits_and_oracle():
    """Each shard writes its own columns of the logits; the merged logprobs match the oracle."""
    from serve_invariant_moe_gb300 import api, binding, sharded
    T, H, V, world = 40, 192, 3000, 3
    g = torch.Generator().manual_seed(77)
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16)
    wv = (torch.randn((V, H), generator=g) * 0.05).to(torch.bfloat16)
    target = torch.randint(0, V, (T,), generator=g, dtype=torch.int32)
    hd, wd, td = hidden.cuda(), wv.cuda(), target.cuda()
    full = api.head_logprob_kl(hd, wd, td, write_logits=True)
    P, shards = sharded.vocab_shards(V, world)
    logits = torch.full((T, V), float("nan"), device="cuda")
    part = torch.zeros((world, T, P, 2), device="cuda")
    tgt = torch.zeros((world, T), device="cuda")
    ws = binding.new_workspace(256)
    for r, (v0, v1) in enumerate(shards):
        binding.lm_logprob_partials(hd, wd[v0:v1], td, V, v0, ws, part[r], tgt[r], logits=logits)
    merged = binding.lm_logprob_merge(part, tgt, td, V)
    torch.cuda.synchronize()
    assert torch.equal(_bits(logits), _bits(full["logits"]))
    assert torch.equal(_bits(merged["logp"]), _bits(full["logp"]))
    ref = ohead.head_forward(f64(hidden), f64(wv), target.numpy())
    assert np.abs(merged["logp"].double().cpu().numpy() - ref["logp"]).max() <= LOGP_ABS


def test_vocab_shard_rejects_unaligned_bounds():
    from serve_invariant_moe_gb300 import _lib, binding
    T, H, V = 4, 64, 1024
    hidden = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    wv = torch.zeros((V, H), dtype=torch.bfloat16, device="cuda")
    target = torch.zeros(T, dtype=torch.int32, device="cuda")
    part = torch.zeros((T, 4, 2), device="cuda")
    tgt = torch.zeros(T, device="cuda")
    ws = binding.new_workspace(256)
    with pytest.raises(_lib.InvmoeError, match="chunk boundary"):
        binding.lm_logprob_partials(hidden, wv[100:612], target, V, 100, ws, part, tgt)
    with pytest.raises(_lib.InvmoeError, match="ld_part"):
        binding.lm_logprob_partials(hidden, wv, target, V, 0, ws, torch.zeros((T, 2, 2), device="cuda"), tgt)


# ----------------------------------------------------------------------------- expert parallel

def _moe_inputs(cfg, starve=()):
    x, wr = synth.moe_activations(cfg)
    if starve:
        # push the starved experts' logits far below the others through the data: a shared
        # direction u in every token, +u in the other router rows, -u in the starved ones
        g = torch.Generator().manual_seed(5)
        u = torch.randn(cfg.H, generator=g)
        u = u / u.norm()
        x = (x.float() + 4.0 * u).to(torch.bfloat16)
        sign = torch.ones(cfg.E)
        sign[list(starve)] = -1.0
        wr = (wr.float() + 2.0 * sign[:, None] * u[None, :]).to(torch.bfloat16)
    w13, w2 = synth.expert_weights(cfg)
    ws13, ws2 = synth.shared_expert_weights(cfg)
    c = lambda t: None if t is None else t.cuda()   # noqa: E731
    return x.cuda(), wr.cuda(), w13.cuda(), w2.cuda(), c(ws13), c(ws2)


EP_CASES = [
    (dataclasses.replace(synth.TINY, name="ep_shared", T=777, H=256, E=16, k=4, F=256, F_shared=128,
                         dup_router_rows=False, seed=41), (2, 4, 8), ()),
    (dataclasses.replace(synth.TINY, name="ep_skew_empty_owner", T=500, H=512, E=8, k=2, F=384,
                         dup_router_rows=False, zipf_s=1.1, zipf_alpha=1.0, seed=42), (2, 4), (6, 7)),
    (dataclasses.replace(synth.TINY, name="ep_wide", T=1500, H=1024, E=64, k=8, F=512, F_shared=256,
                         dup_router_rows=False, seed=43), (4, 8), ()),
]


@pytest.mark.parametrize("cfg,worlds,starve", EP_CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_expert_parallel_layer_bit_identical(cfg, worlds, starve):
    from serve_invariant_moe_gb300 import api, sharded
    x, wr, w13, w2, ws13, ws2 = _moe_inputs(cfg, starve)
    layer = api.MoELayer(api.MoEWeights(wr, w13, w2, cfg.k, ws13, ws2))
    ref = layer.prefill(x, return_all=True)
    counts = ref["plan"][:cfg.E].cpu()
    if starve:
        assert (counts[list(starve)] == 0).all()        # the owner of experts 6, 7 receives no rows
    for world in worlds:
        # uneven token shards; with more than two ranks the first one holds no token
        gen = torch.Generator().manual_seed(world)
        cuts = sorted(torch.randint(0, cfg.T + 1, (world - 1,), generator=gen).tolist())
        if world > 2:
            cuts[0] = 0
        bounds = [0] + cuts + [cfg.T]
        shards = [x[a:b] for a, b in zip(bounds[:-1], bounds[1:])]
        outs = sharded.emulate_expert_parallel(wr, w13, w2, cfg.k, shards, world, ws13, ws2)
        torch.cuda.synchronize()
        got = torch.cat(outs)
        assert torch.equal(_bits(got), _bits(ref["out"])), f"{cfg.name}: {world} expert-parallel ranks differ"


def test_ep_regroup_order_and_plan():
    """The regroup kernel alone: source-major rows in, expert-major rows out, sources ascending."""
    from serve_invariant_moe_gb300 import binding
    n_src, E_local, H = 3, 4, 64
    counts = torch.tensor([[2, 0, 1, 3], [0, 0, 2, 1], [1, 4, 0, 0]], dtype=torch.int32)
    R = int(counts.sum())
    # row i of the received buffer holds the value i everywhere
    recv = torch.arange(R, dtype=torch.float32)[:, None].repeat(1, H).to(torch.bfloat16).cuda()
    ws = binding.new_workspace(256)
    g = binding.moe_ep_regroup(recv, counts.cuda(), ws)
    binding.check_status(ws)
    # expected: for each expert, for each source, that source's rows for the expert
    src_start = torch.cumsum(counts.view(-1), 0) - counts.view(-1)
    order = []
    for e in range(E_local):
        for s in range(n_src):
            a = int(src_start[s * E_local + e])
            order += list(range(a, a + int(counts[s, e])))
    assert g["row_src"][:R].cpu().tolist() == order
    assert torch.equal(g["xp_local"].float().cpu()[:, 0], torch.tensor(order, dtype=torch.float32))
    tot = counts.sum(0)
    plan = g["plan_local"].cpu()
    assert plan[:E_local].tolist() == tot.tolist()
    assert plan[E_local:].tolist() == [0] + torch.cumsum(tot, 0).tolist()
    # and back: ungroup restores the received order
    y = g["xp_local"].float()
    back = binding.moe_ep_ungroup(y.contiguous(), g["row_src"][:R])
    assert torch.equal(back, recv.float())


def test_ep_regroup_counts_that_do_not_add_up_are_reported():
    from serve_invariant_moe_gb300 import _lib, binding
    counts = torch.tensor([[5, 5]], dtype=torch.int32).cuda()      # 10 rows claimed
    recv = torch.zeros((6, 64), dtype=torch.bfloat16, device="cuda")  # 6 rows given
    ws = binding.new_workspace(256)
    binding.moe_ep_regroup(recv, counts, ws)
    with pytest.raises(_lib.InvmoeError, match="do not add up"):
        binding.check_status(ws)
    # the context still works
    binding.check_status(ws)


def test_shared_expert_alone_matches_the_fused_call():
    from serve_invariant_moe_gb300 import api, binding
    cfg = dataclasses.replace(synth.TINY, name="shared_alone", T=333, H=384, E=8, k=2, F=256, F_shared=384,
                              dup_router_rows=False, seed=44)
    x, wr, w13, w2, ws13, ws2 = _moe_inputs(cfg)
    ref = api.MoELayer(api.MoEWeights(wr, w13, w2, cfg.k, ws13, ws2)).prefill(x, return_all=True)
    ws = binding.new_workspace(binding.workspace_size(cfg.T, cfg.H, F_shared=cfg.F_shared))
    ys = binding.moe_shared_expert(x, ws13, ws2, ws)
    torch.cuda.synchronize()
    assert torch.equal(_bits(ys), _bits(ref["y_shared"]))


def test_sharded_classes_over_nccl_with_one_rank():
    """The torch.distributed path itself (ExpertParallelMoE, VocabParallelHead, Collectives) on a
    one-rank NCCL group: every collective runs for real (with one rank it moves the data to itself),
    and the outputs are the unsharded calls' bits."""
    import socket

    import torch.distributed as dist
    from serve_invariant_moe_gb300 import api, sharded
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        coll = sharded.Collectives()
        cfg = EP_CASES[0][0]
        x, wr, w13, w2, ws13, ws2 = _moe_inputs(cfg)
        ref = api.MoELayer(api.MoEWeights(wr, w13, w2, cfg.k, ws13, ws2)).prefill(x)
        ep = sharded.ExpertParallelMoE(wr, w13, w2, cfg.k, coll, ws13, ws2)
        got = ep.forward(x)
        torch.cuda.synchronize()
        assert torch.equal(_bits(got), _bits(ref))
        T, H, V = 70, 128, 3000
        g = torch.Generator().manual_seed(91)
        hidden = torch.randn((T, H), generator=g).to(torch.bfloat16).cuda()
        wv = (torch.randn((V, H), generator=g) * 0.05).to(torch.bfloat16).cuda()
        target = torch.randint(0, V, (T,), generator=g, dtype=torch.int32).cuda()
        rollout = (torch.randn(T, generator=g) * 0.5 - math.log(V)).cuda()
        href = api.head_logprob_kl(hidden, wv, target, rollout_logp=rollout)
        vp = sharded.VocabParallelHead(wv, V, coll)
        hgot = vp.forward(hidden, target, rollout)
        torch.cuda.synchronize()
        for key in ("logp", "lse", "k3", "mask"):
            assert torch.equal(_bits(hgot[key]), _bits(href[key])), key
    finally:
        dist.destroy_process_group()
