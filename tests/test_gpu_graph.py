"""The decode entry point captured into a CUDA graph and replayed: the same bits as
the eager decode path (no host synchronisation or allocation inside the path)."""
import dataclasses

import pytest
import torch

from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu


def test_decode_graph_replay_matches_eager():
    from serve_invariant_moe_gb300 import api, build
    build.build()
    cfg = dataclasses.replace(synth.GLM_MOE, name="graph_small", H=512, E=32, k=8, F=256, F_shared=256, seed=41)
    _, wr = synth.moe_activations(cfg, T=1)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    ws13, ws2 = synth.shared_expert_weights(cfg, "cuda")
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13, w2, cfg.k, ws13, ws2))
    B = 48
    layer.alloc_decode(B)
    static_x = torch.zeros((B, cfg.H), dtype=torch.bfloat16, device="cuda")
    g = torch.Generator().manual_seed(7)
    batches = [synth.to_bf16(torch.randn((B, cfg.H), generator=g)).cuda() for _ in range(3)]
    eager = [layer.decode(x).clone() for x in batches]
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        static_x.copy_(batches[0])
        layer.decode(static_x)                      # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        static_out = layer.decode(static_x)
    for x, ref in zip(batches, eager):
        static_x.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(static_out, ref)


def test_decode_graph_buckets_match_eager_decode():
    from serve_invariant_moe_gb300 import api, build
    build.build()
    cfg = dataclasses.replace(synth.GLM_MOE, name="graph_buckets", H=512, E=32, k=8, F=256, F_shared=256, seed=42)
    _, wr = synth.moe_activations(cfg, T=1)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    ws13, ws2 = synth.shared_expert_weights(cfg, "cuda")
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13, w2, cfg.k, ws13, ws2))
    graphs = api.DecodeGraphs(layer, buckets=(1, 4, 16))
    eager_layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13, w2, cfg.k, ws13, ws2))
    g = torch.Generator().manual_seed(11)
    for b in (1, 3, 4, 9, 16):
        x = synth.to_bf16(torch.randn((b, cfg.H), generator=g)).cuda()
        ref = eager_layer.decode(x).clone()
        got = graphs(x).clone()
        torch.cuda.synchronize()
        assert torch.equal(got, ref), b


def test_input_stager_double_buffers_in_order():
    """Copies of batch i+1 overlap the work on batch i; every batch reaches the device intact and
    no buffer is overwritten while the current stream still reads it."""
    from serve_invariant_moe_gb300 import api
    like = dict(x=torch.empty((4096, 1024), dtype=torch.bfloat16, device="cuda"),
                t=torch.empty(4096, dtype=torch.int32, device="cuda"))
    stager = api.InputStager(like)
    g = torch.Generator().manual_seed(5)
    host = [dict(x=torch.randn((4096, 1024), generator=g).to(torch.bfloat16).pin_memory(),
                 t=torch.randint(0, 1000, (4096,), generator=g, dtype=torch.int32).pin_memory()) for _ in range(6)]
    outs = []
    stager.stage(host[0])
    for i in range(6):
        inp = stager.next()
        if i + 1 < 6:
            stager.stage(host[i + 1])
        # some work on the current stream that reads the buffers for a while
        acc = inp["x"].float()
        for _ in range(20):
            acc = acc * 1.0 + 0.0
        outs.append((acc.to(torch.bfloat16), inp["t"].clone()))
        stager.release()
    torch.cuda.synchronize()
    for i, (x, t) in enumerate(outs):
        assert torch.equal(x.cpu(), host[i]["x"]) and torch.equal(t.cpu(), host[i]["t"]), i
