"""Out-of-bounds and unwritten-element checks (the sanitizer's job, done with poisoned buffers).

Every output buffer is filled with a NaN bit pattern that no kernel computes (finite inputs give
finite results), with guard rows past the region a call may write.  After the call, the region it
owns must hold no poison (every element written) and the guard rows must hold nothing else (no
store past the end).  Covered: the routing's permuted rows, both engines of the grouped expert GEMMs
(the token-column engine's 64- and 128-token unit forms, several-chunk experts and empty
experts included), and the decode buffers, of which a call on fewer requests than they were sized for owns
only the leading rows."""
import dataclasses

import pytest
import torch

from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu

POISON_BF16 = 0x7FC1            # a NaN payload no kernel writes
POISON_F32 = 0x7FC00123
GUARD = 67                      # guard rows past the owned region


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _poisoned(rows, cols, dtype):
    if dtype == torch.bfloat16:
        return torch.full((rows, cols), POISON_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return torch.full((rows, cols), POISON_F32, dtype=torch.int32, device="cuda").view(torch.float32)


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _check(name, buf, owned_rows):
    poison = POISON_BF16 if buf.dtype == torch.bfloat16 else POISON_F32
    b = _bits(buf)
    assert not (b[:owned_rows] == poison).any(), f"{name}: element of rows [0, {owned_rows}) never written"
    assert (b[owned_rows:] == poison).all(), f"{name}: store past row {owned_rows}"


CFGS = [
    dataclasses.replace(synth.TINY, name="heavy_and_empty", T=900, H=256, E=16, k=2, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=2.5, seed=71),
    dataclasses.replace(synth.TINY, name="decode_form", T=8, H=2048, E=16, k=8, F=256,
                        dup_router_rows=False, seed=72),
    dataclasses.replace(synth.TINY, name="one_token", T=1, H=512, E=8, k=8, F=128, dup_router_rows=False, seed=73),
    dataclasses.replace(synth.TINY, name="ragged_rows", T=333, H=512, E=24, k=4, F=384, dup_router_rows=False,
                        seed=74),
    # the decode form with experts of more than 64 tokens (several 64-token units each)
    dataclasses.replace(synth.TINY, name="decode_form_multi_unit", T=300, H=512, E=8, k=2, F=256,
                        dup_router_rows=False, seed=76),
    # the 128-token units (at most 64 slots per expert on average), skewed: empty experts, experts
    # of 33-64 and 65-128 tokens, experts of several units
    dataclasses.replace(synth.TINY, name="unit128_form", T=600, H=512, E=64, k=4, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=0.4, seed=69),
    # seven K blocks (H = 448) in the forms whose stages hold two
    dataclasses.replace(synth.TINY, name="odd_k_blocks_units64", T=200, H=448, E=16, k=4, F=256,
                        dup_router_rows=False, seed=79),
]


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: c.name)
def test_routing_and_expert_gemms_write_exactly_their_rows(cfg):
    from serve_invariant_moe_gb300 import _lib, binding
    lib = _lib.lib()
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    x, wr = x.cuda(), wr.cuda()
    S = cfg.T * cfg.k
    ws = binding.new_workspace(binding.workspace_size(cfg.T, cfg.H, cfg.E, cfg.k, cfg.F, 0, 0))
    xp = _poisoned(S + GUARD, cfg.H, torch.bfloat16)
    r = binding.moe_route_topk(x, wr, cfg.k, ws, xp=xp)
    torch.cuda.synchronize()
    _check("xp", xp, S)
    try:
        for eng in (0, 1):
            assert lib.invmoe_expert_engine(eng) == 0
            h = _poisoned(S + GUARD, cfg.F, torch.bfloat16)
            y = _poisoned(S + GUARD, cfg.H, torch.float32)
            binding.moe_grouped_ffn(r["xp"], r["plan"], w13, w2, cfg.T, cfg.k, ws, h=h, y=y)
            torch.cuda.synchronize()
            binding.check_status(ws)
            _check(f"h (engine {eng})", h, S)
            _check(f"y (engine {eng})", y, S)
    finally:
        lib.invmoe_expert_engine(2)


def test_decode_on_fewer_requests_writes_only_their_rows():
    from serve_invariant_moe_gb300 import api
    cfg = dataclasses.replace(synth.GLM_MOE, name="guard_decode", H=512, E=32, k=8, F=256, F_shared=256, seed=75)
    x, wr = synth.moe_activations(cfg, T=64)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    ws13, ws2 = synth.shared_expert_weights(cfg, "cuda")
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13, w2, cfg.k, ws13, ws2))
    Bmax = 64
    layer.alloc_decode(Bmax)
    d = layer._decode
    for B in (1, 5, 37):
        for key, dtype in (("xp", torch.bfloat16), ("h", torch.bfloat16), ("y", torch.float32),
                           ("ys", torch.float32), ("out", torch.float32)):
            t = d[key]
            t.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).fill_(
                POISON_BF16 if dtype == torch.bfloat16 else POISON_F32)
        layer.decode(x[:B].cuda())
        torch.cuda.synchronize()
        for key, rows in (("xp", B * cfg.k), ("h", B * cfg.k), ("y", B * cfg.k), ("ys", B), ("out", B)):
            _check(f"{key} (B={B})", d[key], rows)


def test_expert_gemms_write_exactly_their_rows_at_exact_chunk_widths():
    # per-expert counts fixed through router replay (k = 1): chunks of 257-320 tokens (a second MMA
    # of each width, one 160-row token box per CTA of the pair) and a 321-token expert split in two
    from serve_invariant_moe_gb300 import _lib, binding
    lib = _lib.lib()
    counts = [0, 1, 15, 16, 17, 255, 256, 257, 272, 273, 288, 289, 304, 305, 320, 321]
    E, T = len(counts), sum(counts)
    cfg = dataclasses.replace(synth.TINY, name="guard_exact", T=T, H=256, E=E, k=1, F=256,
                              dup_router_rows=False, seed=77)
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    experts = torch.repeat_interleave(torch.arange(E), torch.tensor(counts))
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(78))
    replay = experts[perm].to(torch.int32).view(T, 1).cuda()
    ws = binding.new_workspace(binding.workspace_size(T, cfg.H, E, 1, cfg.F, 0, 0))
    r = binding.moe_route_replay(x.cuda(), wr.cuda(), replay, ws)
    torch.cuda.synchronize()
    assert r["plan"][:E].cpu().tolist() == counts
    try:
        for eng in (0, 1):
            assert lib.invmoe_expert_engine(eng) == 0
            h = _poisoned(T + GUARD, cfg.F, torch.bfloat16)
            y = _poisoned(T + GUARD, cfg.H, torch.float32)
            binding.moe_grouped_ffn(r["xp"], r["plan"], w13, w2, T, 1, ws, h=h, y=y)
            torch.cuda.synchronize()
            binding.check_status(ws)
            _check(f"h (engine {eng})", h, T)
            _check(f"y (engine {eng})", y, T)
    finally:
        lib.invmoe_expert_engine(2)
