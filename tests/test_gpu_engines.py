"""The two engines of the grouped expert GEMMs give the same bits.

moe_grouped_ffn runs the routed experts' two GEMMs either with each expert's tokens on the MMA's
M side in 128-row tiles (the row-tile engine) or with its weights on the M side and its tokens on
the N side (the token-column engine, in 64-, 128- or 320-token units by batch size; by default it
runs every gate/up GEMM and some down projections).  Every element is the same K-ascending chain of
bf16 products accumulated in fp32 either way ("位级一致：前沿训练的差异化关键", section
"为什么比特级一致是一个复杂的问题": one fixed reduction order per element whatever the token
count), so h, Y and the layer output must match bit for bit: on layers with empty experts, experts
with one token, experts split into several token chunks, and at full size."""
import dataclasses

import pytest
import torch

from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _both_engines(cfg, expert_device="cpu"):
    from serve_invariant_moe_gb300 import _lib, api
    lib = _lib.lib()
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, expert_device)
    ws13, ws2 = synth.shared_expert_weights(cfg, expert_device)
    c = lambda t: None if t is None else t.cuda()   # noqa: E731
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), c(w13), c(w2), cfg.k, c(ws13), c(ws2)))
    S = cfg.T * cfg.k
    out = {}
    try:
        for eng in (0, 1):
            assert lib.invmoe_expert_engine(eng) == 0
            r = layer.prefill(x.cuda(), return_all=True)
            torch.cuda.synchronize()
            out[eng] = dict(h=r["h"][:S].clone(), y=r["y"][:S].clone(), out=r["out"].clone(),
                            counts=r["plan"][:cfg.E].cpu())
    finally:
        lib.invmoe_expert_engine(2)
    return out


SMALL = [
    # a heavy expert (several token chunks of the token-column engine), empty and one-token experts
    dataclasses.replace(synth.TINY, name="heavy_and_empty", T=900, H=256, E=16, k=2, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=2.5, seed=61),
    # H = 384 is not a multiple of 256: the down projection falls back to the row tiles
    dataclasses.replace(synth.TINY, name="h384_shared", T=190, H=384, E=12, k=4, F=384, F_shared=256,
                        dup_router_rows=False, seed=62),
    # one token in all
    dataclasses.replace(synth.TINY, name="one_token", T=1, H=512, E=8, k=8, F=128, dup_router_rows=False, seed=63),
    # every expert just above and below a chunk boundary
    dataclasses.replace(synth.TINY, name="near_chunk_edges", T=1300, H=256, E=8, k=2, F=512,
                        dup_router_rows=False, seed=64),
    # at most 64 slots in all (the decode form: 64-token units, a 32-row token tile per CTA):
    # one expert holding all 64, and 8 slots per token spread over 16 experts
    dataclasses.replace(synth.TINY, name="decode_form_one_full_unit", T=64, H=512, E=4, k=1, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=5.0, seed=65),
    dataclasses.replace(synth.TINY, name="decode_form_mixed", T=8, H=2048, E=16, k=8, F=256, F_shared=128,
                        dup_router_rows=False, seed=66),
    # up to 1024 slots run the decode form too: experts of more than 64 tokens take several units
    dataclasses.replace(synth.TINY, name="decode_form_multi_unit", T=480, H=1024, E=8, k=2, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=1.5, seed=67),
    # at most 64 slots per expert on average (128-token units, a 32- or 64-row token tile per CTA):
    # empty experts, experts of up to 32, 33-64 and 65-128 tokens, and experts of several units
    dataclasses.replace(synth.TINY, name="unit128_form", T=600, H=512, E=64, k=4, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=0.4, seed=69),
    # H = 448: seven 64-wide K blocks, so the forms whose ring stages hold two K blocks (64-token
    # units; 128-token SwiGLU units) end on a stage with one
    dataclasses.replace(synth.TINY, name="odd_k_blocks_units64", T=200, H=448, E=16, k=4, F=256,
                        dup_router_rows=False, seed=70),
    dataclasses.replace(synth.TINY, name="odd_k_blocks_units128", T=600, H=448, E=64, k=4, F=256,
                        dup_router_rows=False, zipf_s=1.1, zipf_alpha=0.4, seed=69),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_engines_bit_identical_small(cfg):
    r = _both_engines(cfg)
    counts = r[1]["counts"]
    if cfg.name == "heavy_and_empty":
        assert counts.max() > 640 and (counts == 0).any()     # three or more chunks; empty experts
    if cfg.name == "decode_form_one_full_unit":
        assert counts.max() == 64                              # one expert fills a whole 64-token unit
    if cfg.name == "decode_form_multi_unit":
        assert counts.max() > 128                              # three or more 64-token units
    if cfg.name == "unit128_form":
        S, E = cfg.T * cfg.k, cfg.E
        assert 16 * E < S <= 64 * E                            # the batch takes the 128-token units
        assert (counts == 0).any() and ((counts > 32) & (counts <= 64)).any()
        assert ((counts > 64) & (counts <= 128)).any() and counts.max() > 256
    for key in ("h", "y", "out"):
        assert torch.equal(_bits(r[0][key]), _bits(r[1][key])), f"{cfg.name}: {key} differs between the engines"


@pytest.mark.slow
@pytest.mark.parametrize("name,T", [("glm_scale_moe", None), ("qwen_moe_like_empty", None),
                                    ("glm_scale_moe", 1024), ("qwen_moe_like_empty", 1024)])
def test_engines_bit_identical_full_size(name, T):
    # at the configurations' own batch sizes the token columns run 320-token units; at 1024 tokens
    # (32 and 64 slots per expert) 128-token units
    cfg = synth.CONFIGS[name]
    if T is not None:
        cfg = dataclasses.replace(cfg, T=T)
    r = _both_engines(cfg, expert_device="cuda")
    for key in ("h", "y", "out"):
        assert torch.equal(_bits(r[0][key]), _bits(r[1][key])), f"{name}: {key} differs between the engines"


# Per-expert token counts fixed through router replay (k = 1), one list per unit form of the token
# columns: every chunk width where a CTA's token rows change box or split.
#   320-token units (more than 64 slots per expert on average): chunks of 257-320 tokens take a
#   second MMA of 16, 32, 48 or 64 columns and one 160-row box per CTA; 321 splits into two chunks.
#   128-token units (at most 64 per expert): a CTA's share of up to 32 rows in a 32-row box, of 33-64
#   rows in a 64-row box; experts of more than 128 tokens split into near-equal chunks.
#   64-token units (at most 1024 slots): one 32-row box; experts of more than 64 tokens split.
EXACT_COUNTS = {
    "units320": (16, [0, 1, 15, 16, 17, 255, 256, 257, 272, 273, 288, 289, 304, 305, 320, 321]),
    "units128": (64, [0, 1, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257] + [0] * 50),
    "units64": (16, [0, 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 129, 0, 0, 0, 0]),
}


@pytest.mark.parametrize("form", sorted(EXACT_COUNTS))
def test_engines_bit_identical_exact_chunk_widths(form):
    from serve_invariant_moe_gb300 import _lib, api
    lib = _lib.lib()
    E, counts = EXACT_COUNTS[form]
    T = sum(counts)
    # the batch takes the intended unit form (same thresholds as the library's dispatch)
    if form == "units320":
        assert T > 64 * E
    elif form == "units128":
        assert 16 * E < T <= 64 * E and T > 1024
    else:
        assert T <= 1024
    cfg = dataclasses.replace(synth.TINY, name=f"exact_{form}", T=T, H=256, E=E, k=1, F=256,
                              dup_router_rows=False, seed=80)
    x, wr = synth.moe_activations(cfg)
    w13, w2 = synth.expert_weights(cfg, "cuda")
    experts = torch.repeat_interleave(torch.arange(E), torch.tensor(counts))
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(81))
    replay = experts[perm].to(torch.int32).view(T, 1).cuda()
    layer = api.MoELayer(api.MoEWeights(wr.cuda(), w13, w2, 1))
    out = {}
    try:
        for eng in (0, 1):
            assert lib.invmoe_expert_engine(eng) == 0
            r = layer.prefill(x.cuda(), return_all=True, replay_idx=replay)
            torch.cuda.synchronize()
            out[eng] = dict(h=r["h"][:T].clone(), y=r["y"][:T].clone(), out=r["out"].clone(),
                            counts=r["plan"][:E].cpu())
    finally:
        lib.invmoe_expert_engine(2)
    assert out[1]["counts"].tolist() == counts
    for key in ("h", "y", "out"):
        assert torch.equal(_bits(out[0][key]), _bits(out[1][key])), f"{form}: {key} differs between the engines"
