"""Seeded synthetic inputs for the MoE layer and the logprob/KL head.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic (no routing, no matmul, no softmax).  Both the CUDA path
and the CPU oracle consume exactly the tensors it returns, so the bf16 bits the
two sides see are identical.

Workload shapes follow the pages' MoE workloads by shape only (a Qwen-MoE-like
layer, a GLM-scale layer with one shared expert, and a 151552-entry vocabulary
head); no dataset, checkpoint or trained weight is involved.

Small tensors (activations, router weights, targets, noise) are always drawn on
the CPU generator so their values do not depend on the device; the large weight
banks (expert weights, vocabulary projection) can be drawn directly on a CUDA
device with a CUDA generator of the same seed to avoid a multi-GB host round
trip.  A run that draws them on the CPU gets different (equally valid) values.
"""
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens
    H: int            # hidden size
    E: int            # routed experts
    k: int            # experts per token
    F: int            # SwiGLU ffn size of one routed expert
    F_shared: int = 0  # ffn size of the always-on shared expert (0 = none)
    w_std: float = 0.02
    x_std: float = 1.0
    dup_router_rows: bool = False   # experts 1,3,5,7.. copy the router row of 0,2,4,6..
    zipf_s: float = 0.0             # >0: skew expert popularity p_e ~ rank^-s
    zipf_alpha: float = 0.0         # logit offset scale c_e = alpha * log p_e
    zipf_m: float = 4.0             # size of the shared input direction
    zipf_starve: int = 0            # the n least popular experts get a further -8 logit offset (no tokens)
    seed: int = 0


@dataclass(frozen=True)
class HeadConfig:
    name: str
    T: int
    H: int
    V: int
    w_std: float = 0.02
    x_std: float = 1.0
    noise_std: float = 0.05
    seed: int = 4


# The workloads.  The Zipf offset scale of the Qwen-MoE-like layer (0.27) was
# chosen once, by bisection on this seed's draw, so that the busiest expert gets
# about 1500 of the 4096 tokens.  The 32768 (token, slot) pairs average 256 per
# expert, so a busiest expert near 1500 leaves the least popular about 80 under a
# log-rank offset (a Zipf(1.1) profile scaled to a head of 1500 would hold only
# about 6400 pairs); the variant below also starves the 8 least popular experts,
# so that its counts run from 0 to about 1500.
TINY = MoEConfig("tiny", T=64, H=256, E=8, k=2, F=512, dup_router_rows=True, seed=0)
TINY_HEAD = HeadConfig("tiny_head", T=64, H=256, V=4096, seed=0)
QWEN_MOE = MoEConfig("qwen_moe_like", T=4096, H=2048, E=128, k=8, F=768,
                     zipf_s=1.1, zipf_alpha=0.27, seed=1)
QWEN_MOE_EMPTY = MoEConfig("qwen_moe_like_empty", T=4096, H=2048, E=128, k=8, F=768,
                           zipf_s=1.1, zipf_alpha=0.27, zipf_starve=8, seed=1)
GLM_MOE = MoEConfig("glm_scale_moe", T=8192, H=6144, E=256, k=8, F=2048, F_shared=2048, seed=2)
GLM_HEAD = HeadConfig("glm_scale_head", T=8192, H=6144, V=151552, seed=4)

CONFIGS = {c.name: c for c in (TINY, TINY_HEAD, QWEN_MOE, QWEN_MOE_EMPTY, GLM_MOE, GLM_HEAD)}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std, gen, device="cpu") -> torch.Tensor:
    """float32 N(0, std^2) draw."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def to_bf16(t: torch.Tensor) -> torch.Tensor:
    """Round float32 to bf16 (PyTorch's conversion, round to nearest even)."""
    return t.to(torch.bfloat16)


def zipf_offsets(E: int, s: float, alpha: float, gen, starve: int = 0) -> torch.Tensor:
    """c_e = alpha * log p_e with p_e ~ rank(e)^-s over a seeded permutation of experts; the
    `starve` experts of the lowest popularity get a further -8 (far below the logit noise)."""
    perm = torch.randperm(E, generator=gen)
    rank = torch.empty(E, dtype=torch.float64)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    logp = -s * torch.log(rank)
    logp = logp - torch.logsumexp(logp, 0)
    c = alpha * logp
    if starve > 0:
        c = c - 8.0 * (rank > E - starve).to(torch.float64)
    return c.to(torch.float32)


def moe_activations(cfg: MoEConfig, T: int = None, seed_offset: int = 0):
    """Token activations x [T, H] bf16 and router weights Wr [E, H] bf16 (CPU).

    For a Zipf-skewed config, expert popularity is pushed through the data, not
    through a bias term: one random unit direction u is added to every token
    (x += m u) and to every router row (Wr_e += (c_e / m) u), so the logit of
    expert e gains about c_e.
    """
    T = cfg.T if T is None else T
    g = _gen(cfg.seed * 7919 + 17 + seed_offset)
    x = normal((T, cfg.H), cfg.x_std, g)
    gw = _gen(cfg.seed * 7919 + 3)
    wr = normal((cfg.E, cfg.H), cfg.w_std, gw)
    if cfg.zipf_s > 0:
        u = torch.randn(cfg.H, generator=gw, dtype=torch.float32)
        u = u / u.norm()
        c = zipf_offsets(cfg.E, cfg.zipf_s, cfg.zipf_alpha, gw, cfg.zipf_starve)
        wr = wr + (c / cfg.zipf_m)[:, None] * u[None, :]
        x = x + cfg.zipf_m * u[None, :]
    x = to_bf16(x)
    wr = to_bf16(wr)
    if cfg.dup_router_rows:
        wr[1::2] = wr[0::2]
    return x, wr


def one_expert(cfg: MoEConfig, e: int, device="cpu"):
    """Weights of expert e alone (its own generator), bf16: W13_e [2F, H], W2_e [H, F]."""
    g = _gen(cfg.seed * 7919 + 101 + 7 * e, device)
    w13 = to_bf16(normal((2 * cfg.F, cfg.H), cfg.w_std, g, device))
    w2 = to_bf16(normal((cfg.H, cfg.F), cfg.w_std, g, device))
    return w13, w2


def expert_weights(cfg: MoEConfig, device="cpu"):
    """Expert weight banks, bf16: W13 [E, 2F, H] (gate rows then up rows), W2 [E, H, F].

    Drawn one expert at a time (each from its own seeded generator, so any one
    expert can be re-drawn alone) to bound the float32 temporary.
    """
    w13 = torch.empty((cfg.E, 2 * cfg.F, cfg.H), dtype=torch.bfloat16, device=device)
    w2 = torch.empty((cfg.E, cfg.H, cfg.F), dtype=torch.bfloat16, device=device)
    for e in range(cfg.E):
        w13[e], w2[e] = one_expert(cfg, e, device)
    return w13, w2


def shared_expert_weights(cfg: MoEConfig, device="cpu"):
    """Shared-expert weights, bf16: Ws13 [2Fs, H], Ws2 [H, Fs]; (None, None) if absent."""
    if not cfg.F_shared:
        return None, None
    g = _gen(cfg.seed * 7919 + 202, device)
    ws13 = to_bf16(normal((2 * cfg.F_shared, cfg.H), cfg.w_std, g, device))
    ws2 = to_bf16(normal((cfg.H, cfg.F_shared), cfg.w_std, g, device))
    return ws13, ws2


def head_inputs(cfg: HeadConfig, device="cpu", T: int = None, seed_offset: int = 0):
    """hidden [T, H] bf16 (CPU), Wv [V, H] bf16 (on ``device``), target ids [T] int32 (CPU),
    and two standard-normal noise vectors [T] float32 (CPU) that callers scale by
    the rollout-perturbation std (0.05, and 0.5 to exercise the mask)."""
    T = cfg.T if T is None else T
    g = _gen(cfg.seed * 7919 + 31 + seed_offset)
    hidden = to_bf16(normal((T, cfg.H), cfg.x_std, g))
    target = torch.randint(0, cfg.V, (T,), generator=g, dtype=torch.int64).to(torch.int32)
    noise = torch.randn(T, generator=g, dtype=torch.float32)
    noise_wide = torch.randn(T, generator=g, dtype=torch.float32)
    gw = _gen(cfg.seed * 7919 + 401, device)
    wv = torch.empty((cfg.V, cfg.H), dtype=torch.bfloat16, device=device)
    step = 8192
    for v0 in range(0, cfg.V, step):
        v1 = min(cfg.V, v0 + step)
        wv[v0:v1] = to_bf16(normal((v1 - v0, cfg.H), cfg.w_std, gw, device))
    return hidden, wv, target, noise, noise_wide


def probe_tokens(cfg: MoEConfig, probe_len: int = 32) -> torch.Tensor:
    """The fixed probe request of the batch-invariance sweep (seed 1234), bf16 [probe_len, H]."""
    return to_bf16(normal((probe_len, cfg.H), cfg.x_std, _gen(1234)))


def probe_and_batch(cfg: MoEConfig, n_other: int, trial: int, probe_len: int = 32, skew: bool = False):
    """Batch-invariance sweep input: a fixed probe request embedded in other traffic.

    Returns (x_batch [n_other + probe_len, H] bf16, probe_offset, lengths) where
    the probe's tokens are always the same seeded draw (seed 1234) and the other
    tokens, their request lengths and the probe's offset vary with ``trial``.
    With ``skew`` the other tokens are perturbed copies of probe tokens, so they
    route to the probe's experts and push the probe's rows to other positions
    inside those experts' tiles.
    """
    probe = probe_tokens(cfg, probe_len)
    g = _gen(100003 + trial * 31 + n_other + (7 if skew else 0))
    other = normal((n_other, cfg.H), cfg.x_std, g)
    if skew and n_other > 0:
        src = torch.randint(0, probe_len, (n_other,), generator=g)
        other = probe.float()[src] + 0.05 * other
    other = to_bf16(other)
    # random request lengths: 1 = a decode token, >1 = a prefill chunk
    lengths = []
    left = n_other
    while left > 0:
        if torch.rand(1, generator=g).item() < 0.5:
            n = 1
        else:
            n = int(torch.randint(2, 257, (1,), generator=g).item())
        n = min(n, left)
        lengths.append(n)
        left -= n
    # probe inserted between two requests
    cut = int(torch.randint(0, len(lengths) + 1, (1,), generator=g).item()) if lengths else 0
    off = sum(lengths[:cut])
    x = torch.cat([other[:off], probe, other[off:]], 0)
    return x, off, lengths
