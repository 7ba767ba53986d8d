"""The tcgen05 GEMM engine on its own, against the float64 oracle product.

Sizes span several tiles in both directions plus ragged row and column tails,
for every tile variant the hot path uses."""
import numpy as np
import pytest
import torch

from helpers import dot_bound, f64
from oracle import moe as omoe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ws():
    from serve_invariant_moe_gb300 import binding, build
    build.build()
    return binding.new_workspace(4096)


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (128, 256, 64), (300, 520, 192), (777, 1028, 512),
                                   (64, 8, 256)])
def test_gemm_matches_oracle(ws, variant, M, N, K):
    from serve_invariant_moe_gb300 import binding
    a = _rand((M, K), 1 + M + K)
    b = _rand((N, K), 2 + N + K, 0.05)
    d = binding.gemm_bf16(a.cuda(), b.cuda(), ws, variant=variant)
    binding.check_status(ws)
    a64, b64 = f64(a), f64(b)
    ref = omoe.router_logits(a64, b64)      # a plain float64 product
    err = np.abs(d.double().cpu().numpy() - ref)
    bound = dot_bound(a64, b64, K)
    assert (err <= bound).all(), f"max err/bound {(err / bound).max():.3f}"


def test_gemm_rows_independent_of_position(ws):
    """The same A row gives the same bits at every row position of a tile and in
    every tile (row-position invariance of the MMA, assumed by batch invariance)."""
    from serve_invariant_moe_gb300 import binding
    K, N = 256, 256
    row = _rand((1, K), 7)
    others = _rand((400, K), 8)
    b = _rand((N, K), 9, 0.05).cuda()
    ref = binding.gemm_bf16(row.cuda(), b, ws, variant=1).cpu()
    for pos in (0, 1, 63, 127, 128, 200, 255, 256, 399):
        a = others.clone()
        a[pos] = row[0]
        d = binding.gemm_bf16(a.cuda(), b, ws, variant=1).cpu()
        assert torch.equal(d[pos], ref[0]), pos


def test_identical_b_rows_give_identical_columns(ws):
    from serve_invariant_moe_gb300 import binding
    K = 512
    a = _rand((200, K), 10).cuda()
    b = _rand((64, K), 11, 0.05)
    b[1::2] = b[0::2]
    d = binding.gemm_bf16(a, b.cuda(), ws, variant=3).cpu()
    assert torch.equal(d[:, 0::2], d[:, 1::2])


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (256, 256, 64), (300, 520, 192), (777, 1028, 512), (1000, 64, 256)])
def test_pair_tile_matches_oracle_and_single_cta_bits(ws, M, N, K):
    """The CTA-pair (cta_group::2) 256 x 256 tile: within the fp32 bound of the oracle
    and bit-identical to the single-CTA 128 x 256 tile."""
    from serve_invariant_moe_gb300 import binding
    a = _rand((M, K), 3 + M + K)
    b = _rand((N, K), 4 + N + K, 0.05)
    d = binding.gemm_bf16(a.cuda(), b.cuda(), ws, variant=4)
    d1 = binding.gemm_bf16(a.cuda(), b.cuda(), ws, variant=1)
    binding.check_status(ws)
    a64, b64 = f64(a), f64(b)
    err = np.abs(d.double().cpu().numpy() - omoe.router_logits(a64, b64))
    assert (err <= dot_bound(a64, b64, K)).all()
    assert torch.equal(d, d1)


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (256, 256, 128), (300, 520, 192), (777, 1032, 512)])
def test_mn_major_operands_give_the_k_major_bits(ws, M, N, K):
    """MN-major operand tiles (b stored [K, N]; a stored [K, M]) give bit-identical
    results to the K-major tiles of the same matrices: only the shared-memory layout
    and the descriptors differ, not the MMAs or their order."""
    from serve_invariant_moe_gb300 import binding
    a = _rand((M, K), 30 + M + K)
    b = _rand((N, K), 31 + N + K, 0.05)
    ref = binding.gemm_bf16(a.cuda(), b.cuda(), ws, variant=4)
    d5 = binding.gemm_bf16(a.cuda(), b.t().contiguous().cuda(), ws, variant=5)
    binding.check_status(ws)
    assert torch.equal(d5, ref)
    if M % 8 == 0:
        d6 = binding.gemm_bf16(a.t().contiguous().cuda(), b.t().contiguous().cuda(), ws, variant=6)
        binding.check_status(ws)
        assert torch.equal(d6, ref)


@pytest.mark.parametrize("variant,M,N,K", [(5, 300, 264, 200), (5, 129, 64, 8), (6, 264, 520, 77),
                                           (6, 1000, 256, 1), (6, 8, 8, 300)])
def test_mn_major_ragged_k_matches_oracle(ws, variant, M, N, K):
    """A reduction length that is not a multiple of 64 (zero-filled tail)."""
    from serve_invariant_moe_gb300 import binding
    a = _rand((M, K), 40 + M + K)
    b = _rand((N, K), 41 + N + K, 0.05)
    if variant == 5:
        d = binding.gemm_bf16(a.cuda(), b.t().contiguous().cuda(), ws, variant=5)
    else:
        d = binding.gemm_bf16(a.t().contiguous().cuda(), b.t().contiguous().cuda(), ws, variant=6)
    binding.check_status(ws)
    a64, b64 = f64(a), f64(b)
    err = np.abs(d.double().cpu().numpy() - omoe.router_logits(a64, b64))
    bound = dot_bound(a64, b64, K)
    assert (err <= bound).all(), f"max err/bound {(err / bound).max():.3f}"


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_m64_tail_tiles_match_m128_tiles(ws, variant):
    """A last tile with at most 64 valid rows runs as an M = 64 MMA; the same rows inside a fuller
    tile run as M = 128.  Both give the same bits (the row-position invariance batch invariance needs)."""
    from serve_invariant_moe_gb300 import binding
    K, N = 320, 256
    a = _rand((600, K), 50)
    b = _rand((N, K), 51, 0.05).cuda()
    full = binding.gemm_bf16(a.cuda(), b, ws, variant=variant)          # tiles of 128 rows (tail 88 rows)
    for M in (129, 140, 192, 256 + 64, 512 + 1):                          # tails of 1, 12, 64, 64 and 1 rows
        d = binding.gemm_bf16(a[:M].contiguous().cuda(), b, ws, variant=variant)
        binding.check_status(ws)
        assert torch.equal(d, full[:M]), M
