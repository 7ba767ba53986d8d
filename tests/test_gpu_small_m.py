"""The small-M GEMM kernel (a router GEMM or shared expert of at most 64 tokens) against the engines
that compute the same rows inside a larger batch: every output bit must be the same
("位级一致：前沿训练的差异化关键", section "为什么比特级一致是一个复杂的问题": a token's result may not
depend on the batch it is computed in).  Cases cover a partial last 64-column tile (E = 72), a
reduction whose K blocks do not fill the last four-block copy (H = 448: 7 blocks), and the one-block
routing's token counts 1, 5, 33 and 64."""
import pytest
import torch

from serve_invariant_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return synth.to_bf16(synth.normal(shape, std, g)).cuda()


def _bits(t):
    return t.contiguous().view(torch.int32)


@pytest.mark.parametrize("H,E", [(256, 8), (448, 72), (6144, 256)])
def test_router_logits_of_small_batches_are_rows_of_a_large_batch(H, E):
    from serve_invariant_moe_gb300 import binding
    k = min(8, E)
    x = _bf16((200, H), 1.0, 1)
    wr = _bf16((E, H), 0.02, 2)
    ws = binding.new_workspace(binding.workspace_size(200, H, E, k), x.device)
    big = binding.moe_route_topk(x, wr, k, ws)          # 200 tokens: the row-tile engine
    big_logits = big["logits"].clone()
    for T, t0 in ((1, 0), (1, 199), (5, 17), (33, 100), (64, 136)):
        small = binding.moe_route_topk(x[t0:t0 + T].contiguous(), wr, k, ws)    # the small-M kernel
        torch.cuda.synchronize()
        assert torch.equal(_bits(small["logits"]), _bits(big_logits[t0:t0 + T])), (T, t0)
    binding.check_status(ws)


@pytest.mark.parametrize("H,Fs", [(256, 128), (448, 384), (6144, 2048)])
def test_shared_expert_of_small_batches_is_rows_of_a_large_batch(H, Fs):
    from serve_invariant_moe_gb300 import binding
    x = _bf16((200, H), 1.0, 3)
    ws13 = _bf16((2 * Fs, H), 0.02, 4)
    ws2 = _bf16((H, Fs), 0.02, 5)
    ws = binding.new_workspace(binding.workspace_size(200, H, F_shared=Fs), x.device)
    big = binding.moe_shared_expert(x, ws13, ws2, ws).clone()    # 200 tokens: the CTA-pair engine
    for T, t0 in ((1, 0), (1, 199), (5, 17), (33, 100), (64, 136)):
        small = binding.moe_shared_expert(x[t0:t0 + T].contiguous(), ws13, ws2, ws)   # the small-M kernel
        torch.cuda.synchronize()
        assert torch.equal(_bits(small), _bits(big[t0:t0 + T])), (T, t0)
    assert torch.isfinite(big).all() and big.abs().max() > 0
    binding.check_status(ws)
