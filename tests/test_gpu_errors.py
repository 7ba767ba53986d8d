"""Failure detection without a GPU fault: a bounded device wait that runs out is
reported through the status word, and the context stays usable afterwards."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from serve_invariant_moe_gb300 import build
    build.build()


def test_timeout_is_reported_and_context_survives():
    from serve_invariant_moe_gb300 import binding
    from serve_invariant_moe_gb300._lib import InvmoeError
    ws = binding.new_workspace(4096)
    binding.check_status(ws)                        # clean
    binding.debug_timeout_probe(ws, timeout_us=20000)
    with pytest.raises(InvmoeError) as e:
        binding.check_status(ws)
    assert e.value.code == -6
    binding.check_status(ws)                        # cleared by the read
    # the context still works: a GEMM runs and is correct
    a = torch.randn(130, 128).to(torch.bfloat16).cuda()
    b = torch.randn(64, 128).to(torch.bfloat16).cuda()
    d = binding.gemm_bf16(a, b, ws, variant=3)
    binding.check_status(ws)
    ref = a.double() @ b.double().T
    assert torch.allclose(d.double(), ref, rtol=1e-4, atol=1e-3)


def test_host_validation_errors_raise():
    from serve_invariant_moe_gb300 import binding
    from serve_invariant_moe_gb300._lib import InvmoeError
    ws = binding.new_workspace(4096)
    a = torch.zeros(16, 100, dtype=torch.bfloat16, device="cuda")   # K not a multiple of 64
    b = torch.zeros(8, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(InvmoeError) as e:
        binding.gemm_bf16(a, b, ws)
    assert e.value.code == -2
    x = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros(8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(InvmoeError) as e:
        binding.moe_route_topk(x, wr, 2, torch.zeros(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -3
