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


def test_binding_refuses_wrong_caller_buffers():
    """Caller-provided buffers of the wrong shape or dtype are refused on the host, before any
    kernel could write past them."""
    from serve_invariant_moe_gb300 import binding
    T, H, V, E, k = 64, 128, 512, 8, 2
    dev = "cuda"
    ws = binding.new_workspace(binding.workspace_size(T, H, E, k, 128, 0, V), dev)
    hidden = torch.zeros(T, H, dtype=torch.bfloat16, device=dev)
    wv = torch.zeros(V, H, dtype=torch.bfloat16, device=dev)
    target = torch.zeros(T, dtype=torch.int32, device=dev)
    with pytest.raises(ValueError, match="logp"):
        binding.lm_logprob_kl(hidden, wv, target, ws, logp=torch.empty(T - 1, device=dev))
    with pytest.raises(ValueError, match="mask"):
        binding.lm_logprob_kl(hidden, wv, target, ws, rollout_logp=torch.zeros(T, device=dev),
                              mask=torch.empty(T, dtype=torch.int32, device=dev))
    x = torch.zeros(T, H, dtype=torch.bfloat16, device=dev)
    wr = torch.zeros(E, H, dtype=torch.bfloat16, device=dev)
    idx = torch.zeros(T, k, dtype=torch.int32, device=dev)
    w = torch.zeros(T, k, dtype=torch.float32, device=dev)
    dxp = torch.zeros(T * k, H, dtype=torch.float32, device=dev)
    small_plan = torch.zeros(binding.plan_len(T, E, k) - 1, dtype=torch.int32, device=dev)
    with pytest.raises(ValueError, match="plan"):
        binding.moe_route_backward(x, wr, idx, w, w, dxp, small_plan, ws)
    plan = torch.zeros(binding.plan_len(T, E, k), dtype=torch.int32, device=dev)
    with pytest.raises(ValueError, match="dw_router"):
        binding.moe_route_backward(x, wr, idx, w, w, dxp, plan, ws, dw_router=torch.empty(E, H - 8, device=dev))
    y = torch.zeros(T * k, H, dtype=torch.float32, device=dev)
    dout = torch.zeros(T, H, dtype=torch.float32, device=dev)
    with pytest.raises(ValueError, match="dy"):
        binding.moe_combine_backward(dout, y, w, plan, E, k, dy=torch.empty(T * k, H, device=dev))
    torch.cuda.synchronize()
