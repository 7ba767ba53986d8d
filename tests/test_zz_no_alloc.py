"""moe_route_topk_noalloc: the routing call for callers that cannot allocate device
memory (its scratch is a fixed array inside the library).  Checked through the C
ABI against the regular moe_route_topk, which takes a caller-allocated workspace,
on two calls in a row (the second call reuses the scratch the first one left)."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(T, E, k, H, plan_len):
    return dict(logits=torch.empty((T, E), dtype=torch.float32, device="cuda"),
                idx=torch.empty((T, k), dtype=torch.int32, device="cuda"),
                w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
                plan=torch.empty(plan_len, dtype=torch.int32, device="cuda"),
                xp=torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda"))


def test_noalloc_routing_matches_workspace_routing_twice():
    from serve_invariant_moe_gb300 import _lib, build
    build.build()
    lib = _lib.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (T, H, E, k, seed) in enumerate([(1000, 256, 64, 6, 1), (333, 512, 128, 8, 2)]):
        g = torch.Generator().manual_seed(seed)
        x = torch.randn((T, H), generator=g).to(torch.bfloat16).cuda()
        wr = (torch.randn((E, H), generator=g) * 0.05).to(torch.bfloat16).cuda()
        n = lib.invmoe_plan_len(T, E, k)
        ref = _outputs(T, E, k, H, n)
        got = _outputs(T, E, k, H, n)
        ws = torch.zeros(lib.invmoe_workspace_size(T, H, E, k, 0, 0, 0), dtype=torch.uint8, device="cuda")
        rc = lib.moe_route_topk(_ptr(x), _ptr(wr), T, H, E, k, _ptr(ref["logits"]), _ptr(ref["idx"]),
                                _ptr(ref["w"]), _ptr(ref["plan"]), _ptr(ref["xp"]), _ptr(ws), ws.numel(), stream)
        assert rc == 0, lib.invmoe_last_error()
        status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
        rc = lib.moe_route_topk_noalloc(_ptr(x), _ptr(wr), T, H, E, k, _ptr(got["logits"]), _ptr(got["idx"]),
                                        _ptr(got["w"]), _ptr(got["plan"]), _ptr(got["xp"]), _ptr(status), stream)
        assert rc == 0, lib.invmoe_last_error()
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device status {status.item()}"
        for key in ref:
            a, b = ref[key], got[key]
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"call {call}: {key} differs"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from serve_invariant_moe_gb300 import _lib, build
    build.build()
    lib = _lib.lib()
    # ceil(T/64) * E = 2048 * 256 = 524288 > 262144: rejected before anything is launched
    rc = lib.moe_route_topk_noalloc(None, None, 131072, 256, 256, 8, None, None, None, None, None, None, None)
    assert rc == -2 and b"fixed scratch" in lib.invmoe_last_error()
