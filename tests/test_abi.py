"""CPU-side checks of the C ABI: the library builds, loads without a GPU and
exports every function include/invmoe.h declares; host-side validation."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|void)\s*\**\s*(\w+)\s*\(", src, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from serve_invariant_moe_gb300 import build, _lib
    build.build()
    return _lib.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("moe_route_topk", "moe_grouped_ffn", "moe_combine", "lm_logprob_kl",
              "invmoe_workspace_size", "invmoe_last_error", "invmoe_plan_len", "invmoe_check"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    from serve_invariant_moe_gb300 import _lib
    assert set(_lib.PROTOTYPES) == set(_declared())


def test_sizes(lib):
    assert lib.invmoe_plan_len(64, 8, 2) == 2 * 8 + 1 + 2 * 64 * 2
    ws = lib.invmoe_workspace_size(8192, 6144, 256, 8, 2048, 2048, 151552)
    assert ws >= 256 + 8192 * 592 * 8
    assert lib.invmoe_version() >= 100


def test_validation_rejects_before_any_launch(lib):
    # invalid arguments return an error code without touching the (absent) GPU
    null = None
    rc = lib.moe_route_topk(null, null, 64, 256, 8, 9, null, null, null, null, null, null, 0, null)
    assert rc == -1 and b"k <=" in lib.invmoe_last_error()
    rc = lib.moe_route_topk(null, null, 64, 100, 8, 2, null, null, null, null, null, null, 0, null)
    assert rc == -2
    rc = lib.moe_grouped_ffn(null, null, null, null, 64, 256, 8, 2, 96, null, null,
                             null, null, null, 0, null, null, 0, null)
    assert rc == -2 and b"F=96" in lib.invmoe_last_error()
    rc = lib.lm_logprob_kl(null, null, null, null, 4, 256, 4096, ctypes.c_float(0.5), null, null, null,
                           null, null, null, 0, null)
    assert rc == -1 and b"beta" in lib.invmoe_last_error()
    rc = lib.lm_logprob_kl(null, null, null, null, 4, 256, 4096, ctypes.c_float(2.0), null, null, null,
                           null, null, ctypes.c_void_p(256), 10, null)
    assert rc == -3
    rc = lib.invmoe_debug_timeout_probe(ctypes.c_void_p(256), 4096, 0, null)
    assert rc == -1
    # head backward: vocabulary not a multiple of 8, hidden not a multiple of 64, no workspace
    rc = lib.lm_head_backward(null, null, null, null, null, 4, 256, 1001, null, null, null, ctypes.c_void_p(256),
                              4096, null)
    assert rc == -2 and b"V=1001" in lib.invmoe_last_error()
    rc = lib.lm_head_backward(null, null, null, null, null, 4, 100, 1024, null, null, null, ctypes.c_void_p(256),
                              4096, null)
    assert rc == -2
    rc = lib.lm_head_backward(null, null, null, null, null, 4, 256, 1024, null, null, null, null, 0, null)
    assert rc == -1
    rc = lib.lm_head_backward(null, null, null, null, null, 4, 256, 1024, null, null, null, ctypes.c_void_p(256),
                              4096, null)
    assert rc == -1                                   # missing input pointers
    # MN-major GEMM test entry: shape rules of variants 5 and 6
    rc = lib.invmoe_gemm_bf16(null, null, 64, 64, 12, null, 5, ctypes.c_void_p(256), 4096, null)
    assert rc == -2
    rc = lib.invmoe_gemm_bf16(null, null, 12, 64, 64, null, 6, ctypes.c_void_p(256), 4096, null)
    assert rc == -2
    rc = lib.invmoe_gemm_bf16(null, null, 64, 64, 64, null, 7, ctypes.c_void_p(256), 4096, null)
    assert rc == -1


def _declared_arity():
    """Number of parameters of every function include/invmoe.h declares (comments stripped)."""
    out = {}
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|void)\s*\**\s*(\w+)\s*\(([^)]*)\)\s*;",
                             src, re.M | re.S):
            params = m.group(2).strip()
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_prototypes_match_the_header_arity():
    """The ctypes prototypes pass exactly as many arguments as the C declarations take: a
    drift between the two would hand a kernel wrong pointers."""
    from serve_invariant_moe_gb300 import _lib
    arity = _declared_arity()
    assert set(arity) == set(_lib.PROTOTYPES)
    for name, (_, args) in _lib.PROTOTYPES.items():
        assert len(args) == arity[name], (name, len(args), arity[name])


def test_binding_refuses_host_tensors_before_any_call():
    """The product path has no CPU fallback: host tensors are refused by the binding."""
    import torch
    from serve_invariant_moe_gb300 import binding
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    wr = torch.zeros(8, 64, dtype=torch.bfloat16)
    ws = torch.zeros(4096, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.moe_route_topk(x, wr, 2, ws)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.rl_token_loss(torch.zeros(4), torch.zeros(4), torch.zeros(4))
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.gemm_bf16(x, wr, ws)
