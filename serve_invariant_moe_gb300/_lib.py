"""ctypes loader for libinvmoe.so (the in-tree C ABI declared in include/invmoe.h).

There is no fallback: if the shared library is missing or fails to load, every
call raises.  Build it with ``serve_invariant_moe_gb300.build.build()``.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libinvmoe.so")

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_f = ctypes.c_float

# name -> (restype, argtypes); mirrors include/invmoe.h
PROTOTYPES = {
    "invmoe_version": (_i, []),
    "invmoe_last_error": (ctypes.c_char_p, []),
    "invmoe_plan_len": (_sz, [_i, _i, _i]),
    "invmoe_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "invmoe_check": (_i, [_vp, _vp]),
    "moe_route_topk": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_route_topk_noalloc": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_route_replay": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_grouped_ffn": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp,
                             _vp, _vp, _vp, _i, _vp, _vp, _sz, _vp]),
    "moe_combine": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp]),
    "moe_layer_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                               _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lm_logprob_kl": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lm_logprob_partials": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, ctypes.c_longlong, _vp, _vp, _sz,
                                 _vp]),
    "lm_logprob_merge": (_i, [_vp, ctypes.c_longlong, _i, ctypes.c_longlong, _vp, ctypes.c_longlong, _vp, _vp, _i,
                              _i, _f, _vp, _vp, _vp, _vp, _vp]),
    "moe_ep_regroup": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_ep_ungroup": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "moe_shared_expert": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "rl_token_loss": (_i, [_vp, _vp, _vp, _vp, _i, _f, _f, _f, _vp, _vp, _vp, _vp, _vp, _vp]),
    "lm_head_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "invmoe_backward_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "moe_combine_backward": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "moe_grouped_ffn_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_route_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _sz,
                                _vp]),
    "invmoe_gemm_bf16": (_i, [_vp, _vp, _i, _i, _i, _vp, _i, _vp, _sz, _vp]),
    "invmoe_debug_timeout_probe": (_i, [_vp, _sz, _i, _vp]),
    "invmoe_profile_enable": (_i, [_i]),
    "invmoe_pdl_enable": (_i, [_i]),
    "invmoe_expert_engine": (_i, [_i]),
    "invmoe_shared_overlap": (_i, [_i]),
    "invmoe_profile_collect": (_i, [ctypes.c_char_p, ctypes.POINTER(_f), ctypes.POINTER(_i), _i]),
}

ERRORS = {
    -1: "INVALID_ARG",
    -2: "UNSUPPORTED_SHAPE",
    -3: "WORKSPACE_TOO_SMALL",
    -4: "MISALIGNED",
    -5: "CUDA",
    -6: "DEVICE_TIMEOUT",
}

_lib = None


class InvmoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"invmoe error {code} ({ERRORS.get(code, '?')}): {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libinvmoe.so once and declare its prototypes."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run serve_invariant_moe_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(rc: int):
    if rc != 0:
        raise InvmoeError(rc, lib().invmoe_last_error().decode(errors="replace"))
