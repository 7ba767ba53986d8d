"""The bench's roofline arithmetic (host logic, no GPU): the algorithmic flops and bytes it divides by
kernel times, checked against hand-computed values for the GLM-scale step (T = 8192, H = 6144, E = 256,
k = 8, F = 2048, shared F = 2048, V = 151552)."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_work_table_glm_step():
    from serve_invariant_moe_gb300 import synth
    b = _bench()
    mc, hc = synth.GLM_MOE, synth.GLM_HEAD
    counts = np.full(mc.E, mc.T * mc.k // mc.E)
    w = b._work_table(mc, hc, counts)
    assert w["expert_gemm1_swiglu"] == ("tensor", 2.0 * 65536 * 4096 * 6144)         # 3.30e12
    assert w["expert_gemm2"] == ("tensor", 2.0 * 65536 * 6144 * 2048)                 # 1.65e12
    assert w["lm_head_gemm_lse"] == ("tensor", 2.0 * 8192 * 151552 * 6144)            # 1.53e13
    assert abs(w["lm_head_gemm_lse"][1] - 1.5256e13) / 1.5256e13 < 1e-3
    # permute: X read once (100.7 MB) + Xp written (805 MB) + the slot-row indices
    assert w["permute_rows"] == ("hbm", 8192 * 6144 * 2 + 65536 * 6144 * 2 + 65536 * 4)
    # combine: Y (1.61 GB) + y_shared + fp32 out + bf16 out + gates and slot rows
    assert w["combine"][1] == 65536 * 6144 * 4 + 2 * 8192 * 6144 * 4 + 8192 * 6144 * 2 + 8192 * 8 * 8
    # every expert in use: 256 experts x (2F + F) x H bf16 = 19.3 GB
    assert w["_expert_weight_bytes"][1] == 256 * 3 * 2048 * 6144 * 2
    w0 = b._work_table(mc, hc, np.zeros(mc.E, dtype=np.int64))
    assert w0["_expert_weight_bytes"][1] == 0


def test_gemm_bytes_glm_step():
    from serve_invariant_moe_gb300 import synth
    b = _bench()
    mc = synth.GLM_MOE
    counts = np.full(mc.E, mc.T * mc.k // mc.E)
    g = b._gemm_bytes(mc, counts)
    # the figures the bench line reported as `algorithmic_bytes`
    assert g["expert_gemm1_swiglu"] == 13958643712       # W13 12.88 GB + Xp 0.81 GB + h 0.27 GB
    assert g["expert_gemm2"] == 8321499136               # W2 6.44 GB + h 0.27 GB + Y 1.61 GB
    # roofline of a memory-bound GEMM: bytes over the copy bandwidth exceed flops over the bf16 peak
    t_flop = 2.0 * 65536 * 4096 * 6144 / 1921.1e12
    t_byte = g["expert_gemm1_swiglu"] / 6774.6e9
    assert t_byte > t_flop


def test_lm_head_traffic_is_tied_to_the_kernel_sources():
    b = _bench()
    # the captured figure is reported only while the sources it was captured from are unchanged
    t = b.TRAFFIC["lm_head_gemm_lse"]
    if t["bytes"] is None:
        assert b.traffic_bytes("lm_head_gemm_lse") is None
    else:
        # read + write of one full-size launch: above the 1.96 GB of algorithmic bytes (Wv, hidden,
        # partials) and far below the 26.9 GB of an unbanded column order
        assert 1.96e9 < t["bytes"] < 10e9
        want = t["bytes"] if t["sources_sha256"] == b.kernel_sources_sha256() else None
        assert b.traffic_bytes("lm_head_gemm_lse") == want
    assert b.traffic_bytes("no_such_kernel") is None
    assert len(b.kernel_sources_sha256()) == 64


def test_head_algorithmic_bytes():
    from serve_invariant_moe_gb300 import synth
    b = _bench()
    # Wv 1.862 GB + hidden 100.7 MB + partials 8192 x 592 x 8 B + target logits
    got = b._head_bytes(synth.GLM_MOE, synth.GLM_HEAD)
    assert got == 151552 * 6144 * 2 + 8192 * 6144 * 2 + 8192 * 592 * 8 + 8192 * 4
