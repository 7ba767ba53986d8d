"""Pins for oracle.numerics: bf16 widening / narrowing against PyTorch's conversions,
and the non-associativity example the pages use to motivate the whole method."""
import numpy as np
import torch

from oracle.numerics import bf16_bits_to_f64, f64_to_bf16_bits, round_to_bf16


def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_non_associativity_example():
    # Bit-agreement page, "为什么比特级一致是一个复杂的问题": (a + b) + c differs
    # from a + (b + c) in the last bits.  Constructed float32 triple:
    a = np.float32(1.0)
    b = c = np.float32(2.0 ** -24)
    left = np.float32(np.float32(a + b) + c)
    right = np.float32(a + np.float32(b + c))
    assert left == np.float32(1.0)
    assert right == np.float32(1.0 + 2.0 ** -23)
    assert left != right


def test_widen_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 16, size=20000, dtype=np.uint32).astype(np.uint16)
    ours = bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_round_matches_torch_on_float32_values():
    # float32 inputs are exact in float64, so torch's single float32->bf16
    # rounding (nearest even) is the reference for the same single rounding.
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(50000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),      # subnormals
        np.clip(rng.standard_normal(5000) * 3e38, -3.4e38, 3.4e38).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                  -(1.0 + 2 ** -8), 3.3895313892515355e38], np.float32),
    ])
    ours = f64_to_bf16_bits(x.astype(np.float64))
    ref = _torch_bf16_bits(x)
    assert np.array_equal(ours, ref)


def test_round_half_even_hand_cases():
    # 1 + 2^-8 sits halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert round_to_bf16(1.0 + 2 ** -8) == 1.0
    # 1 + 3*2^-8 sits halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert round_to_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6
    # just above the halfway point rounds up
    assert round_to_bf16(1.0 + 2 ** -8 + 2 ** -30) == 1.0 + 2 ** -7
    # a float64 value that is not a float32: rounding must be single-step
    v = 1.0 + 2 ** -8 + 2 ** -40        # float32 would round this to 1 + 2^-8 (a tie)
    assert round_to_bf16(v) == 1.0 + 2 ** -7
    assert np.signbit(round_to_bf16(-0.0))
    assert np.isnan(round_to_bf16(np.nan))
