"""Pins for the oracle's bf16 rounding (CPU only).

bf16 rounding has a plain definition (IEEE round-to-nearest-even into an
8-bit significand); torch's CPU ``Tensor.to(torch.bfloat16)`` is a library
routine for the same definition on fp32 inputs, so the oracle must agree with
it bit for bit.  The fp64 single-rounding case is pinned by a closed form.
"""
import numpy as np
import pytest
import torch

from oracle import bf16

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def torch_bits(f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(f32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def edge_values() -> np.ndarray:
    rng = np.random.default_rng(1)
    upper = rng.integers(0, 1 << 16, size=20000, dtype=np.uint32)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    u = (upper[:, None] << np.uint32(16)) | lows[None, :]
    vals = u.reshape(-1).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0,
                        np.float32(3.3895314e38), np.finfo(np.float32).max,
                        np.finfo(np.float32).tiny, np.float32(1e-45), np.float32(-1e-45)], dtype=np.float32)
    return np.concatenate([vals[np.isfinite(vals)], special])


def test_round_matches_library_on_fp32_edges():
    v = edge_values()
    np.testing.assert_array_equal(bf16.round_rne(v), torch_bits(v))


def test_round_matches_library_on_normals():
    v = np.random.default_rng(2).standard_normal(1 << 20).astype(np.float32) * 3.0
    np.testing.assert_array_equal(bf16.round_rne(v), torch_bits(v))


def test_widen_closed_forms():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x3F81, 0x0001], dtype=np.uint16)
    expect = np.array([1.0, -2.0, 0.0, -0.0, np.inf, 1.0 + 2.0 ** -7, 2.0 ** -133])
    got = bf16.widen64(bits)
    np.testing.assert_array_equal(got, expect)
    assert np.signbit(got[3])


def test_single_rounding_from_fp64():
    # 1 + 2^-8 + 2^-30 lies above the midpoint between 1 and 1 + 2^-7, so the
    # nearest bf16 is 1 + 2^-7 (0x3F81).  Going through fp32 first would land
    # exactly on the midpoint and round to even (1.0): the oracle must not.
    v = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30, -(1.0 + 2.0 ** -8 + 2.0 ** -30)])
    np.testing.assert_array_equal(bf16.round_rne(v), np.array([0x3F81, 0xBF81], dtype=np.uint16))
    # exact ties go to even
    t = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8])
    np.testing.assert_array_equal(bf16.round_rne(t), np.array([0x3F80, 0x3F82], dtype=np.uint16))


def test_overflow_and_nan():
    big = np.array([3.4e38, -3.4e38, 1e300, np.nan], dtype=np.float64)
    got = bf16.round_rne(big)
    assert got[0] == 0x7F80 and got[1] == 0xFF80 and got[2] == 0x7F80
    assert (got[3] & 0x7F80) == 0x7F80 and (got[3] & 0x007F) != 0
