"""Pins of the oracle's FP8 projection operands (Engram notes 3.4: the fused W_V + M W_K GEMM
runs in FP8; reading R16: OCP E4M3 rows with one fp32 absmax scale per row).

Pinned against torch's float8_e4m3fn conversions (IEEE-style round to nearest even) and
against what the format and the absmax rule fix: zero rows, the largest element landing
on +-448, and the rounding bound of a 3-bit mantissa.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc


def test_e4m3_encoding_matches_torch_below_the_saturation_point():
    rng = np.random.default_rng(31)
    vals = np.concatenate([
        (2.0 ** rng.uniform(-12, 9, 5000) * rng.choice([-1, 1], 5000)).astype(np.float32),
        np.float32([0.0, -0.0, 448.0, 464.0, -464.0, 2.0 ** -6, 2.0 ** -9, 2.0 ** -10, 1.5 * 2.0 ** -10]),
    ])
    # exact ties: midpoints of adjacent positive E4M3 values
    pos = orc.e4m3_to_f32(np.arange(0, 0x7E, dtype=np.uint8))
    vals = np.concatenate([vals, ((pos[:-1] + pos[1:]) / 2).astype(np.float32)])
    vals = vals[np.abs(vals) <= 464]               # above, torch overflows to NaN and R16 saturates
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([orc.f32_to_e4m3_sat(v) for v in vals], np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_where_torch_overflows():
    for v in (465.0, 500.0, 1e9, float("inf")):
        assert orc.f32_to_e4m3_sat(v) == 0x7E and orc.f32_to_e4m3_sat(-v) == 0xFE


def test_e4m3_decoding_matches_torch_for_every_byte():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    ours = orc.e4m3_to_f32(b)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_fp8_rows_zero_row_and_extremes():
    x = np.zeros((3, 128), np.float32)
    x[1, 17] = -3.5
    x[2] = np.linspace(-1, 2, 128, dtype=np.float32)
    q, s = orc.fp8_quantize(x)
    assert s[0] == 0 and (q[0] == 0).all()
    assert q[1, 17] == 0xFE and s[1] == np.float32(3.5) / np.float32(448)   # the absmax lands on -448
    assert q[2, 127] == 0x7E
    assert (orc.fp8_dequantize(q, s)[0] == 0).all()


@pytest.mark.parametrize("dist", ["normal", "heavy", "tiny", "wide"])
def test_fp8_rows_error_within_the_rounding_bound(dist):
    # a normal E4M3 value carries 3 mantissa bits: |y - e4m3(y)| <= 2^-4 |y| for |y| >= 2^-6,
    # and <= 2^-10 (half the subnormal step) below; scaled back by s
    rng = np.random.default_rng(32)
    x = {"normal": rng.standard_normal((200, 256)),
         "heavy": rng.standard_t(1.2, (200, 256)),
         "tiny": rng.standard_normal((200, 256)) * 1e-30,
         "wide": rng.standard_normal((200, 256)) * 10.0 ** rng.uniform(-8, 8, (200, 1))}[dist].astype(np.float32)
    q, s = orc.fp8_quantize(x)
    deq = orc.fp8_dequantize(q, s)
    bound = 2.0 ** -4 * np.abs(x.astype(np.float64)) + 2.0 ** -10 * s.astype(np.float64)[:, None] * (1 + 1e-6)
    assert (np.abs(deq - x) <= bound + 1e-45).all()
    assert np.allclose(np.abs(deq).max(axis=1), np.abs(x).max(axis=1), rtol=2.0 ** -4)
