"""Pins of the oracle's NF4 export (PageGram report 3.3 storage format; report 9.4, check 5:
all-zero rows keep full fidelity and the quantisation error stays within its bound).

The quantiser is QLoRA's absmax rule (reading R15): scale = fp16(max |x|), code = the
nearest NF4 level of x / scale. The pins below come from the pages and from mathematics,
not from retyping the rule: fp16 rounding against numpy's IEEE conversion, the zero row,
rows built from exact levels, the error bound, idempotence through the stored format.
"""
import numpy as np
import pytest

from oracle import oracle as orc


def _levels():
    return orc.nf4_levels().astype(np.float64)


def test_fp16_scale_rounding_matches_ieee_conversion():
    # numpy's float32 -> float16 cast is IEEE round-to-nearest-even; the oracle's
    # conversion is written from the format definition and must agree everywhere
    # except past 65504, where the reading saturates instead of producing infinity
    rng = np.random.default_rng(11)
    exps = rng.uniform(-30, 17, 4000)
    vals = (2.0 ** exps * rng.uniform(1, 2, exps.size)).astype(np.float32)
    # exact ties: midpoints of adjacent fp16 values (exact in fp32)
    h = rng.integers(1, 0x7BFE, 2000).astype(np.uint16)
    lo, hi = h.view(np.float16).astype(np.float32), (h + 1).view(np.float16).astype(np.float32)
    vals = np.concatenate([vals, (lo + hi) / 2, lo, np.float32([0, 65504, 65519.996, 6.1035156e-05])])
    for v in vals:
        with np.errstate(over="ignore"):
            ref = np.float32(v).astype(np.float16)
        want = 0x7BFF if np.isinf(ref) else int(ref.view(np.uint16))
        assert orc.f32_to_f16_sat(v) == want, (float(v), hex(want))
    assert orc.f32_to_f16_sat(65520.0) == 0x7BFF and orc.f32_to_f16_sat(1e30) == 0x7BFF


def test_zero_row_is_exact():
    rows = orc.nf4_quantize(np.zeros((3, 64), np.float32))
    assert (rows[:, :32] == 0x77).all() and (rows[:, 32:] == 0).all()   # code 7 = the zero level
    assert (orc.nf4_dequantize(rows) == 0).all()
    assert _levels()[7] == 0.0


def test_rows_of_exact_levels_return_their_codes():
    # x = level[c] * s with the row's absmax equal to s (an extreme level present):
    # the nearest level of x / s is level[c] itself
    rng = np.random.default_rng(12)
    lv = orc.nf4_levels()
    for s in (1.0, 0.375, 3.0, 1000.0, 2.0 ** -10):
        codes = rng.integers(0, 16, (20, 64))
        codes[:, 5] = 15                                 # level +1: absmax = s
        x = (lv[codes] * np.float32(s)).astype(np.float32)
        rows = orc.nf4_quantize(x)
        got = np.empty_like(codes)
        got[:, 0::2] = rows[:, :32] & 15
        got[:, 1::2] = rows[:, :32] >> 4
        assert (got == codes).all()
        assert (orc.nf4_dequantize(rows) == x).all()


def test_exact_ties_between_two_levels_take_the_lower_code():
    # Reading R15 breaks a tie between two equally near levels toward the lower code. Exact
    # ties: with the row's absmax 1.0 the scale is fp16(1.0) = 1, and half of the level next
    # to zero lies exactly half-way between it and the zero level (halving is exact in fp32)
    lv = orc.nf4_levels()
    assert lv[7] == 0.0
    x = np.zeros((1, 64), np.float32)
    x[0, 0] = 1.0
    x[0, 1] = lv[8] / np.float32(2)      # between level 7 (zero) and level 8
    x[0, 2] = lv[6] / np.float32(2)      # between level 6 and level 7 (zero)
    rows = orc.nf4_quantize(x)
    assert rows[0, 0] == 15 | (7 << 4)   # codes of elements 0 and 1
    assert rows[0, 1] & 15 == 6          # element 2


@pytest.mark.parametrize("dist", ["normal", "uniform", "heavy", "tiny", "huge", "sparse"])
def test_error_within_the_quantisation_bound(dist):
    # |x - dequant(x)| <= s * g / 2 + |a - s| (+ fp32 rounding of x / s), with a = max |x|,
    # s the stored scale and g the widest gap between adjacent levels: the nearest level
    # of a value inside [-a/s, a/s] is at most half a gap away, and values beyond +-1
    # (scale rounded below a) are at most a - s past the extreme level
    rng = np.random.default_rng(13)
    n = 300
    x = {"normal": rng.standard_normal((n, 64)),
         "uniform": rng.uniform(-1, 1, (n, 64)),
         "heavy": rng.standard_t(1.5, (n, 64)),
         "tiny": rng.standard_normal((n, 64)) * 1e-6,
         "huge": rng.standard_normal((n, 64)) * 1e4,
         "sparse": rng.standard_normal((n, 64)) * (rng.random((n, 64)) < 0.05)}[dist].astype(np.float32)
    rows = orc.nf4_quantize(x)
    deq = orc.nf4_dequantize(rows).astype(np.float64)
    lv = _levels()
    g = np.diff(lv).max()
    a = np.abs(x).max(axis=1).astype(np.float64)
    sbits = rows[:, 32].astype(np.uint16) | (rows[:, 33].astype(np.uint16) << 8)
    s = sbits.view(np.float16).astype(np.float64)
    bound = s * g / 2 + np.abs(a - s) + 4e-7 * np.maximum(a, s)
    err = np.abs(deq - x.astype(np.float64)).max(axis=1)
    assert (err <= bound).all(), float((err - bound).max())


def test_export_is_idempotent_through_the_stored_format():
    # dequantising and exporting again reproduces the same bytes: the largest element
    # maps to an extreme level (+-1), so the second scale equals the first and every
    # value is a level times it
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((200, 64)) * rng.uniform(1e-3, 1e3, (200, 1))).astype(np.float32)
    rows = orc.nf4_quantize(x)
    again = orc.nf4_quantize(orc.nf4_dequantize(rows))
    assert (again == rows).all()


def test_nibble_order_and_scale_bytes():
    # element 2i in the low nibble of byte i, 2i+1 in the high nibble; scale little-endian
    lv = orc.nf4_levels()
    x = np.zeros((1, 64), np.float32)
    x[0, 0], x[0, 1], x[0, 63] = lv[3] * 2, lv[12] * 2, 2.0    # absmax 2 -> scale 0x4000
    rows = orc.nf4_quantize(x)
    assert rows[0, 0] == (3 | (12 << 4)) and rows[0, 31] == (7 | (15 << 4))
    assert rows[0, 32] == 0x00 and rows[0, 33] == 0x40
