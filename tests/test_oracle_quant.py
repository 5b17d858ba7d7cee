"""Pins for the oracle's dynamic e4m3 quantisers (per tensor, per row and
128-column group).

The expected codes follow from the OCP e4m3 definition (sign, 4 exponent bits with
bias 7, 3 mantissa bits; 448 = 0x7E is the largest finite value) and from the
scale rule s = amax / 448 in fp32 (s = 1 for an all-zero tensor or group), worked
out by hand here, not by calling the oracle's encoder."""
import numpy as np
import pytest

from oracle import moe as O

# codes of a few values, from the format definition
C_448 = 0x7E    # 1.75 * 2^8: exponent field 15, mantissa 110
C_1 = 0x38      # exponent field 7, mantissa 000
C_M1 = 0xB8     # sign bit + C_1
C_1125 = 0x39   # 1 + 1/8
C_125 = 0x3A    # 1 + 2/8
C_HALF = 0x30   # exponent field 6
C_0 = 0x00


def test_scale_rule_and_zero_tensor():
    assert O.scale_of(np.float32(896.0)) == np.float32(2.0)
    assert O.scale_of(np.float32(0.0)) == np.float32(1.0)
    codes, s = O.quant_per_tensor(np.zeros((3, 5), dtype=np.float32))
    assert s == np.float32(1.0) and np.all(codes == C_0)


def test_per_tensor_codes_from_the_definition():
    # amax 896 -> s = 2: 896 -> 448, -2 -> -1, 1 -> 0.5, 2.25 -> 1.125
    v = np.array([896.0, -2.0, 1.0, 2.25], dtype=np.float32)
    codes, s = O.quant_per_tensor(v)
    assert s == np.float32(2.0)
    assert codes.tolist() == [C_448, C_M1, C_HALF, C_1125]


def test_per_tensor_ties_to_even_after_scaling():
    # amax 448 -> s = 1; 1.0625 lies halfway between 1 (even mantissa) and 1.125,
    # 1.1875 halfway between 1.125 and 1.25 (even): both round to the even neighbour
    v = np.array([448.0, 1.0625, 1.1875, -1.0625], dtype=np.float32)
    codes, s = O.quant_per_tensor(v)
    assert s == np.float32(1.0)
    assert codes.tolist() == [C_448, C_1, C_125, 0x80 | C_1]


def test_amax_element_saturates_to_the_largest_code():
    # s = amax / 448 is rounded to fp32, so amax / s may land just above 448: the
    # encoding saturates to 448 rather than overflowing
    for amax in (1.0, 3.0, 7.3, 1e-3, 123.456):
        codes, _ = O.quant_per_tensor(np.array([amax, -amax], dtype=np.float32))
        assert codes.tolist() == [C_448, 0x80 | C_448]


def test_per_group_scales_and_ragged_last_group():
    # one row of 260 columns: groups [0,128) max 896 (s=2), [128,256) all zero
    # (s=1), and a ragged last group [256,260) with max 1 (s=1/448)
    v = np.zeros((1, 260), dtype=np.float32)
    v[0, 5], v[0, 6], v[0, 7] = 896.0, -2.0, 2.25
    v[0, 256], v[0, 259] = 1.0, -0.5
    codes, scales = O.quant_per_group(v, 128)
    assert scales.shape == (1, 3)
    assert scales[0, 0] == np.float32(2.0) and scales[0, 1] == np.float32(1.0)
    assert scales[0, 2] == np.float32(1.0) / np.float32(448.0)
    assert codes[0, 5] == C_448 and codes[0, 6] == C_M1 and codes[0, 7] == C_1125
    assert np.all(codes[0, 128:256] == C_0)
    assert codes[0, 256] == C_448
    # -0.5 / (1/448) = -224 = -1.75 * 2^7: exponent field 14, mantissa 110
    assert codes[0, 259] == (0x80 | 0x76)


@pytest.mark.parametrize("rows", [1, 4])
def test_per_group_rows_are_independent(rows):
    # each row takes its own scale: row r has max 2^r * 448
    v = np.array([[448.0 * 2 ** r, 2.0 ** r] + [0.0] * 126 for r in range(rows)], dtype=np.float32)
    codes, scales = O.quant_per_group(v, 128)
    for r in range(rows):
        assert scales[r, 0] == np.float32(2.0 ** r)
        assert codes[r, 0] == C_448 and codes[r, 1] == C_1
