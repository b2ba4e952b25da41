"""The E4M3 codec of the input module (FP8 operands of the FP8 variant): values
fixed by the E4M3 format definition (1 sign, 4 exponent bits with bias 7, 3
mantissa bits, no infinities, 0x7F NaN)."""
import numpy as np

import flce_inputs


def test_known_codes():
    d = flce_inputs.e4m3_decode
    assert d(np.array([0x00]))[0] == 0.0
    assert d(np.array([0x01]))[0] == 2.0 ** -9          # smallest subnormal
    assert d(np.array([0x07]))[0] == 7 * 2.0 ** -9      # largest subnormal
    assert d(np.array([0x08]))[0] == 2.0 ** -6          # smallest normal
    assert d(np.array([0x38]))[0] == 1.0
    assert d(np.array([0x3C]))[0] == 1.5
    assert d(np.array([0x7E]))[0] == 448.0              # largest finite
    assert d(np.array([0xB8]))[0] == -1.0
    assert np.isnan(d(np.array([0x7F]))[0]) and np.isnan(d(np.array([0xFF]))[0])


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = flce_inputs.e4m3_decode(codes)
    back = flce_inputs.e4m3_encode(vals)
    # -0 encodes as +0; every other code round-trips
    nz = vals != 0
    np.testing.assert_array_equal(back[nz], codes[nz])


def test_encode_rounds_to_nearest_with_ties_to_even_and_saturates():
    e = flce_inputs.e4m3_encode
    d = flce_inputs.e4m3_decode
    # between 1.0 (0x38) and 1.125 (0x39): 1.0625 is a tie -> even code 0x38
    assert e(np.array([1.0625]))[0] == 0x38
    assert e(np.array([1.07]))[0] == 0x39
    # between 1.125 (0x39) and 1.25 (0x3A): tie 1.1875 -> even code 0x3A
    assert e(np.array([1.1875]))[0] == 0x3A
    assert d(e(np.array([1e6])))[0] == 448.0
    assert d(e(np.array([-1e6])))[0] == -448.0
    x = np.random.default_rng(0).standard_normal(10000) * 50
    q = d(e(x))
    # nearest: no other finite value is strictly closer
    tab = flce_inputs.e4m3_table()
    allv = np.concatenate([-tab[::-1], tab])
    best = np.min(np.abs(allv[None, :] - np.clip(x, -448, 448)[:, None]), axis=1)
    np.testing.assert_allclose(np.abs(q - np.clip(x, -448, 448)), best, rtol=0, atol=1e-12)


def test_per_tensor_scale_maps_amax_to_448():
    H = flce_inputs.normal_bf16((64, 32), 2.0, 0, 1)
    codes, s = flce_inputs.to_fp8_per_tensor(H)
    deq = flce_inputs.e4m3_decode(codes) * np.float64(s)
    Hf = flce_inputs.bf16_bits_to_f64(H)
    assert np.max(np.abs(deq)) <= np.max(np.abs(Hf)) * (1 + 2 ** -4)
    assert np.max(np.abs(flce_inputs.e4m3_decode(codes))) == 448.0
    # relative error of E4M3 rounding is at most 2^-4 for normal values
    big = np.abs(Hf) > 2.0 ** -6 * float(s)
    assert np.max(np.abs(deq[big] - Hf[big]) / np.abs(Hf[big])) <= 2.0 ** -4 + 1e-12
