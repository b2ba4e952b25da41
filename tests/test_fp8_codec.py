"""Pins for the oracle's E4M3 reference (oracle/e4m3.py), which the FP8
variant's tests and the device quantiser's regression test use.

The codec is pinned by values the E4M3 format fixes (1 sign, 4 exponent bits
with bias 7, 3 mantissa bits, no infinities, 0x7F NaN) and by a brute-force
search over every finite code. The per-tensor quantisation is pinned by its
properties, not by a second copy of its steps: inv and scale are the float32
values nearest to 448 / amax and amax / 448, scale * 448 gives back amax within
one float32 ulp (normal scales), every code is
the E4M3 value nearest to fl32(x * inv) (ties to the even code), magnitudes at
or above 448 saturate, and zeros give +0."""
import numpy as np
import pytest

import flce_inputs
from oracle import e4m3


def test_known_codes():
    d = e4m3.e4m3_decode
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
    vals = e4m3.e4m3_decode(codes)
    back = e4m3.e4m3_encode(vals)
    # -0 encodes as +0; every other code round-trips
    nz = vals != 0
    np.testing.assert_array_equal(back[nz], codes[nz])


def test_encode_rounds_to_nearest_with_ties_to_even_and_saturates():
    e = e4m3.e4m3_encode
    d = e4m3.e4m3_decode
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
    tab = e4m3.e4m3_table()
    allv = np.concatenate([-tab[::-1], tab])
    best = np.min(np.abs(allv[None, :] - np.clip(x, -448, 448)[:, None]), axis=1)
    np.testing.assert_allclose(np.abs(q - np.clip(x, -448, 448)), best, rtol=0, atol=1e-12)


def _nearest_codes_brute_force(t):
    """For each value: the codes whose values are nearest to clip(t, +-448), with
    the even one (mantissa bit 0) taken on a tie; +0 for zero results."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and c != 0x80], dtype=np.int64)
    vals = e4m3.e4m3_decode(codes.astype(np.uint8))
    tc = np.clip(np.asarray(t, dtype=np.float64), -448.0, 448.0)
    dist = np.abs(vals[None, :] - tc[:, None])
    best = dist.min(axis=1, keepdims=True)
    out = np.empty(len(tc), dtype=np.int64)
    for k in range(len(tc)):
        cand = codes[dist[k] == best[k, 0]]
        even = cand[(cand & 1) == 0]
        out[k] = even[0] if len(even) else cand[0]
    return out.astype(np.uint8)


def _wide(shape, seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal(shape).astype(np.float32) * np.float32(10.0) ** g.uniform(-7, 1, shape).astype(np.float32)
    return flce_inputs.bf16_bits_to_f64(flce_inputs.f32_to_bf16_bits(x))


@pytest.mark.parametrize("case", ["normal", "wide", "subnormal", "zeros", "one"])
def test_per_tensor_quantisation_properties(case):
    if case == "normal":
        x = flce_inputs.bf16_bits_to_f64(flce_inputs.normal_bf16((64, 48), 0.05, 3, 0))
    elif case == "wide":
        x = _wide((97, 40), 4)
    elif case == "subnormal":   # amax ~1e-39: 448 / amax exceeds float32, inv is capped
        u = np.random.default_rng(7).uniform(-1, 1, (16, 40)).astype(np.float32) * np.float32(1e-39)
        x = flce_inputs.bf16_bits_to_f64(flce_inputs.f32_to_bf16_bits(u))
    elif case == "zeros":
        x = np.zeros((4, 8))
        x[1, 2] = -0.0
    else:
        x = np.full((1, 8), 3.0)
    r = e4m3.quantize_per_tensor(x)
    amax = float(np.max(np.abs(x)))
    assert float(r["amax"]) == amax
    if amax == 0.0:
        assert r["scale"] == 1.0 and r["inv"] == 1.0 and np.all(r["codes"] == 0)
        return
    inv = float(r["inv"])
    if 448.0 / amax <= float(np.finfo(np.float32).max):
        # the float32 nearest to 448 / amax: no float32 neighbour is closer
        q = 448.0 / amax
        assert abs(inv - q) <= abs(float(np.nextafter(r["inv"], np.float32(np.inf))) - q)
        assert abs(inv - q) <= abs(float(np.nextafter(r["inv"], np.float32(0))) - q)
    else:
        assert inv == float(np.finfo(np.float32).max)
    # scale is the float32 nearest to amax / 448; where it is a normal float32,
    # scale * 448 reproduces amax within one float32 ulp of amax
    q = amax / 448.0
    sc = float(r["scale"])
    assert abs(sc - q) <= abs(float(np.nextafter(r["scale"], np.float32(np.inf))) - q)
    assert abs(sc - q) <= abs(float(np.nextafter(r["scale"], np.float32(0))) - q)
    if sc >= float(np.finfo(np.float32).tiny):
        assert abs(sc * 448.0 - amax) <= float(np.spacing(np.float32(amax)))
    t = (x.astype(np.float32) * r["inv"]).astype(np.float32).ravel()
    np.testing.assert_array_equal(r["codes"].ravel(), _nearest_codes_brute_force(t))
    if inv < float(np.finfo(np.float32).max):
        # the largest magnitude lands on (or saturates to) 448
        assert np.max(np.abs(e4m3.e4m3_decode(r["codes"]))) == 448.0


def test_dequantised_values_within_e4m3_rounding_of_the_input():
    H = flce_inputs.normal_bf16((64, 32), 2.0, 0, 1)
    Hf = flce_inputs.bf16_bits_to_f64(H)
    r = e4m3.quantize_per_tensor(Hf)
    deq = e4m3.e4m3_decode(r["codes"]) * np.float64(r["scale"])
    assert np.max(np.abs(deq)) <= np.max(np.abs(Hf)) * (1 + 2 ** -4)
    # relative error of E4M3 rounding is at most 2^-4 for normal values
    big = np.abs(Hf) > 2.0 ** -6 * float(r["scale"])
    assert np.max(np.abs(deq[big] - Hf[big]) / np.abs(Hf[big])) <= 2.0 ** -4 + 1e-6
