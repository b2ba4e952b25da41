"""E4M3 operands for the FP8 variant: the codec and the per-tensor quantisation.
TEST INFRASTRUCTURE, like the rest of oracle/: only the tests, the package's
smoke check and the benchmark's CPU-baseline leg may use it; the product path
never does, and it shares no code with the CUDA quantiser.

Source: the GPU MODE lecture 28 notes close with open questions, one of them
whether the loss can use FP8 matrix units; the pages give no method. The
reading taken (the FP8 entry points and the device quantiser follow it):

  * E4M3 format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
    infinities, codes 0x7F and 0xFF are NaN; largest finite value 448, smallest
    subnormal 2^-9.
  * per-tensor scaling: amax = max_i |x_i|; scale = amax / 448 and
    inv = 448 / amax, each computed in float64 and rounded once to float32
    (inv capped at the largest finite float32; both 1 when amax == 0);
    q_i = e4m3(x_i * inv) with the product rounded to float32, then to the
    nearest E4M3 value (ties to the even code), saturating at +-448; a zero
    result is the code +0. The dequantised operand is scale * e4m3(q).

Pins (tests/test_fp8_codec.py): codes fixed by the format, a brute-force
nearest-value search over all finite codes, and the scaling properties
(inv is the float32 rounding of 448 / amax; scale * 448 reproduces amax to one
float32 ulp; every code is the E4M3 value nearest x * inv).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_F32_MAX = float(np.finfo(np.float32).max)


def e4m3_table() -> np.ndarray:
    """float64 value of each non-negative finite code 0x00..0x7E (index = code)."""
    codes = np.arange(0x7F)
    e = codes >> 3
    m = codes & 7
    return np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


def e4m3_decode(bits: np.ndarray) -> np.ndarray:
    """float64 values of E4M3 bytes (NaN codes decode to NaN)."""
    b = np.asarray(bits, dtype=np.uint8)
    tab = np.append(e4m3_table(), np.nan)
    v = tab[b & 0x7F]
    return np.where(b & 0x80, -v, v)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code of each value (ties to the even code), saturating at
    +-448; a result of zero is +0. Returns uint8 codes."""
    x = np.asarray(x, dtype=np.float64)
    tab = e4m3_table()
    a = np.minimum(np.abs(x), tab[-1])
    hi = np.clip(np.searchsorted(tab, a, side="left"), 1, len(tab) - 1)
    lo = hi - 1
    dlo = a - tab[lo]
    dhi = tab[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == tab[hi], hi, code).astype(np.uint8)
    return np.where(np.signbit(x) & (code != 0), code | 0x80, code).astype(np.uint8)


def scales(amax: float):
    """(scale, inv) as float32 for a tensor whose largest magnitude is amax."""
    amax = float(amax)
    if amax == 0.0:
        return np.float32(1.0), np.float32(1.0)
    return np.float32(amax / E4M3_MAX), np.float32(min(E4M3_MAX / amax, _F32_MAX))


def quantize_per_tensor(x: np.ndarray, block_rows: int = 8192) -> dict:
    """Per-tensor E4M3 quantisation of real values x (the exact values of a bf16
    tensor). Returns dict(codes uint8 [same shape], scale, inv, amax), the three
    scalars as float32."""
    x = np.asarray(x)
    flat = x.reshape(x.shape[0], -1) if x.ndim > 1 else x.reshape(1, -1)
    amax = 0.0
    for r0 in range(0, flat.shape[0], block_rows):
        amax = max(amax, float(np.max(np.abs(flat[r0:r0 + block_rows]), initial=0.0)))
    scale, inv = scales(amax)
    codes = np.empty(flat.shape, dtype=np.uint8)
    for r0 in range(0, flat.shape[0], block_rows):
        t = (flat[r0:r0 + block_rows].astype(np.float32) * inv).astype(np.float32)
        codes[r0:r0 + block_rows] = e4m3_encode(t.astype(np.float64))
    return dict(codes=codes.reshape(x.shape), scale=scale, inv=inv, amax=np.float32(amax))
