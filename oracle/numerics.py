"""Element formats of the cache, decoded and encoded exactly in fp64.

Sources:
  * bf16: IEEE-754 binary32 with the low 16 mantissa bits dropped; a bf16 bit
    pattern ``u`` is the binary32 pattern ``u << 16``.
  * fp8 E4M3: the OCP 8-bit floating point specification (OFP8, "E4M3"):
    1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities; S.1111.111
    is NaN; the largest finite magnitude is 448 (S.1111.110). Subnormals
    (exponent field 0) are m/8 * 2^-6. "KV cache", section "Fewer bits per
    number", names fp8 as the default cache precision; the 448 maximum is the
    one "890 bytes a token ...", section 6, multiplies by 6 to get 2688.

Parity: pinned (tests/test_oracle_pins.py: closed-form codes, library
conversions for in-range values, exhaustive round trip, midpoints).
"""
import numpy as np


def bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16) -> exact float64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def e4m3_value_table():
    """float64 value of each of the 256 E4M3 codes (NaN for S.1111.111)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        mant = code & 0x7
        if exp_field == 0xF and mant == 0x7:
            vals[code] = np.nan
        elif exp_field == 0:
            vals[code] = sign * (mant / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)
    return vals


_E4M3 = e4m3_value_table()
_E4M3_POS = _E4M3[:127]          # codes 0x00..0x7E, strictly increasing


def e4m3_codes_to_f64(codes):
    """uint8 E4M3 codes -> exact float64 values."""
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_f32(x):
    """Encode float32 values as E4M3 codes: round to nearest, ties to even,
    saturating to +-448 ("satfinite"): any magnitude >= 448, infinities
    included, becomes the largest finite code. NaN stays NaN (S.1111.111).
    The sign is kept, so a negative value that rounds to zero gives 0x80.
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    # largest code whose value is <= a (a < 448 here)
    lo = np.searchsorted(_E4M3_POS, a, side="right") - 1
    lo = np.clip(lo, 0, 125)
    v_lo = _E4M3_POS[lo]
    v_hi = _E4M3_POS[lo + 1]
    d_lo = a - v_lo
    d_hi = v_hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo & 1) == 1))
    mag = np.where(pick_hi, lo + 1, lo).astype(np.uint8)
    mag = np.where(a >= 448.0, np.uint8(0x7E), mag)
    out = (mag | sign).astype(np.uint8)
    out = np.where(np.isnan(x), (np.uint8(0x7F) | sign), out).astype(np.uint8)
    return out
