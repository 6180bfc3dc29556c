"""Element formats of the cache, decoded and encoded exactly in fp64.

TEST INFRASTRUCTURE (see the package docstring).

Sources:
  * bf16: IEEE-754 binary32 with the low 16 mantissa bits dropped; a bf16 bit
    pattern ``u`` is the binary32 pattern ``u << 16``.
  * fp8 E4M3: the OCP 8-bit floating point specification (OFP8, "E4M3"):
    1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities; S.1111.111
    is NaN; the largest finite magnitude is 448 (S.1111.110). Subnormals
    (exponent field 0) are m/8 * 2^-6. "KV cache", section "Fewer bits per
    number", names fp8 as the default cache precision; the 448 maximum is the
    one "890 bytes a token ...", section 6, multiplies by 6 to get 2688.

  * fp4 E2M1: the OCP Microscaling Formats (MX) specification, "FP4 (E2M1)":
    1 sign, 2 exponent (bias 1), 1 mantissa bit; no infinities or NaN;
    exponent field 0 holds the subnormal m * 0.5; magnitudes 0, 0.5, 1, 1.5,
    2, 3, 4, 6.
  * MXFP4 cache rows ("890 bytes a token ...", section 6: E2M1 with one
    E4M3 scale per 16 channels, NVFP4's layout without its second-level
    global scale, so the largest value is 448 x 6 = 2688). The encoder's
    rule for choosing the scale and rounding is this repository's reading of
    that sentence (the page gives none): per 16-channel group, scale =
    E4M3(amax / 6) and code = E2M1(x / scale), each rounded to nearest even
    and saturated, the divisions in fp32; a group whose scale rounds to 0
    stores all-zero codes.

Parity: pinned (tests/test_oracle_pins.py: closed-form codes, library
conversions for in-range values, exhaustive round trip, midpoints; E2M1:
the OCP value list, round trip, every midpoint, saturation and sign; MXFP4:
exact round trip of scaled grid values, the 2688 bound, the per-element
error bound, the page's size figure against fp8).
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


# ---------------------------------------------------------------------------
# fp4 E2M1 and MXFP4 rows
# ---------------------------------------------------------------------------
def e2m1_value_table():
    """float64 value of each of the 16 E2M1 codes (code 8 is -0)."""
    vals = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        exp_field = (code >> 1) & 0x3
        mant = code & 0x1
        if exp_field == 0:
            vals[code] = sign * mant * 0.5
        else:
            vals[code] = sign * (1.0 + mant / 2.0) * 2.0 ** (exp_field - 1)
    return vals


_E2M1 = e2m1_value_table()
_E2M1_POS = _E2M1[:8]            # codes 0..7, strictly increasing


def e2m1_codes_to_f64(codes):
    """uint8 E2M1 codes (low 4 bits) -> exact float64 values."""
    return _E2M1[np.asarray(codes, dtype=np.uint8) & np.uint8(0xF)]


def e2m1_encode_f32(x):
    """Encode float32 values as E2M1 codes: round to nearest, ties to the
    code with mantissa bit 0, saturating to +-6 (anything >= 6 in
    magnitude, infinities and NaN included, becomes the largest code). The
    sign is kept, so a negative value that rounds to zero gives 0x8."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << np.uint8(3)
    lo = np.searchsorted(_E2M1_POS, np.nan_to_num(a, nan=6.0), side="right") - 1
    lo = np.clip(lo, 0, 6)
    d_lo = a - _E2M1_POS[lo]
    d_hi = _E2M1_POS[lo + 1] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo & 1) == 1))
    mag = np.where(pick_hi, lo + 1, lo).astype(np.uint8)
    mag = np.where((a >= 6.0) | np.isnan(a), np.uint8(7), mag)
    return (mag | sign).astype(np.uint8)


MXFP4_GROUP = 16


def mxfp4_row_bytes(d):
    """Bytes of one MXFP4 cache row of d channels: d/2 bytes of packed E2M1
    codes (channel 2j in the low nibble of byte j, 2j+1 in the high one),
    then d/16 E4M3 scale codes (scale g covers channels 16g .. 16g+15)."""
    return d // 2 + d // MXFP4_GROUP


def mxfp4_encode_rows(bits):
    """bf16 rows (uint16 bit patterns, [..., d]) -> MXFP4 rows
    ([..., d/2 + d/16] uint8), following the reading stated above: per
    group, amax = max |x| (exact in fp32; NaNs ignored), scale code =
    E4M3(fp32(amax / 6)), s = its value, codes = E2M1(fp32(x / s)); s = 0
    gives codes 0."""
    x = bf16_bits_to_f64(bits).astype(np.float32)
    d = x.shape[-1]
    g = x.reshape(x.shape[:-1] + (d // MXFP4_GROUP, MXFP4_GROUP))
    amax = np.fmax.reduce(np.abs(g), axis=-1).astype(np.float32)
    t = (amax / np.float32(6.0)).astype(np.float32)       # one fp32 rounding
    scodes = e4m3_encode_f32(t)
    s = e4m3_codes_to_f64(scodes).astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (g / np.where(s > 0, s, np.float32(1.0))).astype(np.float32)
    codes = np.where(s > 0, e2m1_encode_f32(q), np.uint8(0)).astype(np.uint8)
    codes = codes.reshape(x.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << np.uint8(4))).astype(
        np.uint8)
    return np.concatenate([packed, scodes.astype(np.uint8)], axis=-1)


def mxfp4_rows_to_f64(raw, d):
    """MXFP4 rows ([..., d/2 + d/16] uint8) -> exact float64 values
    [..., d]: code value times its group's scale value."""
    raw = np.asarray(raw, dtype=np.uint8)
    packed, scodes = raw[..., :d // 2], raw[..., d // 2:]
    codes = np.empty(raw.shape[:-1] + (d,), dtype=np.uint8)
    codes[..., 0::2] = packed & np.uint8(0xF)
    codes[..., 1::2] = packed >> np.uint8(4)
    vals = e2m1_codes_to_f64(codes)
    s = e4m3_codes_to_f64(scodes)
    return vals * np.repeat(s, MXFP4_GROUP, axis=-1)
