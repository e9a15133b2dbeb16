"""E4M3 (OCP OFP8 "E4M3FN") encode and decode, bit-exact, in plain numpy.

Format (OCP 8-bit Floating Point Specification, E4M3): 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits.  No infinities.  The single NaN pattern per
sign is exponent 1111 with mantissa 111 (0x7F / 0xFF).  Largest finite value is
0x7E = 1.75 * 2^8 = 448; smallest normal 0x08 = 2^-6; smallest subnormal
0x01 = 2^-9.

The pages ("FP8 ViT Encoder Attention", intro and note) only say that Q/K/V
are quantized "to FP8" on the fly; E4M3 is the reading taken here.

Encoding rule used by the whole path (a reading the pages leave open):

* round to nearest, ties to even mantissa, on the E4M3 grid including
  subnormals;
* after rounding, any magnitude above 448 saturates to 448 (0x7E | sign);
  +-inf saturates to +-448 as well ("satfinite");
* NaN maps to 0x7F with the input's sign bit (0xFF for a negative NaN);
* the sign is kept for results that round to zero (-tiny -> 0x80).

Everything here works on exact float64 values.  Every float32 (and bf16) input
is exactly representable in float64, and the rounding is done with
``np.rint`` (IEEE round-half-even) on a value that has been scaled by an exact
power of two, so no intermediate step rounds.
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9
NAN_CODE = 0x7F


def decode(codes):
    """Decode uint8 E4M3 codes to float64 values (NaN codes give NaN).

    value = (-1)^s * 2^(e-7) * (1 + m/8)   for e in 1..15 (except e=15, m=7)
    value = (-1)^s * 2^-6 * (m/8)          for e = 0 (subnormal / zero)
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(
        e == 0,
        np.ldexp(m.astype(np.float64), -9),            # m/8 * 2^-6
        np.ldexp((8 + m).astype(np.float64), (e - 10).astype(np.int64)),  # (1+m/8)*2^(e-7)
    )
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def encode(x):
    """Encode float values (float32 / float64 array) to uint8 E4M3 codes.

    Rounding: nearest, ties to even; saturating to +-448; NaN -> 0x7F|sign.
    """
    x = np.asarray(x)
    xf = x.astype(np.float64)  # exact for float32 / bf16 inputs
    sign = np.signbit(xf).astype(np.uint8) << 7
    a = np.abs(xf)
    isnan = np.isnan(a)
    a = np.where(isnan, 0.0, a)

    out = np.zeros(a.shape, dtype=np.int64)

    # Subnormal range (including zero): a < 2^-6.  Grid step 2^-9.  Rounding to
    # 8 * 2^-9 = 2^-6 gives code 8, which is exactly the smallest normal, so
    # the two ranges join without a special case.
    sub = a < E4M3_MIN_NORMAL
    q_sub = np.rint(np.ldexp(np.where(sub, a, 0.0), 9))  # a / 2^-9, exact scaling
    out = np.where(sub, q_sub.astype(np.int64), out)

    # Normal range: a = f * 2^E with f in [0.5, 1); unbiased exponent e = E-1.
    norm = ~sub
    an = np.where(norm, a, 1.0)
    an_fin = np.where(np.isinf(an), 1.0, an)
    _, E = np.frexp(an_fin)
    e = E.astype(np.int64) - 1
    # Significand scaled to [8, 16): q = a * 2^(3-e); 3 mantissa bits after the point.
    q = np.rint(np.ldexp(an_fin, (3 - e)))
    carry = q >= 16.0                      # rounding 1.111.. up to 10.000
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8.0, q)
    biased = e + 7
    code_n = (biased << 3) | (q.astype(np.int64) - 8)
    # Saturation: anything above 0x7E (448) after rounding, and +-inf.
    over = (biased > 15) | ((biased == 15) & (q.astype(np.int64) - 8 == 7)) | np.isinf(an)
    code_n = np.where(over, 0x7E, code_n)
    out = np.where(norm, code_n, out)

    out = np.where(isnan, NAN_CODE, out)
    return (out.astype(np.uint8) | sign).astype(np.uint8)


def round_significand(x, bits=4):
    """Round float64 values to ``bits`` significant bits (RNE), no exponent limits.

    E4M3 normal numbers carry 4 significant bits (1 implicit + 3 stored).  This
    is the rounding E4M3 applies inside its normal range, written without the
    range limits; the P-rounding attention variant uses it because the hot path
    scales P by an exact power of two before converting, which keeps P inside
    the normal range for every element that matters.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    safe = np.where((a == 0) | ~np.isfinite(a), 1.0, a)
    _, E = np.frexp(safe)
    e = E.astype(np.int64) - 1
    q = np.rint(np.ldexp(safe, (bits - 1) - e))
    r = np.ldexp(q, e - (bits - 1))
    r = np.where((a == 0) | ~np.isfinite(a), a, r)
    return np.copysign(r, x)
