"""Element formats and dequantisation of the logical checkpoint layouts (oracle).

TEST INFRASTRUCTURE ONLY: see the package docstring.

[P1] "How it works" and [P2] "Summary" name the formats but do not define them.
The kept tier is NVFP4 (MXFP4 under ``kept_format``) and the tail is NF3,
3-bit. This module takes the plainest definitions:

* E2M1 (OCP FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. The
  exponent field 0 encodes the subnormals 0 and 0.5. The value set is
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}, each with either sign.
* E4M3 "fn" (OCP FP8): bias 7, no infinities. The all-ones pattern
  S.1111.111 is NaN. Subnormals are m/8 * 2**-6.
* E8M0 (OCP MX scale): value 2**(b - 127). The byte 0xFF is NaN.
* NF3: the NormalFloat construction of Dettmers et al. ("QLoRA", 2023, Sec. 3)
  at 3 bits. Quantiles of N(0,1) are taken at 4 positive and 3 negative
  probability levels, an exact 0 is added, the set is normalised by its
  maximum, and every entry is rounded to bf16.

Logical checkpoint layouts (the input to the packer and the oracle):

* NVFP4 matrix [N, K]: codes uint8 [N, K/2], where element 2i is in the low
  nibble and 2i+1 in the high nibble. Scales are E4M3 uint8 [N, K/16]. There
  is one fp32 global scale g per matrix.
  w = e2m1(code) * e4m3(scale) * g.
* MXFP4 matrix [N, K]: codes as NVFP4. Scales are E8M0 uint8 [N, K/32].
  w = e2m1(code) * 2**(b-127).
* NF3 matrix [N, K]: codes are an LSB-first bitstream, uint8 [N, 3K/8].
  Code j occupies bits [3j, 3j+3) of the row's little-endian byte string.
  Scales are bf16 [N, K/64], stored as uint16 bit patterns.
  w = bf16_rne(cb[code] * scale).

The "dequantised tile" is the 16-bit operand a kernel feeds to its matrix
unit, in the layer's activation type ([P3] "Summary", item 2: the W4A16
activations are bfloat16 or float16, and the weights are dequantised to the
activation type). With rne the rounding to that type:
  NVFP4: e2m1*e4m3. This is exact in bf16 and in fp16; g is applied to the
         fp32 sum.
  MXFP4: e2m1*2**(b-127). Exact in bf16; in fp16 exact for b in 104..140
         and rounded (to 0 or infinity) outside.
  NF3:   rne(cb*s). For bf16 layers this is the logical weight above; for
         fp16 layers the same product rounded once to fp16 (the pages give
         no fp16 NF3 rule: this is the plainest reading of "dequantised to
         the activation type").
"""

import numpy as np
from scipy.stats import norm

NVFP4_GROUP = 16
MXFP4_GROUP = 32
NF3_GROUP = 64

FMT_NF3 = 3
FMT_NVFP4 = 4
FMT_MXFP4 = 5


# ---------------------------------------------------------------- element decoders
def e2m1_value(code):
    """Decode 4-bit E2M1 codes (any integer array, values 0..15) to float64.

    Sign is bit 3, exponent bits 2..1, mantissa bit 0. Exponent bias is 1.
    Exponent 0 is subnormal: 0.5 * mantissa.
    """
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e - 1.0))
    return np.where(s == 1, -mag, mag)


def e4m3_value(byte):
    """Decode E4M3 "fn" bytes to float64. S.1111.111 decodes to NaN."""
    b = np.asarray(byte, dtype=np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e8m0_value(byte):
    """Decode E8M0 scale bytes: 2**(b-127). Byte 0xFF decodes to NaN."""
    b = np.asarray(byte, dtype=np.int64)
    v = np.exp2(b.astype(np.float64) - 127.0)
    return np.where(b == 255, np.nan, v)


def bf16_bits_to_f64(bits):
    """Reinterpret uint16 bf16 bit patterns as float64 values."""
    u = np.asarray(bits, dtype=np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_rne(x):
    """Round float64 values, which must be exactly representable in fp32, to bf16.

    The rule is round-to-nearest-even on the 16 dropped fraction bits of the
    fp32 pattern. Values are returned as float64. NaN is not supported.
    """
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), x, equal_nan=False):
        raise ValueError("bf16_rne: input not exactly representable in fp32")
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def f16_rne(x):
    """Round float64 values to IEEE binary16 (fp16), round-to-nearest-even, as float64.

    binary16 has 11 significant bits, a minimum normal exponent of -14 and
    subnormals spaced 2**-24 apart, so a value of binary exponent e is
    rounded to a multiple of 2**(max(e, -14) - 10), ties to the even
    multiple. Results above the largest finite value 65504 after rounding
    become infinity (with the sign). NaN is not supported.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e2 = np.frexp(a)                  # a = m * 2**e2, m in [0.5, 1): binary exponent e2 - 1
    e = np.where(a > 0, e2 - 1, -14)
    q = np.exp2(np.maximum(e, -14) - 10.0)
    r = np.rint(a / q) * q               # np.rint rounds half to even; a / q is exact
    r = np.where(r > 65504.0, np.inf, r)
    return np.copysign(r, x)


def act_rne(x, act):
    """Round to the activation type: act is "bf16" or "f16"."""
    if act == "bf16":
        return bf16_rne(x)
    if act == "f16":
        return f16_rne(x)
    raise ValueError(f"unknown activation type {act!r}")


# ---------------------------------------------------------------- NF3 codebook
def normalfloat_levels(bits):
    """NormalFloat code values from Dettmers et al., "QLoRA" (2023), Sec. 3.

    The construction produces 2**bits sorted values in [-1, 1]. It takes
    2**(bits-1) positive N(0,1) quantiles and 2**(bits-1)-1 negative ones,
    both at evenly spaced probabilities from an offset down to 0.5. The
    offset is the mean of 1-1/(2(n-1)) and 1-1/(2n), with n = 2**bits. An
    exact zero is added and the set is divided by its maximum. The result is
    float64 and not yet rounded.
    """
    n = 2 ** bits
    offset = 0.5 * ((1.0 - 1.0 / (2 * (n - 1))) + (1.0 - 1.0 / (2 * n)))
    pos = norm.ppf(np.linspace(offset, 0.5, n // 2 + 1)[:-1])
    neg = -norm.ppf(np.linspace(offset, 0.5, n // 2)[:-1])
    v = np.sort(np.concatenate([pos, neg, [0.0]]))
    return v / v.max()


def nf3_codebook():
    """The 8-entry NF3 codebook: NormalFloat(3 bits), each entry rounded to bf16.

    The result is sorted ascending. Index 3 is the exact zero, and indices 0
    and 7 are -1 and +1.
    """
    return bf16_rne(normalfloat_levels(3).astype(np.float32).astype(np.float64))


# ---------------------------------------------------------------- unpacking
def unpack_nibbles(codes, K):
    """uint8 [N, K/2] -> int64 [N, K]. Element 2i is the low nibble, 2i+1 the high one."""
    c = np.asarray(codes, dtype=np.uint8)
    N = c.shape[0]
    out = np.empty((N, K), dtype=np.int64)
    out[:, 0::2] = c & 0x0F
    out[:, 1::2] = c >> 4
    return out


def unpack_nf3(codes, K):
    """LSB-first 3-bit bitstream uint8 [N, 3K/8] -> int64 [N, K]."""
    c = np.asarray(codes, dtype=np.uint8)
    N = c.shape[0]
    bits = np.unpackbits(c, axis=1, bitorder="little").astype(np.int64)  # [N, 3K]
    bits = bits[:, : 3 * K].reshape(N, K, 3)
    return bits[:, :, 0] | (bits[:, :, 1] << 1) | (bits[:, :, 2] << 2)


# ---------------------------------------------------------------- dequantisation
def dequant_tile(fmt, codes, scales, K, act="bf16"):
    """The dequantised tile: [N, K] float64. Every entry is a value of the activation type.

    NVFP4: e2m1 * e4m3 (global scale excluded). MXFP4: e2m1 * 2**(b-127).
    NF3: rne(cb * s). act: "bf16" or "f16". The NVFP4 and MXFP4 products
    are exact in bf16, so only fp16 rounds them (an identity inside the fp16
    ranges stated in the module docstring).
    """
    if fmt == FMT_NVFP4:
        v = e2m1_value(unpack_nibbles(codes, K))
        s = e4m3_value(np.asarray(scales, dtype=np.uint8))
        t = v * np.repeat(s, NVFP4_GROUP, axis=1)
        return t if act == "bf16" else act_rne(t, act)
    if fmt == FMT_MXFP4:
        v = e2m1_value(unpack_nibbles(codes, K))
        s = e8m0_value(np.asarray(scales, dtype=np.uint8))
        t = v * np.repeat(s, MXFP4_GROUP, axis=1)
        return t if act == "bf16" else act_rne(t, act)
    if fmt == FMT_NF3:
        cb = nf3_codebook()
        v = cb[unpack_nf3(codes, K)]
        s = bf16_bits_to_f64(np.asarray(scales, dtype=np.uint16))
        return act_rne(v * np.repeat(s, NF3_GROUP, axis=1), act)
    raise ValueError(f"unknown format {fmt}")


def dequant(fmt, codes, scales, g, K, act="bf16"):
    """Full dequantised weights [N, K] float64. This is the tile times g for NVFP4."""
    t = dequant_tile(fmt, codes, scales, K, act)
    if fmt == FMT_NVFP4:
        return t * float(g)
    return t
