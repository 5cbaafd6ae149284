"""NVFP4 activation quantisation for the W4A4 layer (oracle).

TEST INFRASTRUCTURE ONLY: see the package docstring.

[P3] "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE + --override-activation-dtype
flag", Summary: the W4A4 NVFP4 backends take the quantisation scheme
(kNvfp4Static, kNvfp4Dynamic): static NVFP4 weights, and activations
quantised to NVFP4 as they arrive. The pages give no formula. The plainest
reading, used here, is the NVFP4 rule the weights follow (oracle.formats), with
a static per-layer global scale g and block scales computed from the data:

  for each block b of 16 consecutive values along a row (K):
      s_b   = E4M3_rne(min(amax_b / (6 g), 448))
      d_b   = e4m3(s_b) * g
      q_i   = E2M1_rne_sat(a_i / d_b)          (0 where d_b = 0)
      a'_i  = e2m1(q_i) * e4m3(s_b) * g        (the dequantised activation)

Every decision (the E4M3 and E2M1 roundings) is taken in fp32 arithmetic:
6 g, amax_b / (6 g), e4m3(s_b) * g and a_i / d_b are each one correctly
rounded fp32 operation, as in the kernels. E2M1 rounding is to nearest with
ties to the even mantissa bit, saturating at 6; a negative value that rounds
to 0 gives code 0.

The W4A4 layer (oracle.layer.moe_forward with act_quant) quantises x before
W13 with the global scale g13 and h before W2 with g2; h is an activation of
the layer's type, so it is rounded to that type first.
"""

import numpy as np

from . import formats

GROUP = 16

# E2M1 magnitudes in code order and the decision points between neighbours.
# A tie at a decision point goes to the neighbour whose mantissa bit is 0.
_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_rne_sat(v):
    """fp32 values -> E2M1 codes (uint8 0..15), round to nearest even, saturating at 6."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    codes = np.zeros(a.shape, dtype=np.int64)
    for m in range(1, 8):
        lo, hi = _MAGS[m - 1], _MAGS[m]
        mid = 0.5 * (lo + hi)
        # code m when a is above the midpoint, or exactly on it and m has an even mantissa bit
        even_up = (m & 1) == 0
        codes += (a > mid) | ((a == mid) & even_up)
    sign = np.signbit(v) & (codes > 0)
    return (codes | (sign.astype(np.int64) << 3)).astype(np.uint8)


def e4m3_rne_sat(t):
    """Non-negative fp32 values (at most 448) -> E4M3 bytes, round to nearest even.

    Written from the E4M3 definition: 3 mantissa bits, exponent bias 7,
    subnormals m/8 * 2**-6, largest finite 448.
    """
    t = np.asarray(t, dtype=np.float64)
    vals = formats.e4m3_value(np.arange(0x7F, dtype=np.int64))   # codes 0x00 .. 0x7E, ascending
    i = np.clip(np.searchsorted(vals, t, side="left"), 1, len(vals) - 1)
    lo, hi = vals[i - 1], vals[i]                                  # lo < t <= hi inside the range
    down = (t - lo < hi - t) | ((t - lo == hi - t) & ((i & 1) == 1))   # a tie goes to the even code
    code = np.where(t <= vals[0], 0, np.where(t >= vals[-1], len(vals) - 1, np.where(down, i - 1, i)))
    return code.astype(np.uint8)


def quantize(a, g):
    """NVFP4 activation quantisation of rows a [R, K] (K a multiple of 16) with global scale g.

    Returns (codes uint8 [R, K/2] in the logical layout of oracle.formats,
    scales uint8 [R, K/16] E4M3 bytes).
    """
    a = np.asarray(a, dtype=np.float32)
    R, K = a.shape
    g32 = np.float32(g)
    blocks = a.reshape(R, K // GROUP, GROUP)
    amax = np.abs(blocks).max(axis=2)
    t = amax / np.float32(np.float32(6.0) * g32)                 # fp32 division
    t = np.minimum(t, np.float32(448.0))
    s = e4m3_rne_sat(t)
    d = (formats.e4m3_value(s).astype(np.float32) * g32).astype(np.float32)
    safe = np.where(d > 0, d, np.float32(1.0))
    v = (blocks / safe[:, :, None]).astype(np.float32)
    v = np.where(d[:, :, None] > 0, v, np.float32(0.0))
    codes = e2m1_rne_sat(v).reshape(R, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, s


def dequantize(codes, scales, g, K):
    """The dequantised activations a' [R, K] float64: e2m1 * e4m3 * g."""
    return formats.dequant(formats.FMT_NVFP4, codes, scales, g, K)


def fake_quant(a, g):
    """a' = dequantize(quantize(a, g)), float64."""
    a = np.asarray(a)
    codes, scales = quantize(a, g)
    return dequantize(codes, scales, g, a.shape[1])
