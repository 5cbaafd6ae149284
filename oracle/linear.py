"""Dense-Linear W4A16 oracle: y = x W^T with a 4-bit (or 3-bit) weight matrix.

TEST INFRASTRUCTURE ONLY: see the package docstring.

[P3] "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE + --override-activation-dtype
flag", Summary and Related: the fused-MoE work follows a dense-Linear W4A16
method, 4-bit weights with 16-bit activations and no activation scales. The
plainest reading for one weight matrix W [N, K] in a logical layout of
``oracle.formats`` and activations x [T, K]:

    y[t, n] = sum_k x[t, k] * W[n, k]        (float64)

with W the full dequantised weights (``formats.dequant``: the NVFP4 global
scale included), dequantised to the activation type act ("bf16" or "f16",
[P3] "Summary", item 2). The rounding of the result to that type is left to
the comparison.
"""

import numpy as np

from . import formats


def linear_forward(x, fmt, codes, scales, g, K, act="bf16"):
    """float64 [T, N]: x [T, K] times the dequantised weights [N, K] transposed."""
    w = formats.dequant(fmt, codes, scales, g, K, act)
    return np.asarray(x, dtype=np.float64) @ w.T
