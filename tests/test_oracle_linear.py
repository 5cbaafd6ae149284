"""Pins for oracle.linear (the dense-Linear W4A16 product) on small matrices.

* scalar loops that decode every code by hand from the format definitions
  (E2M1 and E4M3 bit fields, E8M0 exponents, the NF3 bitstream and codebook)
  and sum x * w in Python floats, for all three formats and both activation
  types (the NF3 product rounded by torch's fp32 -> bf16 / fp16 conversion,
  a single rounding since the product is exact in fp32);
* the SwiGLU layer with one expert and top-1 gate 1, whose W2 step is the same
  product: with W13 chosen so that h = silu(gate) * up is known, the layer's
  output equals linear_forward(h, W2).
"""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import formats as F, layer, linear

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3(b):
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return -v if s else v


def _w_scalar(fmt, codes, scales, g, n, k, act="bf16"):
    if fmt in (F.FMT_NVFP4, F.FMT_MXFP4):
        byte = int(codes[n, k // 2])
        c = byte & 15 if k % 2 == 0 else byte >> 4
        v = E2M1[c & 7] * (-1 if c & 8 else 1)
        if fmt == F.FMT_NVFP4:
            return v * _e4m3(int(scales[n, k // 16])) * g
        return v * 2.0 ** (int(scales[n, k // 32]) - 127)
    row = [int(b) for b in codes[n]]
    bit = 3 * k
    c = sum(((row[(bit + i) // 8] >> ((bit + i) % 8)) & 1) << i for i in range(3))
    cb = [float(v) for v in torch.tensor([int(h, 16) for h in ("BF80", "BF09", "BE7D", "0000", "3E3C", "3EC4",
                                                                  "3F1F", "3F80")], dtype=torch.int32)
          .mul(65536).view(torch.float32)]
    s = float(torch.tensor([int(scales[n, k // 64])], dtype=torch.int32).mul(65536).view(torch.float32)[0])
    dt = torch.bfloat16 if act == "bf16" else torch.float16
    return float(torch.tensor(cb[c] * s, dtype=torch.float32).to(dt).float())


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_linear_matches_scalar_loops_all_formats(act):
    N, K, T = 4, 128, 3
    xdt = torch.bfloat16 if act == "bf16" else torch.float16
    x = synth.gen_x(T, K, seed=9, dtype=xdt).float().numpy().astype(np.float64)
    for fmt in (F.FMT_NVFP4, F.FMT_MXFP4, F.FMT_NF3):
        w = synth.gen_master(0, 2, N, K, seed=5)
        codes, scales, g = synth.quantise(fmt, w)
        c, s = codes.numpy(), scales.numpy()
        if fmt == F.FMT_NF3:
            s = s.view(np.uint16)
        ref = linear.linear_forward(x, fmt, c, s, g, K, act)
        for t in range(T):
            for n in range(N):
                acc = sum(float(x[t, k]) * _w_scalar(fmt, c, s, g, n, k, act) for k in range(K))
                assert math.isclose(acc, ref[t, n], rel_tol=1e-12, abs_tol=1e-15), (fmt, t, n)


def test_linear_is_the_layer_w2_step():
    """Top-1 layer, gate 1: out = W2 h with h = silu(W1 x) * (W3 x); the oracle layer and the
    linear oracle applied to the same h agree to rounding."""
    L = synth.make_layer(256, 128, 2, 1, kept_ids=[0])
    x = synth.gen_x(5, 256, seed=2).float().numpy().astype(np.float64)
    ids = np.zeros((5, 1), dtype=np.int32)
    gates = np.ones((5, 1))
    ex = L.expert_numpy(0)
    out = layer.moe_forward(x, ids, gates, L.expert_numpy, 256, 128)
    w13, _ = layer.expert_weights(ex, 256, 128)
    gu = x @ w13.T
    h = layer.silu(gu[:, :128]) * gu[:, 128:]
    c2, s2, g2 = ex["w2"]
    ref = linear.linear_forward(h, ex["fmt"], c2, s2, g2, 128)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-15)
