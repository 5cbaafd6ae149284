"""Pins for oracle.actquant (NVFP4 activation quantisation, the W4A4 layer).

Each check ties the oracle to something outside itself:
* E2M1 rounding: the weight encoder in synth (torch ops, written separately)
  on dense sweeps and every decision point, and a hand table of ties;
* E4M3 rounding: torch's float32 -> float8_e4m3fn conversion (round to
  nearest even), including every midpoint between neighbouring codes;
* the whole quantiser: the weight encoder on identical data with the same
  global scale (the same NVFP4 rule, independent code), exact round trips of
  values on the NVFP4 grid, zero and saturated blocks;
* the W4A4 layer: a top-1 expert recomputed with torch float64 ops around the
  oracle's quantiser (the order of the steps: x quantised before W13, h
  rounded to the activation type and quantised before W2).
"""

import numpy as np
import torch
import torch.nn.functional as Fn

import synth
from oracle import actquant as A, formats as F, layer


def test_e2m1_rounding_matches_encoder_and_ties():
    v = np.concatenate([np.linspace(-8, 8, 40001), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0],
                        -np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]), [1e9, -1e9, -0.0, 0.0, -0.2]])
    v = v.astype(np.float32)
    got = A.e2m1_rne_sat(v)
    ref = synth._e2m1_encode(torch.from_numpy(v)).numpy()
    assert np.array_equal(got, ref)
    table = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 5.01: 7, 7.0: 7, -0.2: 0, -0.3: 9,
             -6.5: 15}
    for x, c in table.items():
        assert A.e2m1_rne_sat(np.array([x], dtype=np.float32))[0] == c, x


def test_e4m3_rounding_matches_torch_including_ties():
    vals = F.e4m3_value(np.arange(0x7F))
    mids = 0.5 * (vals[:-1] + vals[1:])                       # exact ties (fp32-exact)
    rng = np.random.default_rng(3)
    t = np.concatenate([vals, mids, rng.uniform(0, 448, 30000), rng.uniform(0, 2.0 ** -6, 3000),
                        [448.0, 447.9, 0.0]]).astype(np.float32)
    got = A.e4m3_rne_sat(t)
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_quantizer_equals_weight_encoder_on_the_same_data():
    # the NVFP4 weight encoder computes g from the matrix amax and then the same per-16 rule
    w = synth.gen_master(1, 13, 64, 256, seed=9)
    codes_w, scales_w, g = synth.quant_nvfp4(w)
    codes_a, scales_a = A.quantize(w.numpy(), g)
    assert np.array_equal(scales_a, scales_w.numpy())
    assert np.array_equal(codes_a, codes_w.numpy())


def test_exact_round_trip_on_the_nvfp4_grid():
    rng = np.random.default_rng(5)
    R, K = 6, 128
    g = 2.0 ** -7                                            # power of two: every product below is exact
    s = rng.integers(0x08, 0x7E, size=(R, K // 16)).astype(np.uint8)   # normal E4M3 scales
    mag = rng.integers(0, 8, size=(R, K)).astype(np.uint8)
    mag.reshape(R, K // 16, 16)[:, :, 0] = 7                # each block's amax is 6 * e4m3(s) * g
    sign = rng.integers(0, 2, size=(R, K)).astype(np.uint8) << 3
    codes = mag | np.where(mag > 0, sign, 0).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    a = A.dequantize(packed, s, g, K)
    assert np.array_equal(a.astype(np.float32).astype(np.float64), a)
    c2, s2 = A.quantize(a, g)
    assert np.array_equal(s2, s)
    assert np.array_equal(c2, packed)
    assert np.array_equal(A.fake_quant(a, g), a)


def test_zero_and_saturated_blocks():
    a = np.zeros((2, 32), dtype=np.float32)
    a[1, 16:] = 1e6                                           # amax / (6 g) far above 448
    codes, scales = A.quantize(a, 1e-3)
    assert scales[0, 0] == 0 and scales[0, 1] == 0 and np.all(codes[0] == 0)
    assert scales[1, 1] == 0x7E                               # 448
    deq = A.dequantize(codes, scales, 1e-3, 32)
    assert np.all(deq[0] == 0)
    assert np.allclose(deq[1, 16:], 6 * 448 * np.float32(1e-3))


def test_w4a4_top1_layer_order_of_steps():
    H, I = 256, 128
    L = synth.make_layer(H, I, 2, 1, kept_ids=[0])
    g13, g2 = 4e-4, 1e-4
    L.act_quant = (g13, g2)
    x = synth.gen_x(5, H, seed=8).float().numpy().astype(np.float64)
    ids = np.zeros((5, 1), dtype=np.int32)
    out = layer.moe_forward(x, ids, np.ones((5, 1)), L.expert_numpy, H, I)
    ex = L.expert_numpy(0)
    w13, w2 = (torch.from_numpy(w) for w in layer.expert_weights(ex, H, I))
    xq = torch.from_numpy(A.fake_quant(x, g13))
    gu = xq @ w13.T
    h = Fn.silu(gu[:, :I]) * gu[:, I:]
    h_act = h.float().to(torch.bfloat16).double()            # h is a bf16 activation
    hq = torch.from_numpy(A.fake_quant(h_act.numpy(), g2))
    ref = (hq @ w2.T).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-15)
    # and the quantisation matters: without it the result differs
    L.act_quant = None
    assert not np.allclose(layer.moe_forward(x, ids, np.ones((5, 1)), L.expert_numpy, H, I), out, rtol=1e-3)
