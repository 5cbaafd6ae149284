"""W4A4 NVFP4: activation quantisation (bit-exact) and the W4A4 layer (within tolerance).

"[Quantization][ModelOpt] W4A16 NVFP4 fused MoE + --override-activation-dtype
flag", Summary: the W4A4 NVFP4 scheme quantises activations to NVFP4 as they
arrive. The quantiser hmoe_quantize_act_nvfp4 is compared element by element
with oracle.actquant.quantize (codes and E4M3 scales, the same fp32
decisions). The W4A4 layer (x quantised before W13, h before W2) is compared
with oracle.layer.moe_forward with act_quant.

Tolerance of the W4A4 layer. x is quantised identically on both sides (the
same 16-bit input, the same fp32 decisions), and both kernels form h from the
same weights as the oracle (for W4A4 layers the streaming kernel decodes NF3
to the tile values rne(cb * s); with its W4A16 decode, the exact cb * s, codes
of h flipped and rows moved by up to 5%). h itself is formed in fp32 by the
kernels and in float64 by the oracle, so an element can still round to a
different 16-bit value and take a neighbouring E2M1 code, one step being up
to a third of its block's largest value, which would move an output row of
these small layers by a few percent. So: every row within 5e-2 * max|ref|,
and the median row within 1e-2, the W4A16 layer's bar (measured: all rows
of the tiny layer at T = 8 and 9 within 3e-3).
"""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from oracle import actquant as A
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

W4A4_ROW_TOL = 5e-2
W4A4_MEDIAN_TOL = 1e-2


def assert_w4a4_close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.abs(got - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)
    assert rel.max() <= W4A4_ROW_TOL, f"row-relative error {rel.max():.3e}"
    assert np.median(rel) <= W4A4_MEDIAN_TOL, f"median row-relative error {np.median(rel):.3e}"


def _quant_dev(x, g):
    R, K = x.shape
    codes = torch.full((R, K // 2), 0xAA, dtype=torch.uint8, device="cuda")
    scales = torch.full((R, K // 16), 0xAA, dtype=torch.uint8, device="cuda")
    hm.hmoe_quantize_act_nvfp4(x, g, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_quantizer_bit_exact(dtype):
    x = synth.gen_x(37, 512, seed=4, device="cuda", dtype=dtype)
    x[3] = 0                                                    # all-zero blocks
    x[5, :16] *= 1e3                                            # a block far above 6 * 448 * g: saturation
    x[6, :16] = torch.tensor([0.5, -0.5, 1.5, 3.0, 6.0, -6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.1,
                              0.0, -0.0], dtype=dtype)          # ties of E2M1 once scaled by d = 1
    g = 6.0 / (6.0 * 6.0)                                       # row 6, block 0: amax 6 -> s = 1, d = 1
    for gg in (g, float(x.float().abs().max()) / (6 * 448), 1e-6):
        c, s = _quant_dev(x, gg)
        rc, rs = A.quantize(x.float().cpu().numpy(), gg)
        assert np.array_equal(s, rs), gg
        assert np.array_equal(c, rc), gg


def _w4a4_layer(L, g13, g2):
    L.act_quant = (g13, g2)
    bm = None if L.bit_map is None else [int(b) for b in L.bit_map]
    return hm.HybridMoELayer(L.H, L.I, L.E, L.topk, bm, U.device_experts(L), kept_format=L.kept_format,
                             max_tokens=1200, act_dtype=U.act_dtype(L), act_globals=(g13, g2))


@pytest.fixture(scope="module")
def tiny_w4a4():
    L = synth.tiny_layer(device="cuda")
    return L, _w4a4_layer(L, 5.0 / (6 * 448), 0.6 / (6 * 448))


@pytest.mark.parametrize("T", [1, 3, 8, 9, 37, 200, 1200])
def test_w4a4_tiny_layer_parity(tiny_w4a4, T):
    L, moe = tiny_w4a4
    x = synth.gen_x(T, L.H, seed=T, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    ref = U.oracle_out(L, x, ids, gates)
    assert_w4a4_close(out.float().cpu().numpy(), ref)
    for order in (hm.TIERS_KEPT_FIRST, hm.TIERS_NF3_FIRST):
        o, _ = U.run(moe, x, logits, tier_order=order)
        assert torch.equal(o, out)
    if T > 8:
        s, _ = U.run(moe, x, logits, path=hm.PATH_STREAM)
        assert_w4a4_close(s.float().cpu().numpy(), ref)


def test_w4a4_differs_from_w4a16(tiny_w4a4):
    """The quantisation is really applied: the W4A16 layer on the same weights gives another result."""
    L, moe = tiny_w4a4
    x = synth.gen_x(16, L.H, seed=1, device="cuda")
    logits = synth.gen_logits(16, L.E, seed=1, device="cuda")
    a, _ = U.run(moe, x, logits)
    L.act_quant = None
    plain = U.build(L, 16)
    L.act_quant = (5.0 / (6 * 448), 0.6 / (6 * 448))
    b, _ = U.run(plain, x, logits)
    assert not torch.equal(a, b)
    assert (a.float() - b.float()).abs().max() < 0.2 * b.float().abs().max()


def test_w4a4_fp16_and_mxfp4():
    L = synth.make_layer(384, 192, 8, 2, kept_ids=[0, 3, 5], kept_format=synth.FMT_MXFP4, device="cuda", act="f16")
    moe = _w4a4_layer(L, 5.0 / (6 * 448), 1.0 / (6 * 448))
    for T, path in ((8, hm.PATH_STREAM), (96, hm.PATH_GROUPED)):
        x = synth.gen_x(T, L.H, seed=T, device="cuda", dtype=torch.float16)
        logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
        out, (ids, gates, _, _) = U.run(moe, x, logits, path=path)
        assert_w4a4_close(out.float().cpu().numpy(), U.oracle_out(L, x, ids, gates))


@pytest.fixture(scope="module")
def hybrid256_w4a4():
    L = synth.make_layer(**synth.HYBRID_256, kept=64, device="cuda")
    return L, _w4a4_layer(L, 5.0 / (6 * 448), 24.0 / (6 * 448))


def test_w4a4_full_size_decode_and_prefill(hybrid256_w4a4):
    """The 256-expert hybrid layer with W4A4: M=8 (every token) and M=1024 (the first and last
    token of every routed expert) against the oracle."""
    L, moe = hybrid256_w4a4
    for T, stride in ((8, 0), (1024, 0)):
        x = synth.gen_x(T, L.H, seed=300 + T, device="cuda")
        logits = synth.gen_logits(T, L.E, seed=300 + T, device="cuda")
        out, (ids, gates, perm, offsets) = U.run(moe, x, logits)
        assert torch.isfinite(out.float()).all()
        tokens = list(range(T)) if T <= 8 else U.cover_tokens(ids, perm, offsets, stride)
        assert_w4a4_close(out.float().cpu().numpy()[tokens], U.oracle_rows(L, x, ids, gates, tokens=tokens))


def test_w4a4_decode_operand_is_the_tile(tiny_w4a4):
    """For W4A4 layers the streaming kernel decodes NF3 to the tile values rne(cb * s) (the weights
    the tensor-core kernel and the definition use) with unit group factors."""
    from oracle import formats as F
    L, moe = tiny_w4a4
    for e in (0, 5):
        ex = L.expert_numpy(e)
        codes, scales, _ = ex["w13"]
        N, K = 2 * L.I, L.H
        vals = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
        fac = torch.full((N, K // 64), float("nan"), dtype=torch.float32, device="cuda")
        hm.hmoe_debug_decode_operand(moe.layer, e, 13, vals, fac)
        torch.cuda.synchronize()
        assert np.array_equal(U.dev_to_f64(vals), F.dequant_tile(ex["fmt"], codes, scales, K))
        assert torch.all(fac == 1.0)
