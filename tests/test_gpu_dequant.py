"""The dequantised operands the kernels feed their matrix units are bit-exact with the oracle.

Two exports, each running the decoder its kernel runs (include/hmoe.h):
- hmoe_debug_dequant: the tensor-core (grouped) kernel's operand tile, equal to
  oracle.formats.dequant_tile for every format;
- hmoe_debug_decode_operand: the weight-streaming (decode) kernel's operand and its
  per-64-group factors. NVFP4 and MXFP4: the same tile, factors 1. NF3: the raw
  codebook entry of each code (oracle.formats.nf3_codebook indexed by
  oracle.formats.unpack_nf3) and the group's bf16 scale, exactly.
Both activation types: the operands are bf16 or fp16 values of the layer's type
(oracle.formats.dequant_tile with act).
"""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from oracle import formats as F
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _check_expert(moe, L, e):
    ex = L.expert_numpy(e)
    act = ex["act"]
    for which, (N, K) in ((13, (2 * L.I, L.H)), (2, (L.H, L.I))):
        codes, scales, _ = ex["w13" if which == 13 else "w2"]
        ref = F.dequant_tile(ex["fmt"], codes, scales, K, act)
        dst = torch.empty((N, K), dtype=moe.dtype, device="cuda")
        hm.hmoe_debug_dequant(moe.layer, e, which, dst)
        torch.cuda.synchronize()
        assert np.array_equal(U.dev_to_f64(dst), ref), f"tile: expert {e} W{which} fmt {ex['fmt']} {act}"
        # the decode kernel's operand
        vals = torch.full((N, K), float("nan"), dtype=moe.dtype, device="cuda")
        fac = torch.full((N, K // 64), float("nan"), dtype=torch.float32, device="cuda")
        hm.hmoe_debug_decode_operand(moe.layer, e, which, vals, fac)
        torch.cuda.synchronize()
        got_v = U.dev_to_f64(vals)
        got_f = fac.cpu().numpy().astype(np.float64)
        if ex["fmt"] == F.FMT_NF3:
            cb = F.nf3_codebook()
            assert np.array_equal(got_v, cb[F.unpack_nf3(codes, K)]), f"decode values: expert {e} W{which}"
            assert np.array_equal(got_f, F.bf16_bits_to_f64(np.asarray(scales, dtype=np.uint16))), \
                f"decode scales: expert {e} W{which}"
        else:
            assert np.array_equal(got_v, ref), f"decode values: expert {e} W{which} fmt {ex['fmt']}"
            assert np.all(got_f == 1.0)


def test_tiny_hybrid_tiles():
    L = synth.tiny_layer(device="cuda")
    moe = U.build(L, 8)
    for e in range(8):
        _check_expert(moe, L, e)


def test_mxfp4_tiles():
    L = synth.make_layer(256, 128, 6, 2, kept_ids=[0, 2, 4], kept_format=synth.FMT_MXFP4, device="cuda")
    moe = U.build(L, 8)
    for e in range(6):
        _check_expert(moe, L, e)


def test_extreme_codes_and_scales():
    """Every code and a wide scale range: random bytes in the logical layout."""
    g = torch.Generator(device="cuda").manual_seed(11)
    H, I, E = 256, 128, 3
    L = synth.make_layer(H, I, E, 1, kept_ids=[0], device="cuda")

    def rnd(shape, lo, hi):
        return torch.randint(lo, hi, shape, generator=g, device="cuda", dtype=torch.int32).to(torch.uint8)

    # expert 0 NVFP4: all 256 code bytes, E4M3 scales over every finite code
    c13, _, g13 = L.experts[0]["w13"]
    s13 = rnd((2 * I, H // 16), 0, 0xFF)
    s13[(s13 & 0x7F) == 0x7F] = 0x7E                      # every finite E4M3 code, both signs
    L.experts[0]["w13"] = (rnd(c13.shape, 0, 256), s13, g13)
    # expert 1 NF3: random bitstream, scales spanning many binades
    c13n, _, _ = L.experts[1]["w13"]
    sc = (torch.rand((2 * I, H // 64), generator=g, device="cuda") * 40 - 20).exp2().to(torch.bfloat16)
    L.experts[1]["w13"] = (rnd(c13n.shape, 0, 256), sc.view(torch.int16), 1.0)
    moe = U.build(L, 8)
    for e in range(2):
        _check_expert(moe, L, e)


def test_mxfp4_extreme_scales_and_subnormals():
    """MXFP4 with random E8M0 bytes over 0..254 and random codes. Byte 0 is 2^-127, a bf16
    subnormal, and its products with E2M1 values are bf16 subnormals; they must come out
    exact. Products beyond the bf16 range are unsupported inputs (the OCP encoder never
    makes them from finite weights), so codes are clamped where the scale is 2^126 or
    2^127: magnitude <= 3 (E2M1 <= 3) at byte 253, <= 1.5 at byte 254."""
    g = torch.Generator(device="cuda").manual_seed(12)
    H, I, E = 256, 128, 2
    L = synth.make_layer(H, I, E, 1, kept_ids=[0, 1], kept_format=synth.FMT_MXFP4, device="cuda")

    def rnd(shape, lo, hi):
        return torch.randint(lo, hi, shape, generator=g, device="cuda", dtype=torch.int32)

    for e in range(E):
        for key, (N, K) in (("w13", (2 * I, H)), ("w2", (H, I))):
            sc = rnd((N, K // 32), 0, 255)
            if e == 1:
                sc[:, ::2] = rnd((N, K // 64), 0, 4)          # many subnormal scales on expert 1
            codes = rnd((N, K), 0, 16)
            mag, sign = codes & 7, codes & 8
            byte = sc.repeat_interleave(32, dim=1)
            mag = torch.where(byte == 254, torch.clamp(mag, max=3), mag)
            mag = torch.where(byte == 253, torch.clamp(mag, max=5), mag)
            codes = (mag | sign).to(torch.uint8)
            packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
            L.experts[e][key] = (packed, sc.to(torch.uint8).contiguous(), 1.0)
    moe = U.build(L, 8)
    for e in range(E):
        _check_expert(moe, L, e)
    ex = L.expert_numpy(1)
    tile = F.dequant_tile(F.FMT_MXFP4, ex["w2"][0], ex["w2"][1], I)
    assert np.any((tile != 0) & (np.abs(tile) < 2.0 ** -126))   # the case really holds subnormals


def test_full_size_hybrid_sample_experts():
    L = synth.make_layer(**synth.HYBRID_256, kept_ids=list(range(0, 256, 4)), device="cuda")
    moe = U.build(L, 8)
    for e in (0, 1, 255):
        _check_expert(moe, L, e)


# ------------------------------------------------------------------ fp16 activations
@pytest.mark.parametrize("kept_format", [synth.FMT_NVFP4, synth.FMT_MXFP4])
def test_f16_tiles(kept_format):
    L = synth.make_layer(256, 128, 6, 2, kept_ids=[0, 2, 4], kept_format=kept_format, device="cuda", act="f16")
    moe = U.build(L, 8)
    assert moe.dtype == torch.float16
    for e in range(6):
        _check_expert(moe, L, e)


def test_f16_extreme_codes_and_scales():
    """fp16 operands over every code byte and the whole supported scale ranges: every finite
    E4M3 scale (NVFP4 products are all exact in fp16), E8M0 bytes 104..140 (MXFP4), and NF3
    scales over the fp16 normal range, where the tile is the product rounded once."""
    g = torch.Generator(device="cuda").manual_seed(13)
    H, I = 256, 128

    def rnd(shape, lo, hi):
        return torch.randint(lo, hi, shape, generator=g, device="cuda", dtype=torch.int32).to(torch.uint8)

    L = synth.make_layer(H, I, 3, 1, kept_ids=[0], device="cuda", act="f16")
    c13, _, g13 = L.experts[0]["w13"]
    s13 = rnd((2 * I, H // 16), 0, 0xFF)
    s13[(s13 & 0x7F) == 0x7F] = 0x7E
    L.experts[0]["w13"] = (rnd(c13.shape, 0, 256), s13, g13)
    c13n, _, _ = L.experts[1]["w13"]
    sc = (torch.rand((2 * I, H // 64), generator=g, device="cuda") * 28 - 14).exp2().to(torch.bfloat16)
    L.experts[1]["w13"] = (rnd(c13n.shape, 0, 256), sc.view(torch.int16), 1.0)
    moe = U.build(L, 8)
    for e in range(2):
        _check_expert(moe, L, e)

    Lm = synth.make_layer(H, I, 2, 1, kept_ids=[0, 1], kept_format=synth.FMT_MXFP4, device="cuda", act="f16")
    for e in range(2):
        for key, (N, K) in (("w13", (2 * I, H)), ("w2", (H, I))):
            c, _, _ = Lm.experts[e][key]
            Lm.experts[e][key] = (rnd(c.shape, 0, 256), rnd((N, K // 32), 104, 141), 1.0)
    moe = U.build(Lm, 8)
    for e in range(2):
        _check_expert(moe, Lm, e)
