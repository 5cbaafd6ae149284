"""The operand tiles the kernels feed the tensor cores are bit-exact with the oracle's dequantised tile."""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from oracle import formats as F
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _bf16_dev_to_f64(t):
    bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
    return F.bf16_bits_to_f64(bits)


def _check_expert(moe, L, e):
    ex = L.expert_numpy(e)
    for which, (N, K) in ((13, (2 * L.I, L.H)), (2, (L.H, L.I))):
        dst = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
        hm.hmoe_debug_dequant(moe.layer, e, which, dst)
        torch.cuda.synchronize()
        got = _bf16_dev_to_f64(dst)
        codes, scales, _ = ex["w13" if which == 13 else "w2"]
        ref = F.dequant_tile(ex["fmt"], codes, scales, K)
        assert np.array_equal(got, ref), f"expert {e} W{which} fmt {ex['fmt']}"


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


def test_full_size_hybrid_sample_experts():
    L = synth.make_layer(**synth.HYBRID_256, kept_ids=list(range(0, 256, 4)), device="cuda")
    moe = U.build(L, 8)
    for e in (0, 1, 255):
        _check_expert(moe, L, e)
