"""fp16 activations: the layer and the dense Linear with act_dtype = HMOE_ACT_F16.

"[Quantization][ModelOpt] W4A16 NVFP4 fused MoE + --override-activation-dtype
flag", Summary item 2: the W4A16 path takes bfloat16 or float16 activations.
The same kernels run with fp16 operands (mma.sync .f16 on the streaming path,
tcgen05.mma kind::f16 with fp16 A and B on the grouped path), fp16 h and an
fp16 result. The oracle dequantises to fp16 (oracle.formats.dequant_tile with
act="f16") and sums in float64.

Tolerance as for bf16 layers: per token row, max|out - ref| <= 2e-2 * max|ref|.
"""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from oracle import linear as olinear
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _x(L, T, seed):
    return synth.gen_x(T, L.H, seed=seed, device="cuda", dtype=torch.float16)


@pytest.fixture(scope="module")
def tiny16():
    L = synth.make_layer(**synth.TINY, kept_ids=[0, 1, 2, 3], device="cuda", act="f16")
    return L, U.build(L, 1200)


@pytest.mark.parametrize("T", [1, 3, 8, 9, 37, 200, 1200])
def test_f16_tiny_layer_parity(tiny16, T):
    L, moe = tiny16
    assert moe.dtype == torch.float16
    x = _x(L, T, T)
    logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    assert out.dtype == torch.float16
    ref = U.oracle_out(L, x, ids, gates)
    U.assert_rows_close(out.float().cpu().numpy(), ref)
    for order in (hm.TIERS_KEPT_FIRST, hm.TIERS_NF3_FIRST):
        o, _ = U.run(moe, x, logits, tier_order=order)
        assert torch.equal(o, out)
    if T > 8:
        s, _ = U.run(moe, x, logits, path=hm.PATH_STREAM)
        U.assert_rows_close(s.float().cpu().numpy(), ref)


def test_f16_token_order_is_bitwise_invariant(tiny16):
    L, moe = tiny16
    for T in (8, 37):
        x = _x(L, T, 0)
        logits = synth.gen_logits(T, L.E, device="cuda")
        p = torch.randperm(T, generator=torch.Generator().manual_seed(T)).cuda()
        a, _ = U.run(moe, x, logits)
        b, _ = U.run(moe, x[p].contiguous(), logits[p].contiguous())
        assert torch.equal(a[p], b)


@pytest.mark.parametrize("kept_format", [synth.FMT_NVFP4, synth.FMT_MXFP4])
def test_f16_odd_k_block_counts(kept_format):
    """I=192 (3 W2 k-blocks, 3 W13 row tiles: a one-row-tile last item), both paths."""
    L = synth.make_layer(384, 192, 8, 2, kept_ids=[0, 3, 5], kept_format=kept_format, device="cuda", act="f16")
    T = 96
    moe = U.build(L, T)
    x = _x(L, T, 11)
    logits = synth.gen_logits(T, L.E, seed=11, device="cuda")
    g, (ids, gates, _, _) = U.run(moe, x, logits, path=hm.PATH_GROUPED)
    s, _ = U.run(moe, x, logits, path=hm.PATH_STREAM)
    ref = U.oracle_out(L, x, ids, gates)
    U.assert_rows_close(g.float().cpu().numpy(), ref)
    U.assert_rows_close(s.float().cpu().numpy(), ref)


def test_f16_rejects_the_pair_kernel(tiny16):
    L, moe = tiny16
    x = _x(L, 64, 1)
    ids, gates, perm, offsets = moe.plan(synth.gen_logits(64, L.E, device="cuda"))
    out = torch.empty((64, L.H), dtype=torch.float16, device="cuda")
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_forward(moe.layer, x, ids, gates, perm, offsets, out, moe.ws, path=hm.PATH_GROUPED,
                        debug_flags=hm.DEBUG_GROUPED_PAIR)
    assert ei.value.status == -1


@pytest.fixture(scope="module")
def hybrid256_f16():
    L = synth.make_layer(**synth.HYBRID_256, kept=64, device="cuda", act="f16")
    return L, U.build(L, 1024)


@pytest.mark.parametrize("T", [4, 8])
def test_f16_full_size_hybrid_decode(hybrid256_f16, T):
    """The 256-expert hybrid layer (H=6144, I=2048, top-8; 64 NVFP4 + 192 NF3) with fp16
    activations at decode sizes; every token against the oracle."""
    L, moe = hybrid256_f16
    x = _x(L, T, 200 + T)
    logits = synth.gen_logits(T, L.E, seed=200 + T, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    assert torch.isfinite(out.float()).all()
    U.assert_rows_close(out.float().cpu().numpy(), U.oracle_rows(L, x, ids, gates))


def test_f16_full_size_hybrid_prefill(hybrid256_f16):
    """T=1024 on the grouped path: the tokens that reach every routed expert's first and last
    (ragged) token tile, against the oracle."""
    L, moe = hybrid256_f16
    T = 1024
    x = _x(L, T, 7)
    logits = synth.gen_logits(T, L.E, seed=7, device="cuda")
    out, (ids, gates, perm, offsets) = U.run(moe, x, logits)
    assert hm.hmoe_auto_path(moe.desc, T) == hm.PATH_GROUPED
    tokens = U.cover_tokens(ids, perm, offsets)
    U.assert_rows_close(out.float().cpu().numpy()[tokens], U.oracle_rows(L, x, ids, gates, tokens=tokens))


# ------------------------------------------------------------------ dense Linear
def _lin_ref(x, fmt, codes, scales, g, K):
    c = codes.cpu().numpy()
    s = scales.cpu().numpy()
    if fmt == synth.FMT_NF3:
        s = s.view(np.uint16)
    return olinear.linear_forward(x.float().cpu().numpy().astype(np.float64), fmt, c, s, g, K, "f16")


@pytest.mark.parametrize("fmt", [synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_NF3])
def test_f16_linear_both_paths(fmt):
    N, K = 256, 384
    w = synth.gen_master(3, 2, N, K, seed=3, device="cuda")
    codes, scales, g = synth.quantise(fmt, w)
    lin = hm.LinearW4A16(N, K, fmt, codes, scales, g, max_tokens=300, act_dtype=hm.ACT_F16)
    for T in (1, 8, 9, 300):
        x = synth.gen_x(T, K, seed=T, device="cuda", dtype=torch.float16)
        ref = _lin_ref(x, fmt, codes, scales, g, K)
        for path in (hm.PATH_STREAM, hm.PATH_GROUPED):
            out = lin(x, path=path)
            torch.cuda.synchronize()
            hm.hmoe_check_device_status(lin.ws)
            assert out.dtype == torch.float16
            U.assert_rows_close(out.float().cpu().numpy(), ref)
