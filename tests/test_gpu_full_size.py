"""Full-size workloads, in the launch configuration bench.py times.

The oracle checks sampled tokens exactly (per token row within 2e-2 * max|ref|).
Properties that hold at any size cover every other row:
- finite;
- bitwise invariance to tier order;
- stream and grouped paths agree within tolerance.

Workloads:
- the 256-expert hybrid layer (H=6144, I=2048, top-8, 64 NVFP4 + 192 NF3) at
  prefill M=4096 with Zipf-skewed routing;
- the same shape with the kept tier in MXFP4 at M in {64, 512};
- the uniform NVFP4 layer (H=2048, I=768, E=128, top-8) for
  M in {1, 8, 128, 1024, 8192}.
"""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _rows(out, tokens):
    return out[tokens].float().cpu().numpy()


@pytest.fixture(scope="module")
def hybrid_prefill():
    L = synth.make_layer(**synth.HYBRID_256, kept=64, device="cuda")
    return L, U.build(L, 4096)


def test_hybrid_prefill_4096_zipf(hybrid_prefill):
    L, moe = hybrid_prefill
    T = 4096
    beta, ratio = synth.calibrate_zipf_beta(T, L.E, L.topk, device="cuda", iters=24)
    assert 9.0 <= ratio <= 11.0
    x = synth.gen_x(T, L.H, seed=7, device="cuda")
    logits = synth.gen_logits(T, L.E, device="cuda") + synth.zipf_bias(L.E, beta, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    assert torch.isfinite(out.float()).all()
    # tokens routed to the hottest expert and a few cold ones
    cnt = torch.bincount(ids.reshape(-1).long(), minlength=L.E)
    hot = int(torch.argmax(cnt))
    hot_tok = int(torch.nonzero((ids == hot).any(dim=1))[0])
    tokens = sorted({0, hot_tok, T - 1})
    ref = U.oracle_out(L, x, ids, gates, tokens=tokens)
    U.assert_rows_close(_rows(out, tokens), ref)
    out2, _ = U.run(moe, x, logits, tier_order=hm.TIERS_KEPT_FIRST)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("T", [64, 512])
def test_mxfp4_kept_tier_full_shape(T):
    """The automatic path streams at T=64 (2 slots per expert) and takes the grouped kernel at
    T=512 (16). Both paths run at both sizes: each matches the oracle on sampled rows, and
    they agree with each other within tolerance on every row."""
    L = synth.make_layer(**synth.HYBRID_256, kept=64, kept_format=synth.FMT_MXFP4, device="cuda")
    moe = U.build(L, T)
    x = synth.gen_x(T, L.H, seed=T, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    assert torch.isfinite(out.float()).all()
    auto_path = hm.hmoe_auto_path(moe.desc, T)
    assert auto_path == (hm.PATH_STREAM if T == 64 else hm.PATH_GROUPED)
    same, _ = U.run(moe, x, logits, path=auto_path)
    assert torch.equal(out, same)
    tokens = [0, T // 2, T - 1]
    ref = U.oracle_out(L, x, ids, gates, tokens=tokens)
    U.assert_rows_close(_rows(out, tokens), ref)
    other, _ = U.run(moe, x, logits, path=hm.PATH_GROUPED if auto_path == hm.PATH_STREAM else hm.PATH_STREAM)
    U.assert_rows_close(_rows(other, tokens), ref)
    U.assert_rows_close(other.float().cpu().numpy(), out.float().cpu().numpy())


@pytest.fixture(scope="module")
def uniform_layer():
    L = synth.make_layer(**synth.UNIFORM_128, uniform=True, device="cuda")
    return L, U.build(L, 8192)


@pytest.mark.parametrize("T", [1, 8, 128, 1024, 8192])
def test_uniform_nvfp4_sweep(uniform_layer, T):
    L, moe = uniform_layer
    x = synth.gen_x(T, L.H, seed=T, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    assert torch.isfinite(out.float()).all()
    tokens = sorted({0, T // 3, T - 1})
    U.assert_rows_close(_rows(out, tokens), U.oracle_out(L, x, ids, gates, tokens=tokens))
