"""Full-size workloads, in the launch configuration bench.py times.

The oracle (its per-expert steps spread over host processes, tests/oracle_pool.py)
checks, per token row within 2e-2 * max|ref|:
- every token where the batch is small (M <= 1024);
- at M=4096 and M=8192, for every routed expert the token of its first and of its
  last routed slot (so every expert of both tiers, and each expert's first and last,
  possibly ragged, token tile), plus a strided sample of tokens.
Properties that hold at any size cover every row:
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
    out, (ids, gates, perm, offsets) = U.run(moe, x, logits)
    assert torch.isfinite(out.float()).all()
    tokens = U.cover_tokens(ids, perm, offsets, stride=16)
    touched = set(np.unique(ids.cpu().numpy()).tolist())
    reached = set(np.unique(ids[tokens].cpu().numpy()).tolist())
    assert reached == touched and len(touched) == L.E        # every expert of both tiers
    U.assert_rows_close(_rows(out, tokens), U.oracle_rows(L, x, ids, gates, tokens=tokens))
    out2, _ = U.run(moe, x, logits, tier_order=hm.TIERS_KEPT_FIRST)
    assert torch.equal(out, out2)


def test_mxfp4_kept_tier_full_shape():
    """The automatic path streams at T=64 (2 slots per expert) and takes the grouped kernel at
    T=512 (16). Both paths run at both sizes: each matches the oracle on every row."""
    L = synth.make_layer(**synth.HYBRID_256, kept=64, kept_format=synth.FMT_MXFP4, device="cuda")
    moe = U.build(L, 512)
    xs, ids_all, gates_all, outs = [], [], [], []
    for T in (64, 512):
        x = synth.gen_x(T, L.H, seed=T, device="cuda")
        logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
        out, (ids, gates, _, _) = U.run(moe, x, logits)
        assert torch.isfinite(out.float()).all()
        auto_path = hm.hmoe_auto_path(moe.desc, T)
        assert auto_path == (hm.PATH_STREAM if T == 64 else hm.PATH_GROUPED)
        same, _ = U.run(moe, x, logits, path=auto_path)
        assert torch.equal(out, same)
        other, _ = U.run(moe, x, logits, path=hm.PATH_GROUPED if auto_path == hm.PATH_STREAM else hm.PATH_STREAM)
        xs.append(x)
        ids_all.append(ids)
        gates_all.append(gates)
        outs.append((out, other))
    # one oracle pass over both batches, so each expert is dequantised once
    ref = U.oracle_rows(L, torch.cat(xs), torch.cat(ids_all), torch.cat(gates_all))
    r0 = 0
    for out, other in outs:
        n = out.shape[0]
        U.assert_rows_close(out.float().cpu().numpy(), ref[r0:r0 + n])
        U.assert_rows_close(other.float().cpu().numpy(), ref[r0:r0 + n])
        r0 += n


@pytest.fixture(scope="module")
def uniform_layer():
    L = synth.make_layer(**synth.UNIFORM_128, uniform=True, device="cuda")
    return L, U.build(L, 8192)


@pytest.mark.parametrize("T", [1, 8, 128, 1024, 8192])
def test_uniform_nvfp4_sweep(uniform_layer, T):
    L, moe = uniform_layer
    x = synth.gen_x(T, L.H, seed=T, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
    out, (ids, gates, perm, offsets) = U.run(moe, x, logits)
    assert torch.isfinite(out.float()).all()
    tokens = list(range(T)) if T <= 1024 else U.cover_tokens(ids, perm, offsets, stride=16)
    U.assert_rows_close(_rows(out, tokens), U.oracle_rows(L, x, ids, gates, tokens=tokens))
