"""GPU routing parity: ids, perm and offsets are bit-exact with the oracle, and gates agree to 1e-6."""

import numpy as np
import pytest
import torch

import synth
from oracle import route
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layers():
    dev = "cuda"
    return {
        (8, 2): U.build(synth.make_layer(128, 64, 8, 2, kept_ids=[0, 1, 2, 3], device=dev), 4096),
        (256, 8): U.build(synth.make_layer(128, 64, 256, 8, kept=64, device=dev), 8192),
        (128, 8): U.build(synth.make_layer(128, 64, 128, 8, uniform=True, device=dev), 8192),
        (384, 6): U.build(synth.make_layer(128, 64, 384, 6, uniform=True, device=dev), 4096),
        (512, 8): U.build(synth.make_layer(128, 64, 512, 8, uniform=True, device=dev), 4096),
    }


def _check(moe, logits, k):
    ids, gates, perm, offsets = moe.plan(logits)
    torch.cuda.synchronize()
    rids, rg, rperm, roff = route.plan(logits.cpu().numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert np.array_equal(perm.cpu().numpy(), rperm)
    assert np.array_equal(offsets.cpu().numpy(), roff)
    assert np.max(np.abs(gates.cpu().numpy().astype(np.float64) - rg), initial=0.0) <= 1e-6


@pytest.mark.parametrize("E,k", [(8, 2), (256, 8), (128, 8)])
@pytest.mark.parametrize("T", [1, 2, 4, 8, 33, 127, 128, 129, 1000, 4096])
def test_route_parity(layers, E, k, T):
    logits = synth.gen_logits(T, E, seed=T, device="cuda")
    _check(layers[(E, k)], logits, k)


def test_route_ties_and_skew(layers):
    moe = layers[(256, 8)]
    logits = synth.gen_logits(300, 256, seed=5, device="cuda")
    logits[::2] = torch.round(logits[::2] * 2) / 2        # many exact ties
    logits[7] = 0.25                                      # a fully tied row
    logits[9, 3] = -0.0
    logits[9, 4] = 0.0
    _check(moe, logits, 8)
    beta, ratio = synth.calibrate_zipf_beta(4096, 256, 8, device="cuda", iters=20)
    biased = synth.gen_logits(4096, 256, device="cuda") + synth.zipf_bias(256, beta, device="cuda")
    _check(moe, biased, 8)
    assert ratio > 5.0


@pytest.mark.parametrize("T", [16, 300])
def test_route_signed_zero_ties_in_topk(layers, T):
    """Equal logits of opposite sign (-0 and +0) inside the top-k tie like any equal values, so
    the lower expert id comes first, on the one-CTA path (T=16) and the chunked path (T=300)."""
    moe = layers[(256, 8)]
    logits = synth.gen_logits(T, 256, seed=11, device="cuda")
    logits[3] = -1.0
    logits[3, 5] = -0.0
    logits[3, 2] = 0.0
    logits[3, 9] = 0.0
    logits[3, 200] = -0.0                                 # top-4: 2, 5, 9, 200; then -1 ties by id
    logits[4] = -0.0
    logits[4, ::3] = 0.0                                  # a row of signed zeros: ids 0..7
    _check(moe, logits, 8)
    ids, _, _, _ = moe.plan(logits)
    assert ids[3].tolist() == [2, 5, 9, 200, 0, 1, 3, 4]
    assert ids[4].tolist() == list(range(8))


@pytest.mark.parametrize("E,k", [(384, 6), (512, 8)])
@pytest.mark.parametrize("T", [5, 127, 170, 4096])
def test_route_parity_wide_expert_counts(layers, E, k, T):
    """Expert counts that do not divide the scan CTA's 1024 threads (E=384: 768 of them take
    part) or fill it with two chunk ranges per expert (E=512), on both routing paths."""
    logits = synth.gen_logits(T, E, seed=T + E, device="cuda")
    _check(layers[(E, k)], logits, k)


def test_route_large_batch(layers):
    logits = synth.gen_logits(8192, 128, seed=3, device="cuda")
    _check(layers[(128, 8)], logits, 8)


def test_route_zero_tokens(layers):
    moe = layers[(8, 2)]
    logits = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    ids, gates, perm, offsets = moe.plan(logits)
    torch.cuda.synchronize()
    assert offsets.cpu().tolist() == [0] * 9
