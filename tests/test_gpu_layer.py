"""GPU layer parity against the oracle, plus the invariances the method has.

Tolerance: per token row, max|out - ref| <= 2e-2 * max|ref| (fp32 accumulation).
"""

import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    L = synth.tiny_layer(device="cuda")
    return L, U.build(L, 256)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 9, 37, 200])
@pytest.mark.parametrize("order", [hm.TIERS_ONE_LAUNCH, hm.TIERS_KEPT_FIRST, hm.TIERS_NF3_FIRST])
def test_tiny_layer_parity(tiny, T, order):
    L, moe = tiny
    x = synth.gen_x(T, L.H, seed=T, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=T, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits, tier_order=order)
    U.assert_rows_close(out.float().cpu().numpy(), U.oracle_out(L, x, ids, gates))


def test_tier_order_is_bitwise_invariant(tiny):
    L, moe = tiny
    for T in (4, 37):
        x = synth.gen_x(T, L.H, device="cuda")
        logits = synth.gen_logits(T, L.E, device="cuda")
        outs = [U.run(moe, x, logits, tier_order=o)[0] for o in (0, 1, 2)]
        assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_token_order_is_bitwise_invariant(tiny):
    L, moe = tiny
    for T in (8, 37):
        x = synth.gen_x(T, L.H, device="cuda")
        logits = synth.gen_logits(T, L.E, device="cuda")
        p = torch.randperm(T, generator=torch.Generator().manual_seed(T)).cuda()
        a, _ = U.run(moe, x, logits)
        b, _ = U.run(moe, x[p].contiguous(), logits[p].contiguous())
        assert torch.equal(a[p], b)


def test_stream_path_equals_decode_path_tolerance(tiny):
    L, moe = tiny
    x = synth.gen_x(8, L.H, device="cuda")
    logits = synth.gen_logits(8, L.E, device="cuda")
    a, (ids, gates, _, _) = U.run(moe, x, logits)
    ref = U.oracle_out(L, x, ids, gates)
    U.assert_rows_close(a.float().cpu().numpy(), ref)


@pytest.mark.parametrize("kept_format", [synth.FMT_NVFP4, synth.FMT_MXFP4])
def test_odd_k_block_counts(kept_format):
    """I=192: W2 has 3 k-blocks and W13 has 3 row tiles, so the last row pair of the CTA-pair
    kernel has no row tile for the second CTA (and the one-CTA kernel's last item holds one).
    Both grouped kernels and the streaming path match the oracle on every row."""
    L = synth.make_layer(384, 192, 8, 2, kept_ids=[0, 3, 5], kept_format=kept_format, device="cuda")
    T = 96
    moe = U.build(L, T)
    x = synth.gen_x(T, L.H, seed=11, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=11, device="cuda")
    g, (ids, gates, _, _) = U.run(moe, x, logits, path=hm.PATH_GROUPED)
    g1, _ = U.run(moe, x, logits, path=hm.PATH_GROUPED, debug_flags=hm.DEBUG_GROUPED_PAIR)
    s, _ = U.run(moe, x, logits, path=hm.PATH_STREAM)
    ref = U.oracle_out(L, x, ids, gates)
    U.assert_rows_close(g.float().cpu().numpy(), ref)
    U.assert_rows_close(g1.float().cpu().numpy(), ref)
    U.assert_rows_close(s.float().cpu().numpy(), ref)
    U.assert_rows_close(g.float().cpu().numpy(), s.float().cpu().numpy())


@pytest.mark.parametrize("kept_format", [synth.FMT_NVFP4, synth.FMT_MXFP4])
def test_stream_pair_items_with_odd_row_tile_counts(kept_format):
    """H=384, I=192: W13 and W2 both have 3 row tiles, so the streaming kernel's last item of
    each phase holds one tile when its items are pairs of row tiles. 512 experts, top-8 and
    T=64 give min(T * topk, E) = 512 token groups, enough W13 pair items per CTA (2 pairs x 512
    against 2 per CTA) for the host to choose pair items on any GPU of up to 256 SMs. Every
    token is checked against the oracle, on both tier orders."""
    L = synth.make_layer(384, 192, 512, 8, kept=128, kept_format=kept_format, device="cuda")
    T = 64
    moe = U.build(L, T)
    x = synth.gen_x(T, L.H, seed=21, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=21, device="cuda")
    s, (ids, gates, _, _) = U.run(moe, x, logits, path=hm.PATH_STREAM)
    U.assert_rows_close(s.float().cpu().numpy(), U.oracle_out(L, x, ids, gates))
    s2, _ = U.run(moe, x, logits, path=hm.PATH_STREAM, tier_order=hm.TIERS_KEPT_FIRST)
    assert torch.equal(s, s2)


def test_top1_single_expert_and_repeat_calls(tiny):
    """top-1 (gate = 1) reduces to one dense expert; repeated calls are bitwise stable."""
    Lh = synth.make_layer(256, 128, 8, 1, kept_ids=[1, 5], device="cuda")
    moe = U.build(Lh, 64)
    x = synth.gen_x(16, 256, device="cuda")
    logits = synth.gen_logits(16, 8, device="cuda")
    a, (ids, gates, _, _) = U.run(moe, x, logits)
    assert torch.all(gates == 1.0)
    U.assert_rows_close(a.float().cpu().numpy(), U.oracle_out(Lh, x, ids, gates))
    b, _ = U.run(moe, x, logits)
    assert torch.equal(a, b)


def test_all_nvfp4_bitmap_equals_uniform_layer():
    H, I, E, k = 256, 128, 8, 2
    hybrid = synth.make_layer(H, I, E, k, kept_ids=list(range(E)), device="cuda")
    uniform = synth.make_layer(H, I, E, k, uniform=True, device="cuda")
    mh, mu = U.build(hybrid, 64), U.build(uniform, 64)
    for T in (3, 40):
        x = synth.gen_x(T, H, device="cuda")
        logits = synth.gen_logits(T, E, device="cuda")
        a, _ = U.run(mh, x, logits)
        b, _ = U.run(mu, x, logits)
        assert torch.equal(a, b)


def test_all_nf3_layer():
    L = synth.make_layer(256, 128, 8, 2, kept_ids=[], device="cuda")
    moe = U.build(L, 16)
    x = synth.gen_x(6, 256, device="cuda")
    logits = synth.gen_logits(6, 8, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    U.assert_rows_close(out.float().cpu().numpy(), U.oracle_out(L, x, ids, gates))


@pytest.mark.parametrize("T", [1, 8, 64])
def test_mxfp4_kept_tier(T):
    L = synth.make_layer(512, 256, 16, 4, kept_ids=[0, 3, 6, 9], kept_format=synth.FMT_MXFP4, device="cuda")
    moe = U.build(L, 64)
    x = synth.gen_x(T, L.H, device="cuda")
    logits = synth.gen_logits(T, L.E, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    U.assert_rows_close(out.float().cpu().numpy(), U.oracle_out(L, x, ids, gates))


@pytest.mark.parametrize("T", [1, 8, 128])
def test_uniform_nvfp4_shape(T):
    """The uniform single-tier NVFP4 layer shape (H=2048, I=768, E=128, top-8)."""
    L = synth.make_layer(**synth.UNIFORM_128, uniform=True, device="cuda")
    moe = U.build(L, 128)
    x = synth.gen_x(T, L.H, device="cuda")
    logits = synth.gen_logits(T, L.E, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    tokens = list(range(min(T, 6)))
    ref = U.oracle_out(L, x, ids, gates, tokens=tokens)
    U.assert_rows_close(out[tokens].float().cpu().numpy(), ref)


@pytest.fixture(scope="module")
def hybrid256():
    L = synth.make_layer(**synth.HYBRID_256, kept=64, device="cuda")
    return L, U.build(L, 8)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_full_size_hybrid_decode(hybrid256, T):
    """256-expert hybrid layer (H=6144, I=2048, top-8; 64 NVFP4 + 192 NF3) at M <= 8, in the
    launch configuration bench.py times. Every token is checked against the oracle (every
    routed expert of the batch, both tiers)."""
    L, moe = hybrid256
    x = synth.gen_x(T, L.H, seed=100 + T, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=100 + T, device="cuda")
    out, (ids, gates, _, _) = U.run(moe, x, logits)
    U.assert_rows_close(out.float().cpu().numpy(), U.oracle_rows(L, x, ids, gates))
    assert torch.isfinite(out.float()).all()
    out2, _ = U.run(moe, x, logits, tier_order=hm.TIERS_NF3_FIRST)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("T", [200, 1200])
def test_grouped_pair_kernel_matches_single_cta_kernel(tiny, T):
    """The grouped path's one-CTA kernel (the default) and its CTA-pair kernel
    (tcgen05.mma.cta_group::2, 256-slot token tiles) agree with the oracle; T=1200 puts about
    300 slots on each expert, so experts span several token tiles with a ragged last one."""
    L, _ = tiny
    moe = U.build(L, T)
    x = synth.gen_x(T, L.H, seed=T + 1, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=T + 1, device="cuda")
    single, (ids, gates, _, _) = U.run(moe, x, logits, path=hm.PATH_GROUPED)
    pair, _ = U.run(moe, x, logits, path=hm.PATH_GROUPED, debug_flags=hm.DEBUG_GROUPED_PAIR)
    ref = U.oracle_out(L, x, ids, gates)
    U.assert_rows_close(single.float().cpu().numpy(), ref)
    U.assert_rows_close(pair.float().cpu().numpy(), ref)
    for order in (hm.TIERS_KEPT_FIRST, hm.TIERS_NF3_FIRST):
        o, _ = U.run(moe, x, logits, path=hm.PATH_GROUPED, tier_order=order)
        assert torch.equal(o, single)


@pytest.mark.parametrize("T", [8, 4200])
def test_stream_path_one_and_two_launch_forms(tiny, T):
    """The streaming path runs W13 and W2 in one launch while its token groups fit the counter
    array, and as two launches past it (T=4200 on this layer). Both match the oracle on sampled
    rows and the grouped path within tolerance, in every tier order."""
    L, _ = tiny
    moe = U.build(L, T)
    x = synth.gen_x(T, L.H, seed=7, device="cuda")
    logits = synth.gen_logits(T, L.E, seed=7, device="cuda")
    s, (ids, gates, _, _) = U.run(moe, x, logits, path=hm.PATH_STREAM)
    tokens = sorted({0, 1, T // 2, T - 1})
    U.assert_rows_close(s.float().cpu().numpy()[tokens], U.oracle_out(L, x, ids, gates, tokens=tokens))
    for order in (hm.TIERS_KEPT_FIRST, hm.TIERS_NF3_FIRST):
        o, _ = U.run(moe, x, logits, path=hm.PATH_STREAM, tier_order=order)
        assert torch.equal(o, s)
    if T > 8:
        g, _ = U.run(moe, x, logits, path=hm.PATH_GROUPED)
        U.assert_rows_close(s.float().cpu().numpy(), g.float().cpu().numpy())


@pytest.mark.parametrize("T", [4, 300])
def test_stage_events_outside_capture(tiny, T):
    """Stage events given to an eager (not captured) forward are recorded in order on its stream."""
    L, _ = tiny
    moe = U.build(L, T)
    x = synth.gen_x(T, L.H, device="cuda")
    ids, gates, perm, offsets = moe.plan(synth.gen_logits(T, L.E, device="cuda"))
    out = torch.empty((T, L.H), dtype=torch.bfloat16, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in ev:
        e.record()  # creates the events; the library records them again below
    ev[0].record()
    hm.hmoe_forward(moe.layer, x, ids, gates, perm, offsets, out, moe.ws, stage_events=ev[1:])
    torch.cuda.synchronize()
    hm.hmoe_check_device_status(moe.ws)
    for a, b in zip(ev[:-1], ev[1:]):
        assert a.elapsed_time(b) >= 0.0
