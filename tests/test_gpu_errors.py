"""Error paths on the GPU. None of them traps, faults or hangs: the kernels skip bad accesses,
bound every wait, and report through the workspace status word."""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    L = synth.tiny_layer(device="cuda")
    return L, U.build(L, 64)


def _inputs(L, T):
    return synth.gen_x(T, L.H, device="cuda"), synth.gen_logits(T, L.E, device="cuda")


def test_workspace_too_small_is_rejected_on_host(tiny):
    L, moe = tiny
    x, logits = _inputs(L, 8)
    ids, gates, perm, offsets = moe.plan(logits)
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    out = torch.empty((8, L.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_forward(moe.layer, x, ids, gates, perm, offsets, out, small)
    assert ei.value.status == -3


def test_bad_offsets_reported_and_context_survives(tiny):
    L, moe = tiny
    x, logits = _inputs(L, 8)
    ids, gates, perm, offsets = moe.plan(logits)
    bad = offsets.clone()
    bad[-1] += 5                                   # offsets[E] != T*k
    out = torch.empty((8, L.H), dtype=torch.bfloat16, device="cuda")
    hm.hmoe_forward(moe.layer, x, ids, gates, perm, bad, out, moe.ws)
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_check_device_status(moe.ws)
    assert ei.value.status == -7
    good, (i2, g2, _, _) = U.run(moe, x, logits)   # the context and the workspace still work
    U.assert_rows_close(good.float().cpu().numpy(), U.oracle_out(L, x, i2, g2))


@pytest.mark.parametrize("path", [hm.PATH_AUTO, hm.PATH_STREAM, hm.PATH_GROUPED])
def test_out_of_range_perm_reported(tiny, path):
    L, moe = tiny
    x, logits = _inputs(L, 37)
    ids, gates, perm, offsets = moe.plan(logits)
    bad = perm.clone()
    bad[3] = 10_000
    bad[5] = -4
    out = torch.empty((37, L.H), dtype=torch.bfloat16, device="cuda")
    hm.hmoe_forward(moe.layer, x, ids, gates, bad, offsets, out, moe.ws, path=path)
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_check_device_status(moe.ws)
    assert ei.value.status == -7
    U.run(moe, x, logits)


def test_bounded_wait_timeout_reported(tiny):
    """The producer issues nothing, so every consumer wait runs out after 2 ms; the call
    must finish and report HMOE_ERR_DEVICE_TIMEOUT, and the next call must work after
    re-initialising the workspace."""
    L, moe = tiny
    x, logits = _inputs(L, 4)
    ids, gates, perm, offsets = moe.plan(logits)
    out = torch.empty((4, L.H), dtype=torch.bfloat16, device="cuda")
    hm.hmoe_forward(moe.layer, x, ids, gates, perm, offsets, out, moe.ws, wait_limit_us=2000,
                    debug_flags=hm._lib.DEBUG_NO_COPIES)
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_check_device_status(moe.ws)
    assert ei.value.status == -6
    hm.hmoe_workspace_init(moe.ws)
    good, (i2, g2, _, _) = U.run(moe, x, logits)
    U.assert_rows_close(good.float().cpu().numpy(), U.oracle_out(L, x, i2, g2))


def test_bad_bitmap_and_shape_rejected():
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_packed_size(hm.LayerDesc(256, 128, 4, 2, 4), [4, 3, 2, 4])
    assert ei.value.status == -4
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_workspace_size(hm.LayerDesc(200, 128, 4, 2, 4), 8)
    assert ei.value.status == -2


GUARD = 4096      # canary bytes on each side of a caller buffer (keeps 256-byte alignment)
CANARY = 0xA5


def _guarded(nbytes):
    """A device buffer with CANARY bands of GUARD bytes around it: (whole allocation, inner view)."""
    full = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    return full, full[GUARD:GUARD + nbytes]


def _bands_intact(full, nbytes):
    return bool((full[:GUARD] == CANARY).all()) and bool((full[GUARD + nbytes:] == CANARY).all())


@pytest.mark.parametrize("T,path", [(8, hm.PATH_STREAM), (64, hm.PATH_STREAM), (64, hm.PATH_GROUPED)])
def test_no_write_outside_caller_buffers(tiny, T, path):
    """Routing and forward write nothing outside the workspace, the plan outputs and the layer
    output: canary bands around each are unchanged, and the result equals the unguarded run."""
    L, moe = tiny
    x, logits = _inputs(L, T)
    ws_bytes = hm.hmoe_workspace_size(moe.desc, T)
    ws_full, ws = _guarded(ws_bytes)
    hm.hmoe_workspace_init(ws)
    bands = {"workspace": (ws_full, ws_bytes)}

    def buffer(name, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        full, view = _guarded(nbytes)
        bands[name] = (full, nbytes)
        return view.view(dtype).view(shape)

    ids = buffer("ids", (T, L.topk), torch.int32)
    gates = buffer("gates", (T, L.topk), torch.float32)
    perm = buffer("perm", (T * L.topk,), torch.int32)
    offsets = buffer("offsets", (L.E + 1,), torch.int32)
    out = buffer("out", (T, L.H), torch.bfloat16)
    hm.hmoe_plan_routes(moe.layer, logits, ids, gates, perm, offsets, ws)
    hm.hmoe_forward(moe.layer, x, ids, gates, perm, offsets, out, ws, path=path)
    torch.cuda.synchronize()
    hm.hmoe_check_device_status(ws)
    for name, (full, nbytes) in bands.items():
        assert _bands_intact(full, nbytes), name
    ref, _ = U.run(moe, x, logits, path=path)
    assert torch.equal(out, ref)
