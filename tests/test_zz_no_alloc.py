"""The allocation-free forward, hmoe_forward_static, called through the C ABI.

Some callers cannot allocate device memory. Their host gives the library
only input and output buffers under a fixed device-memory plan, or the code
must never reach the allocator or cudaFree's device-wide synchronisation.
Such callers cannot provide a workspace. hmoe_forward_static runs the same
layer with its scratch in a fixed device array inside the library.

These tests make two calls in a row, on different batches. Each result must
agree with the workspace entry point, hmoe_forward, within the per-row
tolerance the other layer tests use. Batches whose scratch exceeds the
array are refused before anything runs.
"""

import ctypes

import pytest
import torch

import synth
from nf3_moe_gb300 import _lib
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _forward_static(moe, x, ids, gates, perm, offsets, out):
    return _lib.lib().hmoe_forward_static(moe.layer.handle, _ptr(x), x.shape[0], _ptr(ids), _ptr(gates), _ptr(perm),
                                          _ptr(offsets), _ptr(out), _stream())


def _forward_ws(moe, x, ids, gates, perm, offsets, out):
    ws = moe.ws
    return _lib.lib().hmoe_forward(moe.layer.handle, _ptr(x), x.shape[0], _ptr(ids), _ptr(gates), _ptr(perm),
                                   _ptr(offsets), _ptr(out), _ptr(ws), ws.numel(), _stream())


def _layer(shape):
    if shape == "tiny":
        return synth.tiny_layer(device="cuda")
    return synth.make_layer(**synth.UNIFORM_128, uniform=True, device="cuda")


@pytest.mark.parametrize("shape", ["tiny", "uniform"])
def test_static_forward_matches_workspace_forward_two_calls(shape):
    L = _layer(shape)
    moe = U.build(L, 8)
    for call, T in enumerate((4, 8)):
        x = synth.gen_x(T, L.H, seed=50 + call, device="cuda")
        logits = synth.gen_logits(T, L.E, seed=50 + call, device="cuda")
        ids, gates, perm, offsets = moe.plan(logits)
        ref = torch.empty((T, L.H), dtype=torch.bfloat16, device="cuda")
        out = torch.full((T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _forward_ws(moe, x, ids, gates, perm, offsets, ref) == 0, _lib.lib().hmoe_last_error()
        assert _forward_static(moe, x, ids, gates, perm, offsets, out) == 0, _lib.lib().hmoe_last_error()
        torch.cuda.synchronize()
        assert _lib.lib().hmoe_check_device_status_static(_stream()) == 0, _lib.lib().hmoe_last_error()
        U.assert_rows_close(out.float().cpu().numpy(), ref.float().cpu().numpy())


def test_static_forward_refuses_oversized_batch():
    L = _layer("uniform")
    moe = U.build(L, 8)
    T = 4096                                   # scratch for 32768 slots exceeds the array
    x = torch.zeros((T, L.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((T, L.topk), dtype=torch.int32, device="cuda")
    gates = torch.zeros((T, L.topk), dtype=torch.float32, device="cuda")
    perm = torch.zeros((T * L.topk,), dtype=torch.int32, device="cuda")
    offsets = torch.zeros((L.E + 1,), dtype=torch.int32, device="cuda")
    out = torch.zeros((T, L.H), dtype=torch.bfloat16, device="cuda")
    assert _forward_static(moe, x, ids, gates, perm, offsets, out) == -3
    assert b"static scratch" in _lib.lib().hmoe_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
