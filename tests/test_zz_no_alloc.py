"""The allocation-free forward, hmoe_forward_static, called through the C ABI.

Some callers cannot allocate device memory. Their host gives the library
only input and output buffers under a fixed device-memory plan, or the code
must never reach the allocator or cudaFree's device-wide synchronisation.
Such callers cannot provide a workspace. hmoe_forward_static runs the same
layer with its scratch in a fixed device array inside the library.

These tests make two calls in a row, on different batches, and on both
paths (the weight-streaming kernel at small batches, the tensor-core grouped
kernel above), for bf16, fp16 and W4A4 layers. Both entry points run the same deterministic kernels, so each
result must equal the workspace entry point's, hmoe_forward, bit for bit.
Batches whose scratch exceeds the array, and calls with bad arguments, are
refused before anything is enqueued.
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
    if shape == "tiny-f16":
        return synth.make_layer(**synth.TINY, kept_ids=[0, 1, 2, 3], device="cuda", act="f16")
    if shape == "tiny-w4a4":
        L = synth.tiny_layer(device="cuda")
        L.act_quant = (5.0 / (6 * 448), 0.6 / (6 * 448))
        return L
    return synth.make_layer(**synth.UNIFORM_128, uniform=True, device="cuda")


def _build(L, max_tokens):
    if getattr(L, "act_quant", None) is None:
        return U.build(L, max_tokens)
    import nf3_moe_gb300 as hm
    return hm.HybridMoELayer(L.H, L.I, L.E, L.topk, [int(b) for b in L.bit_map], U.device_experts(L),
                             max_tokens=max_tokens, act_globals=L.act_quant)


# (layer, tokens of the two calls): the tiny layer (E=8, top-2) takes the grouped path at
# T=64 (128 slots > 8 per expert); the 128-expert layer streams at every T here.
CASES = [("tiny", (4, 8)), ("tiny", (64, 37)), ("uniform", (4, 8)), ("uniform", (64, 1)),
         ("tiny-f16", (8, 64)), ("tiny-w4a4", (8, 64))]


@pytest.mark.parametrize("shape,Ts", CASES)
def test_static_forward_equals_workspace_forward_two_calls(shape, Ts):
    L = _layer(shape)
    moe = _build(L, max(Ts))
    for call, T in enumerate(Ts):
        x = synth.gen_x(T, L.H, seed=50 + call, device="cuda", dtype=L.x_dtype)
        logits = synth.gen_logits(T, L.E, seed=50 + call, device="cuda")
        ids, gates, perm, offsets = moe.plan(logits)
        ref = torch.empty((T, L.H), dtype=L.x_dtype, device="cuda")
        out = torch.full((T, L.H), float("nan"), dtype=L.x_dtype, device="cuda")
        assert _forward_ws(moe, x, ids, gates, perm, offsets, ref) == 0, _lib.lib().hmoe_last_error()
        assert _forward_static(moe, x, ids, gates, perm, offsets, out) == 0, _lib.lib().hmoe_last_error()
        torch.cuda.synchronize()
        assert _lib.lib().hmoe_check_device_status_static(_stream()) == 0, _lib.lib().hmoe_last_error()
        assert torch.equal(out, ref), f"{shape} T={T}: static and workspace forwards differ"


def test_static_forward_refuses_bad_arguments_before_enqueueing():
    L = _layer("tiny")
    moe = U.build(L, 8)
    T = 4
    x = synth.gen_x(T, L.H, device="cuda")
    ids, gates, perm, offsets = moe.plan(synth.gen_logits(T, L.E, device="cuda"))
    out = torch.zeros((T, L.H), dtype=torch.bfloat16, device="cuda")
    assert _lib.lib().hmoe_forward_static(moe.layer.handle, _ptr(x), T, _ptr(ids), _ptr(gates), _ptr(perm),
                                          ctypes.c_void_p(0), _ptr(out), _stream()) == -1
    assert _lib.lib().hmoe_forward_static(moe.layer.handle, ctypes.c_void_p(x.data_ptr() + 2), T, _ptr(ids),
                                          _ptr(gates), _ptr(perm), _ptr(offsets), _ptr(out), _stream()) == -1
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


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
