"""The binding's host-side tensor checks, on CPU.

The library sees raw pointers only, so the Python binding checks each tensor it passes
(dtype, shape or byte size, contiguity, device) before calling it. Here:
* the argument sets the GPU tests and the bench build (the same synthetic layers, made on
  the CPU) pass every check but the device one;
* each kind of wrong tensor is refused with a ValueError naming the argument;
* the public calls refuse CPU tensors before the library is reached.
"""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    from nf3_moe_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()


def _layer_args(L):
    bm = None if L.bit_map is None else [int(b) for b in L.bit_map]
    act = hm.ACT_F16 if L.act == "f16" else hm.ACT_BF16
    desc = hm.LayerDesc(L.H, L.I, L.E, L.topk, L.kept_format, act)
    experts = [(ex["w13"][0], ex["w13"][1], ex["w13"][2], ex["w2"][0], ex["w2"][1], ex["w2"][2])
               for ex in L.experts]
    kb, nb = hm.hmoe_packed_size(desc, bm)
    kept = torch.empty(max(kb, 16), dtype=torch.uint8) if kb else None
    nf3 = torch.empty(max(nb, 16), dtype=torch.uint8) if nb else None
    return desc, bm, experts, kept, nf3


def _route_bufs(desc, T):
    k, E = desc.topk, desc.E
    return (torch.empty((T, k), dtype=torch.int32), torch.empty((T, k), dtype=torch.float32),
            torch.empty((T * k,), dtype=torch.int32), torch.empty((E + 1,), dtype=torch.int32))


LAYERS = {
    "tiny": lambda: synth.tiny_layer(),
    "tiny-f16": lambda: synth.make_layer(256, 128, 8, 2, kept_ids=[0, 1, 2, 3], act="f16"),
    "uniform": lambda: synth.make_layer(128, 64, 8, 2, uniform=True),
    "mxfp4-f16": lambda: synth.make_layer(384, 192, 8, 2, kept_ids=[0, 3, 5], kept_format=synth.FMT_MXFP4,
                                          act="f16"),
    "all-nf3": lambda: synth.make_layer(128, 64, 4, 2, kept_ids=[]),
}


@pytest.mark.parametrize("name", sorted(LAYERS))
def test_legitimate_arguments_pass(name):
    L = LAYERS[name]()
    desc, bm, experts, kept, nf3 = _layer_args(L)
    hm._check_pack(desc, bm, experts, kept, nf3, cuda=False)
    ws = torch.empty(hm.hmoe_workspace_size(desc, 64), dtype=torch.uint8)
    for T in (0, 1, 8, 64):
        x = synth.gen_x(T, L.H, dtype=L.x_dtype)
        logits = synth.gen_logits(T, L.E)
        ids, gates, perm, offsets = _route_bufs(desc, T)
        out = torch.empty((T, L.H), dtype=L.x_dtype)
        hm._check_plan(desc, logits, ids, gates, perm, offsets, ws, cuda=False)
        hm._check_forward(desc, x, ids, gates, perm, offsets, out, ws, cuda=False)
        hm._check_forward(desc, x, ids, gates, perm, offsets, out, None, cuda=False)


def test_wrong_tensors_are_named():
    L = synth.tiny_layer()
    desc, bm, experts, kept, nf3 = _layer_args(L)
    T = 5
    x = synth.gen_x(T, L.H)
    ids, gates, perm, offsets = _route_bufs(desc, T)
    out = torch.empty((T, L.H), dtype=torch.bfloat16)
    ws = torch.empty(1024, dtype=torch.uint8)
    good = dict(x=x, ids=ids, gates=gates, perm=perm, offsets=offsets, out=out, ws=ws)
    bad = {
        "x": [x.float(), x[:, :-128], torch.empty((L.H, T), dtype=torch.bfloat16).t()],
        "ids": [ids.long(), ids[:, :1], ids.t()],
        "gates": [gates.double(), gates.reshape(-1)],
        "perm": [perm[:-1], perm.reshape(T, -1)],
        "offsets": [offsets[:-1], offsets.float()],
        "out": [out.float(), out[:-1], torch.empty((L.H, T), dtype=torch.bfloat16).t()],
        "ws": [ws[::2]],
    }
    for name, cases in bad.items():
        for b in cases:
            args = dict(good, **{name: b})
            with pytest.raises(ValueError, match=rf"^{name} "):
                hm._check_forward(desc, args["x"], args["ids"], args["gates"], args["perm"], args["offsets"],
                                  args["out"], args["ws"], cuda=False)
    with pytest.raises(TypeError, match="gates"):
        hm._check_forward(desc, x, ids, gates.numpy(), perm, offsets, out, ws, cuda=False)
    with pytest.raises(ValueError, match="logits"):
        hm._check_plan(desc, synth.gen_logits(T, L.E + 1), ids, gates, perm, offsets, ws, cuda=False)
    with pytest.raises(ValueError, match="logits"):
        hm._check_plan(desc, synth.gen_logits(T, L.E).double(), ids, gates, perm, offsets, ws, cuda=False)


def test_pack_buffers_and_checkpoint_sizes():
    L = synth.tiny_layer()
    desc, bm, experts, kept, nf3 = _layer_args(L)
    kb, nb = hm.hmoe_packed_size(desc, bm)
    with pytest.raises(ValueError, match="kept_buf"):
        hm._check_pack(desc, bm, experts, kept[:kb - 1], nf3, cuda=False)
    assert kb > 0 and nb > 0
    with pytest.raises(ValueError, match="nf3_buf"):
        hm._check_pack(desc, bm, experts, kept, nf3[:nb - 16], cuda=False)
    nf3_e = next(e for e in range(L.E) if bm[e] == 3)
    kept_e = next(e for e in range(L.E) if bm[e] == 4)
    for e, slot, label in ((nf3_e, 0, "W13 codes"), (kept_e, 1, "W13 scales"), (nf3_e, 4, "W2 scales"),
                           (kept_e, 3, "W2 codes")):
        ex = list(experts[e])
        ex[slot] = ex[slot].reshape(-1)[:-1]
        args = list(experts)
        args[e] = tuple(ex)
        with pytest.raises(ValueError, match=f"expert {e} {label}"):
            hm._check_pack(desc, bm, args, kept, nf3, cuda=False)
    with pytest.raises(ValueError, match="experts"):
        hm._check_pack(desc, bm, experts[:-1], kept, nf3, cuda=False)
    with pytest.raises(hm.HmoeError) as ei:                       # the library's bit map check
        hm._check_pack(desc, [4] * (L.E - 1) + [2], experts, kept, nf3, cuda=False)
    assert ei.value.status == -4


def test_matrix_bytes_match_the_encoder():
    rng = np.random.default_rng(0)
    for fmt in (synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_NF3):
        for N, K in ((128, 256), (256, 384), (64, 640)):
            w = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32))
            c, s, _ = synth.quantise(fmt, w)
            assert hm._matrix_bytes(fmt, N, K) == (hm._nbytes(c), hm._nbytes(s)), (fmt, N, K)


def test_linear_checks():
    desc = hm.LinearDesc(256, 384, hm.FMT_NF3, hm.ACT_F16)
    ws = torch.empty(4096, dtype=torch.uint8)
    x = torch.empty((7, 384), dtype=torch.float16)
    out = torch.empty((7, 256), dtype=torch.float16)
    hm._check_linear_forward(desc, x, out, ws, cuda=False)
    for bad_x, bad_out, name in ((x.bfloat16(), out, "x"), (x[:, :128], out, "x"), (x, out[:6], "out"),
                                 (x, out.bfloat16(), "out")):
        with pytest.raises(ValueError, match=rf"^{name} "):
            hm._check_linear_forward(desc, bad_x, bad_out, ws, cuda=False)


def test_public_calls_refuse_host_tensors():
    """The calls check before touching the library: host tensors never reach it."""
    L = synth.tiny_layer()
    desc, bm, experts, kept, nf3 = _layer_args(L)
    layer = hm.Layer(None, desc, None, None)                    # no library handle is needed to refuse
    T = 4
    x = synth.gen_x(T, L.H)
    ids, gates, perm, offsets = _route_bufs(desc, T)
    out = torch.empty((T, L.H), dtype=torch.bfloat16)
    ws = torch.empty(hm.hmoe_workspace_size(desc, T), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        hm.hmoe_plan_routes(layer, synth.gen_logits(T, L.E), ids, gates, perm, offsets, ws)
    with pytest.raises(ValueError, match="CUDA"):
        hm.hmoe_forward(layer, x, ids, gates, perm, offsets, out, ws)
    with pytest.raises(ValueError, match="CUDA"):
        hm.hmoe_forward_static(layer, x, ids, gates, perm, offsets, out)
    with pytest.raises(ValueError, match="CUDA"):
        hm.hmoe_pack_weights(desc, bm, experts, kept, nf3)
    with pytest.raises(ValueError, match="CUDA"):
        hm.hmoe_quantize_act_nvfp4(x, 1.0, torch.empty((T, L.H // 2), dtype=torch.uint8),
                                   torch.empty((T, L.H // 16), dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        hm.hmoe_debug_dequant(layer, 0, 13, torch.empty((2 * L.I, L.H), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="dst"):
        hm.hmoe_debug_dequant(layer, 0, 2, torch.empty((2 * L.I, L.H), dtype=torch.bfloat16))
