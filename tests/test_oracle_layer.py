"""Pins for oracle.layer on the tiny hybrid layer (T=4, H=256, I=128, E=8, top-2).

* a pure-Python scalar loop, written from the SwiGLU definition;
* top-1 routing reduces the layer to one dense expert, computed with torch
  float64 (F.silu, matmul);
* an all-NVFP4 bit map equals the uniform single-tier layer;
* permuting tokens permutes the output rows;
* zero gates on one slot leave only the other expert.
"""

import math

import numpy as np
import torch
import torch.nn.functional as Fn

import synth
from oracle import formats as F, layer, route

H, I, E, K = 256, 128, 8, 2


def _tiny():
    L = synth.tiny_layer()
    x = synth.gen_x(4, H).float().numpy().astype(np.float64)
    logits = synth.gen_logits(4, E).numpy()
    return L, x, logits


def test_vectorised_oracle_matches_scalar_loops():
    L, x, logits = _tiny()
    ids, g, _, _ = route.plan(logits, K)
    ref = layer.moe_forward(x, ids, g, L.expert_numpy, H, I)
    # scalar loops on 2 tokens x 6 output columns (full inner sums)
    cols = [0, 1, 77, 128, 200, 255]
    for t in (0, 3):
        for c in cols:
            acc = 0.0
            for j in range(K):
                ex = L.expert_numpy(int(ids[t, j]))
                w13, w2 = layer.expert_weights(ex, H, I)
                w13l, w2l, xl = w13.tolist(), w2.tolist(), x[t].tolist()
                hsum = 0.0
                for i in range(I):
                    gate = sum(w13l[i][kk] * xl[kk] for kk in range(H))
                    up = sum(w13l[I + i][kk] * xl[kk] for kk in range(H))
                    hsum += w2l[c][i] * (gate / (1.0 + math.exp(-gate)) * up)
                acc += float(g[t, j]) * hsum
            assert abs(acc - ref[t, c]) <= 1e-12 * max(1.0, abs(ref[t, c]))


def test_top1_reduces_to_dense_expert_torch():
    L, x, logits = _tiny()
    ids, g, _, _ = route.plan(logits, 1)
    assert np.all(g == 1.0)
    ref = layer.moe_forward(x, ids, g, L.expert_numpy, H, I)
    for t in range(4):
        e = int(ids[t, 0])
        ex = L.expert_numpy(e)
        c13, s13, g13 = ex["w13"]
        c2, s2, g2 = ex["w2"]
        w13 = torch.from_numpy(F.dequant(ex["fmt"], c13, s13, g13, H))
        w2 = torch.from_numpy(F.dequant(ex["fmt"], c2, s2, g2, I))
        xt = torch.from_numpy(x[t])
        gate, up = torch.matmul(w13, xt).split(I)
        dense = torch.matmul(w2, Fn.silu(gate) * up).numpy()
        assert np.max(np.abs(dense - ref[t])) <= 1e-12 * np.max(np.abs(dense))


def test_all_nvfp4_bit_map_equals_uniform_layer():
    hybrid = synth.make_layer(H, I, E, K, kept_ids=list(range(E)))
    uniform = synth.make_layer(H, I, E, K, uniform=True)
    assert hybrid.bit_map.tolist() == [4] * E and uniform.bit_map is None
    x = synth.gen_x(4, H).float().numpy().astype(np.float64)
    ids, g, _, _ = route.plan(synth.gen_logits(4, E).numpy(), K)
    a = layer.moe_forward(x, ids, g, hybrid.expert_numpy, H, I)
    b = layer.moe_forward(x, ids, g, uniform.expert_numpy, H, I)
    assert np.array_equal(a, b)


def test_token_permutation_permutes_rows():
    L, x, logits = _tiny()
    ids, g, _, _ = route.plan(logits, K)
    ref = layer.moe_forward(x, ids, g, L.expert_numpy, H, I)
    p = np.array([2, 0, 3, 1])
    ids2, g2, _, _ = route.plan(logits[p], K)
    out2 = layer.moe_forward(x[p], ids2, g2, L.expert_numpy, H, I)
    assert np.array_equal(out2, ref[p])


def test_gate_linearity_and_subsets():
    L, x, logits = _tiny()
    ids, g, _, _ = route.plan(logits, K)
    g0 = g.copy()
    g0[:, 1] = 0.0
    only_first = layer.moe_forward(x, ids, g0, L.expert_numpy, H, I)
    one = layer.moe_forward(x, ids[:, :1], g0[:, :1], L.expert_numpy, H, I)
    assert np.max(np.abs(only_first - one)) <= 1e-13 * np.max(np.abs(one))
    full = layer.moe_forward(x, ids, g, L.expert_numpy, H, I)
    sub = layer.moe_forward(x, ids, g, L.expert_numpy, H, I, tokens=[1, 3], cols=[5, 9, 250])
    want = full[[1, 3]][:, [5, 9, 250]]
    assert np.max(np.abs(sub - want)) <= 1e-13 * np.max(np.abs(want))


def test_f16_layer_differs_from_bf16_only_in_nf3_rounding():
    """The activation type enters the layer only through the NF3 tile rounding (fp16 keeps
    more bits of cb * s; NVFP4 and MXFP4 tiles are exact in both): with the same x, an
    all-kept layer gives identical results, and a hybrid one differs by at most one bf16
    rounding of each NF3 weight."""
    T = 6
    xs = synth.gen_x(T, 256, seed=4, dtype=torch.float16).float().numpy().astype(np.float64)
    logits = synth.gen_logits(T, 8, seed=4).numpy()
    ids, g, _, _ = route.plan(logits, 2)
    for kept in ([0, 1, 2, 3, 4, 5, 6, 7], [0, 1, 2, 3]):
        Lb = synth.make_layer(256, 128, 8, 2, kept_ids=kept, kept_format=synth.FMT_MXFP4)
        Lf = synth.make_layer(256, 128, 8, 2, kept_ids=kept, kept_format=synth.FMT_MXFP4, act="f16")
        ob = layer.moe_forward(xs, ids, g, Lb.expert_numpy, 256, 128)
        of = layer.moe_forward(xs, ids, g, Lf.expert_numpy, 256, 128)
        if len(kept) == 8:
            assert np.array_equal(ob, of)
        else:
            assert not np.array_equal(ob, of)
            assert np.abs(ob - of).max() <= 2.0 ** -8 * np.abs(ob).max()
