"""Layer oracle: the hybrid W4A16 SwiGLU mixture-of-experts layer, dequantise-then-matmul.

TEST INFRASTRUCTURE ONLY: see the package docstring.

[P1] "How it works": each MoE layer holds two tier-local weight sets. Both
tiers use one route geometry and sum into one output (topk_sum). [P3]
"Summary" and "What's in this PR", item 1: W4A16 means the weights are
4-bit and the activations stay 16-bit, with no activation scales. Each
expert is a SwiGLU feed-forward block with W13 [2I, H] (gate rows 0..I-1,
then up rows I..2I-1) and W2 [H, I].

For token t and slot j, with e = ids[t, j]:
    gu      = W13_e @ float(x[t])                 (float64)
    h       = silu(gu[:I]) * gu[I:]               silu(z) = z / (1 + exp(-z))
    y       = W2_e @ h
    out[t] += gates[t, j] * y                     (summed over j in slot order)

All arithmetic is float64. The final bf16 rounding of the output is left to
the comparison: the reference value is the float64 sum.

Experts are supplied through ``get_expert(e)``. It returns a dict with keys
``fmt``, ``w13`` and ``w2``. Each of ``w13`` and ``w2`` is a tuple
(codes, scales, g) in the logical layout of ``oracle.formats``. This lets a
caller stream experts one at a time at full size. An optional key ``act``
("bf16", the default, or "f16") names the layer's activation type, to which
the weights are dequantised ([P3] "Summary", item 2).

W4A4 ([P3] "Summary": the W4A4 NVFP4 scheme, activations quantised to NVFP4
as they arrive): an optional key ``act_quant`` = (g13, g2) holds the static
global scales of the two activations. Then x is replaced by
actquant.fake_quant(x, g13) before W13, and h, rounded to the activation type
(it is an activation of the layer), by actquant.fake_quant(h, g2) before W2.
"""

import numpy as np

from . import actquant, formats


def silu(z):
    return z / (1.0 + np.exp(-z))


def expert_weights(ex, H, I):
    """Dequantised (W13 [2I, H], W2 [H, I]) float64 for one expert dict."""
    fmt = ex["fmt"]
    c13, s13, g13 = ex["w13"]
    c2, s2, g2 = ex["w2"]
    act = ex.get("act", "bf16")
    w13 = formats.dequant(fmt, c13, s13, g13, H, act)
    w2 = formats.dequant(fmt, c2, s2, g2, I, act)
    assert w13.shape == (2 * I, H) and w2.shape == (H, I)
    return w13, w2


def round_act(h, act):
    """h rounded to the activation type (through fp32, as the kernels form h in fp32)."""
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32).astype(np.float64)
    return formats.bf16_rne(h32) if act == "bf16" else formats.f16_rne(h32)


def expert_ffn(w13, w2, xf, I, out_rows=None, act_quant=None, act="bf16"):
    """SwiGLU FFN of one expert on a batch of rows xf [n, H] -> [n, H] (or [n, len(out_rows)]).

    act_quant = (g13, g2): the W4A4 activation quantisation (module docstring)."""
    if act_quant is not None:
        xf = actquant.fake_quant(xf, act_quant[0])
    gu = xf @ w13.T                       # [n, 2I]
    h = silu(gu[:, :I]) * gu[:, I:]       # [n, I]
    if act_quant is not None:
        h = actquant.fake_quant(round_act(h, act), act_quant[1])
    w2r = w2 if out_rows is None else w2[out_rows]
    return h @ w2r.T


def moe_forward(x, ids, gates, get_expert, H, I, tokens=None, cols=None):
    """Reference layer output, float64 [len(tokens), len(cols)].

    x      -- activations [T, H]. Any float dtype; bf16 callers pass float32 views.
    ids    -- int [T, k]. gates -- float [T, k].
    tokens -- optional subset of token indices (default: all).
    cols   -- optional subset of output columns (default: all H).
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    gates = np.asarray(gates, dtype=np.float64)
    T, k = ids.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    ncol = H if cols is None else len(cols)
    # y[t_local, j] holds each slot's expert output. Slots are grouped by expert
    # so that each expert is dequantised once. The sum over j runs afterwards,
    # in slot order.
    y = np.zeros((len(tokens), k, ncol), dtype=np.float64)
    sub_ids = ids[tokens]
    for e in np.unique(sub_ids):
        tl, jj = np.nonzero(sub_ids == e)
        ex = get_expert(int(e))
        w13, w2 = expert_weights(ex, H, I)
        y[tl, jj] = expert_ffn(w13, w2, x[tokens[tl]], I, out_rows=cols, act_quant=ex.get("act_quant"),
                               act=ex.get("act", "bf16"))
    out = np.zeros((len(tokens), ncol), dtype=np.float64)
    for j in range(k):
        out += gates[tokens, j][:, None] * y[:, j]
    return out
