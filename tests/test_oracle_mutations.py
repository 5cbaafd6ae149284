"""Planted mistakes: every oracle function is pinned tightly enough that a plausible slip fails a pin.

Each case below replaces one function of the oracle, for the length of one
test, by a copy carrying a single mistake of the kind a careful reader could
still make: a wrong exponent bias, a dropped sign or term, a reversed bit or
nibble order, a wrong tie rule, a shifted index, a swapped operand, a scale
applied at the wrong step. The named pins from ``tests/test_oracle_*.py`` are
then run against the mutated oracle, and each must fail with an assertion (not
a crash): the pin sees the wrong numbers. A last case runs the same pins on
the unmutated oracle and expects them to pass.

Nothing here touches the CUDA path: the mistakes are planted in the oracle, on
the CPU.
"""

import functools

import numpy as np
import pytest

from oracle import actquant, formats, layer, linear, route
from tests import test_oracle_actquant as PA
from tests import test_oracle_formats as PF
from tests import test_oracle_layer as PL
from tests import test_oracle_linear as PN
from tests import test_oracle_route as PR

_e2m1 = formats.e2m1_value
_e4m3 = formats.e4m3_value
_e8m0 = formats.e8m0_value
_unpack_nibbles = formats.unpack_nibbles
_dequant_tile = formats.dequant_tile
_topk = route.topk_ids
_silu = layer.silu


# ---------------------------------------------------------------- formats
def e2m1_bias0(code):
    """Exponent bias 0 instead of 1: every normal value doubled."""
    c = np.asarray(code, dtype=np.int64)
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e * 1.0))
    return np.where(s == 1, -mag, mag)


def e2m1_unsigned(code):
    """Sign bit ignored."""
    return np.abs(_e2m1(code))


def e4m3_bias8(byte):
    """Exponent bias 8 instead of 7."""
    return _e4m3(byte) * 0.5


def e4m3_subnormal_as_normal(byte):
    """Exponent field 0 decoded with the implicit leading 1."""
    b = np.asarray(byte, dtype=np.int64)
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    mag = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e8m0_bias128(byte):
    return _e8m0(byte) * 0.5


def nibbles_high_first(codes, K):
    """Element 2i read from the high nibble."""
    out = _unpack_nibbles(codes, K)
    return np.stack([out[:, 1::2], out[:, 0::2]], axis=2).reshape(out.shape)


def nf3_msb_first_code(codes, K):
    """The three bits of each code read most significant first."""
    c = np.asarray(codes, dtype=np.uint8)
    bits = np.unpackbits(c, axis=1, bitorder="little").astype(np.int64)[:, : 3 * K].reshape(c.shape[0], K, 3)
    return (bits[:, :, 0] << 2) | (bits[:, :, 1] << 1) | bits[:, :, 2]


def nf3_big_endian_bytes(codes, K):
    """The bitstream read from each byte's most significant bit."""
    c = np.asarray(codes, dtype=np.uint8)
    bits = np.unpackbits(c, axis=1, bitorder="big").astype(np.int64)[:, : 3 * K].reshape(c.shape[0], K, 3)
    return bits[:, :, 0] | (bits[:, :, 1] << 1) | (bits[:, :, 2] << 2)


def bf16_truncate(x):
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)


def bf16_ties_away(x):
    """Round half up on the dropped 16 bits (ties not to even)."""
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + np.uint64(0x8000)) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def f16_variant(emin=-14, frac_bits=10):
    def f16(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, e2 = np.frexp(a)
        e = np.where(a > 0, e2 - 1, emin)
        q = np.exp2(np.maximum(e, emin) - float(frac_bits))
        r = np.rint(a / q) * q
        r = np.where(r > 65504.0, np.inf, r)
        return np.copysign(r, x)
    return f16


def normalfloat_variant(offset_rule="mean", normalise=True):
    from scipy.stats import norm

    def levels(bits):
        n = 2 ** bits
        if offset_rule == "mean":
            offset = 0.5 * ((1.0 - 1.0 / (2 * (n - 1))) + (1.0 - 1.0 / (2 * n)))
        else:                                  # only one of the two candidates
            offset = 1.0 - 1.0 / (2 * n)
        pos = norm.ppf(np.linspace(offset, 0.5, n // 2 + 1)[:-1])
        neg = -norm.ppf(np.linspace(offset, 0.5, n // 2)[:-1])
        v = np.sort(np.concatenate([pos, neg, [0.0]]))
        return v / v.max() if normalise else v
    return levels


def nf3_codebook_unrounded():
    return formats.normalfloat_levels(3)


def dequant_tile_variant(nvfp4_expand="repeat", nf3_round=True, nf3_reversed=False):
    def tile(fmt, codes, scales, K, act="bf16"):
        if fmt == formats.FMT_NVFP4:
            v = formats.e2m1_value(formats.unpack_nibbles(codes, K))
            s = formats.e4m3_value(np.asarray(scales, dtype=np.uint8))
            # "tile" repeats the scale row instead of each scale: column k takes scale k % (K/16)
            sx = np.repeat(s, 16, axis=1) if nvfp4_expand == "repeat" else np.tile(s, (1, 16))
            t = v * sx
            return t if act == "bf16" else formats.act_rne(t, act)
        if fmt == formats.FMT_NF3:
            cb = formats.nf3_codebook()
            cb = cb[::-1] if nf3_reversed else cb
            v = cb[formats.unpack_nf3(codes, K)]
            t = v * np.repeat(formats.bf16_bits_to_f64(np.asarray(scales, dtype=np.uint16)), 64, axis=1)
            return formats.act_rne(t, act) if nf3_round else t
        return _dequant_tile(fmt, codes, scales, K, act)
    return tile


def dequant_without_global_scale(fmt, codes, scales, g, K, act="bf16"):
    return formats.dequant_tile(fmt, codes, scales, K, act)


# ---------------------------------------------------------------- route
def topk_ties_to_higher_id(logits, k):
    l = np.asarray(logits, dtype=np.float32)
    E = l.shape[1]
    return (E - 1 - np.argsort(-l[:, ::-1], axis=1, kind="stable"))[:, :k].astype(np.int32)


def topk_ascending_ids(logits, k):
    """The right set, listed by expert id instead of by descending logit."""
    return np.sort(_topk(logits, k), axis=1)


def gates_not_renormalised(logits, ids):
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    z = np.exp(l - l.max(axis=1, keepdims=True))
    return np.take_along_axis(z / z.sum(axis=1, keepdims=True), np.asarray(ids, dtype=np.int64), axis=1)


def gates_negated(logits, ids):
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    chosen = -np.take_along_axis(l, np.asarray(ids, dtype=np.int64), axis=1)
    z = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def permutation_descending_slots(ids, E):
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    perm = np.lexsort((-np.arange(flat.size), flat)).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]).astype(np.int32)
    return perm, offsets


def permutation_inclusive_offsets(ids, E):
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E)
    return perm, np.concatenate([np.cumsum(counts), [flat.size]]).astype(np.int32)


# ---------------------------------------------------------------- layer
def silu_wrong_sign(z):
    return z / (1.0 + np.exp(z))


def _swiglu(gu, I):
    return layer.silu(gu[:, :I]) * gu[:, I:]


def ffn_variant(h_of=_swiglu, g_x=0, g_h=1, quant_x=True):
    def ffn(w13, w2, xf, I, out_rows=None, act_quant=None, act="bf16"):
        if act_quant is not None and quant_x:
            xf = actquant.fake_quant(xf, act_quant[g_x])
        gu = xf @ w13.T
        h = h_of(gu, I)
        if act_quant is not None:
            h = actquant.fake_quant(layer.round_act(h, act), act_quant[g_h])
        w2r = w2 if out_rows is None else w2[out_rows]
        return h @ w2r.T
    return ffn


def moe_forward_variant(weight="gate", x_rows="tokens"):
    def moe(x, ids, gates, get_expert, H, I, tokens=None, cols=None):
        x = np.asarray(x, dtype=np.float64)
        ids = np.asarray(ids)
        gates = np.asarray(gates, dtype=np.float64)
        T, k = ids.shape
        tokens = np.arange(T) if tokens is None else np.asarray(tokens)
        ncol = H if cols is None else len(cols)
        y = np.zeros((len(tokens), k, ncol))
        sub = ids[tokens]
        for e in np.unique(sub):
            tl, jj = np.nonzero(sub == e)
            ex = get_expert(int(e))
            w13, w2 = layer.expert_weights(ex, H, I)
            rows = x[tokens[tl]] if x_rows == "tokens" else x[tl]
            y[tl, jj] = layer.expert_ffn(w13, w2, rows, I, out_rows=cols, act_quant=ex.get("act_quant"),
                                         act=ex.get("act", "bf16"))
        out = np.zeros((len(tokens), ncol))
        for j in range(k):
            if weight == "gate":
                out += gates[tokens, j][:, None] * y[:, j]
            elif weight == "none":
                out += y[:, j]
            else:                               # the gate of the mirrored slot
                out += gates[tokens, k - 1 - j][:, None] * y[:, j]
        return out
    return moe


# ---------------------------------------------------------------- actquant
def e2m1_rne_variant(tie_up=False, keep_negative_zero=False):
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def rne(v):
        v = np.asarray(v, dtype=np.float32)
        a = np.abs(v).astype(np.float64)
        codes = np.zeros(a.shape, dtype=np.int64)
        for m in range(1, 8):
            mid = 0.5 * (mags[m - 1] + mags[m])
            up = True if tie_up else (m & 1) == 0
            codes += (a > mid) | ((a == mid) & up)
        sign = np.signbit(v) if keep_negative_zero else np.signbit(v) & (codes > 0)
        return (codes | (sign.astype(np.int64) << 3)).astype(np.uint8)
    return rne


def e4m3_rne_variant(ties="even"):
    def rne(t):
        t = np.asarray(t, dtype=np.float64)
        vals = formats.e4m3_value(np.arange(0x7F, dtype=np.int64))
        i = np.clip(np.searchsorted(vals, t, side="left"), 1, len(vals) - 1)
        lo, hi = vals[i - 1], vals[i]
        if ties == "odd":
            down = (t - lo < hi - t) | ((t - lo == hi - t) & ((i & 1) == 0))
        else:                                    # truncation: down unless exactly on hi
            down = t < hi
        code = np.where(t <= vals[0], 0, np.where(t >= vals[-1], len(vals) - 1, np.where(down, i - 1, i)))
        return code.astype(np.uint8)
    return rne


def quantize_variant(max_code=6.0, g_in_step=True, swap_nibbles=False):
    def quantize(a, g):
        a = np.asarray(a, dtype=np.float32)
        R, K = a.shape
        g32 = np.float32(g)
        blocks = a.reshape(R, K // 16, 16)
        t = np.minimum(np.abs(blocks).max(axis=2) / np.float32(np.float32(max_code) * g32), np.float32(448.0))
        s = actquant.e4m3_rne_sat(t)
        d = formats.e4m3_value(s).astype(np.float32)
        d = (d * g32).astype(np.float32) if g_in_step else d
        safe = np.where(d > 0, d, np.float32(1.0))
        v = np.where(d[:, :, None] > 0, (blocks / safe[:, :, None]).astype(np.float32), np.float32(0.0))
        codes = actquant.e2m1_rne_sat(v).reshape(R, K)
        lo, hi = (codes[:, 1::2], codes[:, 0::2]) if swap_nibbles else (codes[:, 0::2], codes[:, 1::2])
        return (lo | (hi << 4)).astype(np.uint8), s
    return quantize


# ---------------------------------------------------------------- linear
def linear_without_global_scale(x, fmt, codes, scales, g, K, act="bf16"):
    return np.asarray(x, dtype=np.float64) @ formats.dequant_tile(fmt, codes, scales, K, act).T


def linear_ignores_act(x, fmt, codes, scales, g, K, act="bf16"):
    return np.asarray(x, dtype=np.float64) @ formats.dequant(fmt, codes, scales, g, K).T


_lin_bf16 = functools.partial(PN.test_linear_matches_scalar_loops_all_formats, "bf16")
_lin_f16 = functools.partial(PN.test_linear_matches_scalar_loops_all_formats, "f16")

# (case id, module, attribute, replacement, pins that must each fail)
CASES = [
    ("e2m1 exponent bias 0", formats, "e2m1_value", e2m1_bias0, [PF.test_e2m1_matches_golden_table]),
    ("e2m1 sign dropped", formats, "e2m1_value", e2m1_unsigned,
     [PF.test_e2m1_matches_golden_table, _lin_bf16]),
    ("e4m3 exponent bias 8", formats, "e4m3_value", e4m3_bias8,
     [PF.test_e4m3_all_codes_match_torch, PF.test_nvfp4_exact_roundtrip_through_encoder]),
    ("e4m3 subnormals with implicit 1", formats, "e4m3_value", e4m3_subnormal_as_normal,
     [PF.test_e4m3_all_codes_match_torch]),
    ("e8m0 bias 128", formats, "e8m0_value", e8m0_bias128,
     [PF.test_e8m0_all_codes, PF.test_mxfp4_exact_roundtrip_and_closed_form]),
    ("nibble order swapped", formats, "unpack_nibbles", nibbles_high_first,
     [PF.test_unpack_nibbles_fixture_and_encoder_roundtrip, _lin_bf16]),
    ("nf3 code bits msb first", formats, "unpack_nf3", nf3_msb_first_code,
     [PF.test_unpack_nf3_against_bigint_reader_and_encoder, PF.test_nf3_exact_roundtrip_through_encoder]),
    ("nf3 bytes read big-endian", formats, "unpack_nf3", nf3_big_endian_bytes,
     [PF.test_unpack_nf3_against_bigint_reader_and_encoder, _lin_bf16]),
    ("bf16 truncation", formats, "bf16_rne", bf16_truncate, [PF.test_bf16_rne_matches_torch]),
    ("bf16 ties away from even", formats, "bf16_rne", bf16_ties_away, [PF.test_bf16_rne_matches_torch]),
    ("fp16 min exponent -15", formats, "f16_rne", f16_variant(emin=-15),
     [PF.test_f16_rne_matches_numpy_and_torch, PF.test_f16_rne_closed_form_cases]),
    ("fp16 with 9 fraction bits", formats, "f16_rne", f16_variant(frac_bits=9),
     [PF.test_f16_rne_matches_numpy_and_torch, PF.test_f16_nf3_tile_rounds_the_product_once]),
    ("normalfloat one-sided offset", formats, "normalfloat_levels", normalfloat_variant(offset_rule="one"),
     [PF.test_normalfloat_construction_reproduces_published_nf4, PF.test_nf3_codebook_matches_golden_and_invariants]),
    ("normalfloat not normalised", formats, "normalfloat_levels", normalfloat_variant(normalise=False),
     [PF.test_normalfloat_construction_reproduces_published_nf4, PF.test_nf3_codebook_matches_golden_and_invariants]),
    ("nf3 codebook not rounded to bf16", formats, "nf3_codebook", nf3_codebook_unrounded,
     [PF.test_nf3_codebook_matches_golden_and_invariants]),
    ("nvfp4 scale index k mod groups", formats, "dequant_tile", dequant_tile_variant(nvfp4_expand="tile"),
     [PF.test_nvfp4_exact_roundtrip_through_encoder, _lin_bf16]),
    ("nf3 product not rounded", formats, "dequant_tile", dequant_tile_variant(nf3_round=False),
     [PF.test_nf3_exact_roundtrip_through_encoder, _lin_bf16]),
    ("nf3 codebook reversed", formats, "dequant_tile", dequant_tile_variant(nf3_reversed=True),
     [PF.test_nf3_exact_roundtrip_through_encoder, _lin_bf16]),
    ("nvfp4 global scale dropped", formats, "dequant", dequant_without_global_scale,
     [PF.test_nvfp4_exact_roundtrip_through_encoder, PF.test_nvfp4_relative_error_is_bounded]),
    ("top-k ties to the higher id", route, "topk_ids", topk_ties_to_higher_id,
     [PR.test_topk_brute_force_with_forced_ties]),
    ("top-k listed by id", route, "topk_ids", topk_ascending_ids,
     [PR.test_topk_brute_force_with_forced_ties, PR.test_topk_matches_torch_on_tie_free_data,
      PR.test_tiny_route_fixture]),
    ("gates not renormalised", route, "gates", gates_not_renormalised,
     [PR.test_gates_renormalised_softmax, PR.test_tiny_route_fixture]),
    ("gates of negated logits", route, "gates", gates_negated,
     [PR.test_gates_renormalised_softmax, PR.test_tiny_route_fixture]),
    ("perm descending within expert", route, "permutation", permutation_descending_slots,
     [PR.test_permutation_and_offsets_invariants, PR.test_tiny_route_fixture]),
    ("offsets inclusive", route, "permutation", permutation_inclusive_offsets,
     [PR.test_permutation_and_offsets_invariants, PR.test_tiny_route_fixture]),
    ("silu sign flipped", layer, "silu", silu_wrong_sign,
     [PL.test_vectorised_oracle_matches_scalar_loops, PL.test_top1_reduces_to_dense_expert_torch]),
    ("gate and up swapped", layer, "expert_ffn", ffn_variant(h_of=lambda gu, I: layer.silu(gu[:, I:]) * gu[:, :I]),
     [PL.test_vectorised_oracle_matches_scalar_loops, PL.test_top1_reduces_to_dense_expert_torch,
      PN.test_linear_is_the_layer_w2_step]),
    ("gate and up rows interleaved", layer, "expert_ffn",
     ffn_variant(h_of=lambda gu, I: layer.silu(gu[:, 0::2]) * gu[:, 1::2]),
     [PL.test_vectorised_oracle_matches_scalar_loops, PL.test_top1_reduces_to_dense_expert_torch]),
    ("w4a4 x and h scales swapped", layer, "expert_ffn", ffn_variant(g_x=1, g_h=0),
     [PA.test_w4a4_top1_layer_order_of_steps]),
    ("w4a4 x not quantised", layer, "expert_ffn", ffn_variant(quant_x=False),
     [PA.test_w4a4_top1_layer_order_of_steps]),
    ("gate weight dropped", layer, "moe_forward", moe_forward_variant(weight="none"),
     [PL.test_vectorised_oracle_matches_scalar_loops, PL.test_gate_linearity_and_subsets]),
    ("gate of the mirrored slot", layer, "moe_forward", moe_forward_variant(weight="mirrored"),
     [PL.test_vectorised_oracle_matches_scalar_loops]),
    ("token subset indexes x locally", layer, "moe_forward", moe_forward_variant(x_rows="local"),
     [PL.test_gate_linearity_and_subsets]),
    ("e2m1 ties away from zero", actquant, "e2m1_rne_sat", e2m1_rne_variant(tie_up=True),
     [PA.test_e2m1_rounding_matches_encoder_and_ties]),
    ("e2m1 negative zero code", actquant, "e2m1_rne_sat", e2m1_rne_variant(keep_negative_zero=True),
     [PA.test_e2m1_rounding_matches_encoder_and_ties]),
    ("e4m3 ties to odd", actquant, "e4m3_rne_sat", e4m3_rne_variant(ties="odd"),
     [PA.test_e4m3_rounding_matches_torch_including_ties]),
    ("e4m3 truncation", actquant, "e4m3_rne_sat", e4m3_rne_variant(ties="truncate"),
     [PA.test_e4m3_rounding_matches_torch_including_ties, PA.test_quantizer_equals_weight_encoder_on_the_same_data]),
    ("block scale from amax / 4", actquant, "quantize", quantize_variant(max_code=4.0),
     [PA.test_quantizer_equals_weight_encoder_on_the_same_data, PA.test_exact_round_trip_on_the_nvfp4_grid]),
    ("block step without g", actquant, "quantize", quantize_variant(g_in_step=False),
     [PA.test_quantizer_equals_weight_encoder_on_the_same_data, PA.test_exact_round_trip_on_the_nvfp4_grid]),
    ("activation nibbles swapped", actquant, "quantize", quantize_variant(swap_nibbles=True),
     [PA.test_quantizer_equals_weight_encoder_on_the_same_data, PA.test_exact_round_trip_on_the_nvfp4_grid]),
    ("linear without global scale", linear, "linear_forward", linear_without_global_scale, [_lin_bf16, _lin_f16]),
    ("linear ignores the activation type", linear, "linear_forward", linear_ignores_act, [_lin_f16]),
]


def _name(pin):
    return getattr(pin, "__name__", None) or f"{pin.func.__name__}[{pin.args[0]}]"


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_fails_its_pins(monkeypatch, case):
    _, module, attr, mutant, pins = case
    assert callable(getattr(module, attr))
    monkeypatch.setattr(module, attr, mutant)
    survived = []
    for pin in pins:
        try:
            pin()
        except AssertionError:
            continue
        survived.append(_name(pin))
    assert not survived, f"pins passed with the mistake planted: {survived}"


def test_pins_pass_on_the_unmutated_oracle():
    pins = {_name(p): p for c in CASES for p in c[4]}
    for pin in pins.values():
        pin()
