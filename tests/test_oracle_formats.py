"""Pins for oracle.formats: element decoders, codebook, bf16 and fp16 rounding, unpacking, dequant.

Each check ties the oracle to something outside itself: a library conversion
(torch float8 / bfloat16), a golden fixture with its citation, an independent
bit reader, or the encoder in ``synth``, written separately.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from tests.conftest import read_golden


def test_e2m1_matches_golden_table():
    rows = read_golden("e2m1_values.txt")
    codes = np.array([int(r[0]) for r in rows])
    want = np.array([float(r[1]) for r in rows])
    got = F.e2m1_value(codes)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
    assert set(np.abs(got).tolist()) == {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}


def test_e4m3_all_codes_match_torch():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    got = F.e4m3_value(b)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e8m0_all_codes():
    b = np.arange(256, dtype=np.uint8)
    got = F.e8m0_value(b)
    assert np.isnan(got[255])
    assert np.array_equal(got[:255], np.ldexp(1.0, np.arange(255) - 127))
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.from_numpy(b).view(torch.float8_e8m0fnu).to(torch.float32).double().numpy()
        assert np.array_equal(got[:255], ref[:255])


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        # exact ties: low 16 bits == 0x8000, both parities of the kept lsb
        (np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x40C08000, 0x00018000], dtype=np.uint32)
         .view(np.float32)),
        np.array([0.0, -0.0, 1.0, 65504.0, 3.0e38], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).double().numpy()
    got = F.bf16_rne(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rne_rejects_non_fp32_inputs():
    with pytest.raises(ValueError):
        F.bf16_rne(np.array([1.0 + 2.0 ** -40]))


def _f16_grid(fine=False):
    """Every finite fp16 value, its neighbours' midpoints (exact ties), and points just off them:
    one fp32 ulp off (fp32-exact inputs), or with fine=True a few float64 ulps off."""
    bits = np.arange(0, 0x7C00, dtype=np.uint16)          # +0 .. largest finite
    v = bits.view(np.float16).astype(np.float64)
    mid = 0.5 * (v[:-1] + v[1:])                           # exact in fp32 (12 significant bits)
    off = np.spacing(mid) * 4 if fine else np.spacing(mid.astype(np.float32)).astype(np.float64)
    pts = np.concatenate([v, mid, mid + off, mid - off, [65519.0, 65520.0, 65536.0, 1e6, 2.0 ** -25,
                                                         3 * 2.0 ** -26, 2.0 ** -26]])
    return np.concatenate([pts, -pts])


def test_f16_rne_matches_numpy_and_torch():
    # torch rounds float64 to fp16 through fp32, so it is a reference only on
    # fp32-exact inputs; numpy rounds float64 directly.
    x = _f16_grid()
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
    got = F.f16_rne(x)
    ref_t = torch.from_numpy(x).to(torch.float16).double().numpy()
    assert np.array_equal(got, ref_t)
    assert np.array_equal(np.signbit(got), np.signbit(ref_t))
    with np.errstate(over="ignore"):
        assert np.array_equal(got, x.astype(np.float16).astype(np.float64))
        xf = _f16_grid(fine=True)
        assert np.array_equal(F.f16_rne(xf), xf.astype(np.float16).astype(np.float64))


def test_f16_rne_closed_form_cases():
    # Ties go to the even significand; the largest finite value is 65504;
    # 65520 (the midpoint to 2**16) rounds to infinity; 2**-25 (half the
    # smallest subnormal) rounds to 0, 3 * 2**-26 to 2**-24.
    cases = {1.0 + 2.0 ** -11: 1.0, 1.0 + 3 * 2.0 ** -11: 1.0 + 2.0 ** -9, 65519.0: 65504.0,
             65520.0: np.inf, 2.0 ** -25: 0.0, 3 * 2.0 ** -26: 2.0 ** -24, 2.0 ** -14: 2.0 ** -14,
             -2.5 * 2.0 ** -24: -2.0 * 2.0 ** -24}
    for x, want in cases.items():
        assert F.f16_rne(np.array([x]))[0] == want, x


def test_act_rne_dispatch():
    x = np.array([1.0 + 2.0 ** -9])                       # exact in fp16, not in bf16
    assert F.act_rne(x, "f16")[0] == x[0]
    assert F.act_rne(x, "bf16")[0] == 1.0
    with pytest.raises(ValueError):
        F.act_rne(x, "fp8")


def test_f16_tiles_nvfp4_mxfp4_are_the_exact_products():
    # Inside the fp16 ranges every NVFP4 and MXFP4 tile value is exact in fp16,
    # so the fp16 tile equals the (exact) bf16 tile.
    rng = np.random.default_rng(11)
    N, K = 8, 128
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    e4m3 = rng.integers(0, 0x7F, size=(N, K // 16)).astype(np.uint8)      # every finite positive E4M3
    e4m3[0, :] = np.arange(K // 16) + 0x76                                  # up to 448 = 0x7E
    e4m3[0, -1] = 0x01                                                      # the smallest subnormal
    a = F.dequant_tile(F.FMT_NVFP4, codes, e4m3, K, "f16")
    assert np.array_equal(a, F.dequant_tile(F.FMT_NVFP4, codes, e4m3, K))
    e8 = rng.integers(104, 141, size=(N, K // 32)).astype(np.uint8)
    e8[0] = [104, 140, 127, 120]
    b = F.dequant_tile(F.FMT_MXFP4, codes, e8, K, "f16")
    assert np.array_equal(b, F.dequant_tile(F.FMT_MXFP4, codes, e8, K))
    assert np.isfinite(b).all()
    # Just outside: b = 141 with code 6 (0x7) overflows fp16, b = 102 with code 0.5 underflows to 0.
    c1 = np.full((1, 16), 0x77, dtype=np.uint8)
    hi = F.dequant_tile(F.FMT_MXFP4, c1, np.full((1, 1), 141, np.uint8), 32, "f16")
    assert np.isinf(hi).all()
    c2 = np.full((1, 16), 0x11, dtype=np.uint8)
    lo = F.dequant_tile(F.FMT_MXFP4, c2, np.full((1, 1), 102, np.uint8), 32, "f16")
    assert np.all(lo == 0.0)


def test_f16_nf3_tile_rounds_the_product_once():
    cb = F.nf3_codebook()
    idx = np.tile(np.arange(8), 16).reshape(1, 128)
    codes = synth.pack_nf3_bits(torch.from_numpy(idx)).numpy()
    # scale 1 and powers of two: the codebook itself, scaled exactly (every
    # entry has at most 8 significant bits, so fits fp16's 11)
    for sc in (1.0, 2.0 ** -6, 2.0 ** 5):
        sbits = np.full((1, 2), torch.tensor(sc, dtype=torch.bfloat16).view(torch.int16).item(), np.int64)
        t = F.dequant_tile(F.FMT_NF3, codes, sbits.astype(np.uint16), 128, "f16")
        assert np.array_equal(t[0], cb[idx[0]] * sc)
    # a general scale: within half an fp16 ulp of the exact product, and the
    # nearest fp16 value (checked against numpy's conversion)
    sb = 0x3D4B                                            # bf16 0.0495...
    s = F.bf16_bits_to_f64(np.array([sb]))[0]
    t = F.dequant_tile(F.FMT_NF3, codes, np.full((1, 2), sb, np.uint16), 128, "f16")[0]
    exact = cb[idx[0]] * s
    assert np.array_equal(t, exact.astype(np.float16).astype(np.float64))
    assert np.all(np.abs(t - exact) <= np.abs(exact) * 2.0 ** -11)
    assert not np.array_equal(t, F.bf16_rne(exact))      # fp16 keeps bits bf16 drops


def test_normalfloat_construction_reproduces_published_nf4():
    want = np.array([float(r[0]) for r in read_golden("nf4_qlora.txt")])
    got = F.normalfloat_levels(4)
    assert got.shape == (16,)
    assert np.max(np.abs(got - want)) < 1e-6


def test_nf3_codebook_matches_golden_and_invariants():
    rows = read_golden("nf3_codebook.txt")
    bits = np.array([int(r[1], 16) for r in rows], dtype=np.uint16)
    vals = np.array([float(r[2]) for r in rows])
    cb = F.nf3_codebook()
    assert np.array_equal(cb, vals)
    assert np.array_equal(F.bf16_bits_to_f64(bits), vals)
    assert cb.shape == (8,) and np.all(np.diff(cb) > 0)
    assert cb[0] == -1.0 and cb[3] == 0.0 and cb[7] == 1.0
    # every entry is a bf16 value: low 16 bits of the fp32 pattern are zero
    assert np.all(cb.astype(np.float32).view(np.uint32) & 0xFFFF == 0)
    # the encoder's private copy agrees
    assert tuple(int(b) for b in bits) == synth.NF3_BF16_BITS


def test_unpack_nibbles_fixture_and_encoder_roundtrip():
    assert F.unpack_nibbles(np.array([[0x21, 0xF0]], dtype=np.uint8), 4).tolist() == [[1, 2, 0, 15]]
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 16, size=(5, 64))
    packed = synth._pack_nibbles(torch.from_numpy(codes)).numpy()
    assert np.array_equal(F.unpack_nibbles(packed, 64), codes)


def test_unpack_nf3_against_bigint_reader_and_encoder():
    rng = np.random.default_rng(3)
    K = 128
    codes = rng.integers(0, 8, size=(6, K))
    packed = synth.pack_nf3_bits(torch.from_numpy(codes)).numpy()
    assert packed.shape == (6, 3 * K // 8)
    got = F.unpack_nf3(packed, K)
    assert np.array_equal(got, codes)
    # independent reader: the row as one little-endian integer
    for r in range(6):
        big = int.from_bytes(bytes(packed[r].tolist()), "little")
        assert [(big >> (3 * j)) & 7 for j in range(K)] == codes[r].tolist()
    # hand fixture: codes 1..7,0 -> bits 001 010 011 100 101 110 111 000 (LSB first)
    eight = np.array([[1, 2, 3, 4, 5, 6, 7, 0]])
    v = sum(int(c) << (3 * j) for j, c in enumerate(eight[0]))
    fixture = np.array([[v & 0xFF, (v >> 8) & 0xFF, (v >> 16) & 0xFF]], dtype=np.uint8)
    assert fixture.tolist() == [[0xD1, 0x58, 0x1F]]
    assert np.array_equal(F.unpack_nf3(fixture, 8), eight)


def _nvfp4_exact_matrix(rng, N, K):
    """Weights that NVFP4 represents exactly: e2m1 * e4m3 * g with a power-of-two g."""
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    v = mags[rng.integers(0, 8, size=(N, K))] * rng.choice([-1, 1], size=(N, K))
    # each 16-group holds a 6 so the encoder picks back exactly the chosen scale
    v[:, ::16] = 6.0
    s = F.e4m3_value(rng.integers(0x30, 0x70, size=(N, K // 16)))
    s[0, 0] = 448.0                        # amax = 6*448*g, so the encoder's g equals g
    g = 2.0 ** -10
    return v * np.repeat(s, 16, axis=1) * g


def test_nvfp4_exact_roundtrip_through_encoder():
    rng = np.random.default_rng(4)
    w = _nvfp4_exact_matrix(rng, 8, 64)
    wt = torch.from_numpy(w.astype(np.float32))
    c, s, g = synth.quant_nvfp4(wt)
    back = F.dequant(F.FMT_NVFP4, c.numpy(), s.numpy(), g, 64)
    assert g == 2.0 ** -10
    assert np.array_equal(back, w)
    tile = F.dequant_tile(F.FMT_NVFP4, c.numpy(), s.numpy(), 64)
    assert np.array_equal(tile * g, back)


def test_mxfp4_exact_roundtrip_and_closed_form():
    rng = np.random.default_rng(5)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    v = mags[rng.integers(0, 8, size=(4, 64))] * rng.choice([-1, 1], size=(4, 64))
    v[:, ::32] = 6.0                       # amax_b = 6 * 2**X -> floor(log2) - 2 = X
    X = rng.integers(-20, 20, size=(4, 2))
    w = v * np.exp2(np.repeat(X, 32, axis=1))
    c, s = synth.quant_mxfp4(torch.from_numpy(w.astype(np.float32)))
    assert np.array_equal(s.numpy().astype(np.int64) - 127, X)
    back = F.dequant(F.FMT_MXFP4, c.numpy(), s.numpy(), 1.0, 64)
    assert np.array_equal(back, w)


def test_nf3_exact_roundtrip_through_encoder():
    rng = np.random.default_rng(6)
    cb = F.nf3_codebook()
    idx = rng.integers(0, 8, size=(4, 128))
    idx[:, ::64] = 7                       # absmax of each group is exactly s
    s = F.bf16_rne(np.abs(rng.standard_normal((4, 2))).astype(np.float32).astype(np.float64))
    w = cb[idx] * np.repeat(s, 64, axis=1)   # fp32-exact (bf16 x bf16)
    c, sc = synth.quant_nf3(torch.from_numpy(w.astype(np.float32)))
    sc = sc.numpy().view(np.uint16)
    assert np.array_equal(F.bf16_bits_to_f64(sc), s)
    assert np.array_equal(F.unpack_nf3(c.numpy(), 128), idx)
    tile = F.dequant_tile(F.FMT_NF3, c.numpy(), sc, 128)
    assert np.array_equal(tile, F.bf16_rne(w))


def test_nf3_zero_group_and_dequant_error_bound():
    w = torch.zeros(2, 128)
    w[1, 64:] = torch.linspace(-1, 1, 64)
    c, s = synth.quant_nf3(w)
    codes = F.unpack_nf3(c.numpy(), 128)
    assert np.all(codes[0] == 3) and np.all(codes[1, :64] == 3)
    d = F.dequant(F.FMT_NF3, c.numpy(), s.numpy().view(np.uint16), 1.0, 128)
    assert np.all(d[0] == 0)
    # nearest-codebook rounding: error <= half the widest gap (times s) plus bf16 rounding
    cb = F.nf3_codebook()
    assert np.max(np.abs(d[1, 64:] - w[1, 64:].numpy())) <= 0.5 * np.max(np.diff(cb)) * 1.0 + 2 ** -8


def test_nvfp4_relative_error_is_bounded():
    w = synth.gen_master(0, 13, 64, 256)
    c, s, g = synth.quant_nvfp4(w)
    d = F.dequant(F.FMT_NVFP4, c.numpy(), s.numpy(), g, 256)
    wn = w.double().numpy()
    # per 16-group: |err| <= half the largest E2M1 step (1.0, between 4 and 6)
    # times the group scale; with s <= amax_b / 6 rounded, this is below amax_b / 4.
    amax_b = np.repeat(np.abs(wn).reshape(64, 16, 16).max(axis=2), 16, axis=1)
    assert np.all(np.abs(d - wn) <= amax_b / 4 + 1e-12)
