"""Seeded synthetic inputs for the hybrid W4A16 MoE layer.

This module is shared by the tests, the benchmark, and the oracle's callers.
It holds none of the layer's arithmetic: no dequantisation, routing or
matmul. It draws the inputs and encodes fp32 master weights into the logical
checkpoint layouts, as an offline quantiser would. The library under test
starts from those packed codes. It is written with torch tensor ops so the
same code runs on the CPU (small cases) or on the GPU (the 4.3 GB layers).
Each op is IEEE-exact or a correctly rounded division, so a given device
always produces the same bytes.

The recipe is that of the workloads in the design notes:
  * x ~ N(0, 1), rounded to bf16 (fp16 for fp16 layers); router logits
    ~ N(0, 1) in fp32.
  * Master weights ~ N(0, 0.02) in fp32, seeded per (seed, layer, expert,
    matrix). Any one expert can be regenerated alone.
  * NVFP4 quantiser. g = amax / (6 * 448), or 1 if amax = 0. Each 16-group
    scale is s = E4M3_rne(min(amax_b / (6 g), 448)). Codes are
    E2M1_rne_sat(w / (e4m3(s) g)), or 0 where s decodes to 0.
  * MXFP4 quantiser (OCP Microscaling v1.0). X = clamp(floor(log2 amax_b) - 2,
    -127, 127), or -127 where amax_b = 0. Codes are E2M1_rne_sat(w / 2**X).
  * NF3 quantiser. The per-64-group scale is s = bf16_rne(absmax). The code
    is the nearest codebook entry to w / s, with ties to the lower index.
    Where s = 0 every code is index 3 (the exact zero).

Encoder tables: the E2M1 decision thresholds and the NF3 codebook bit
patterns below are the encoder's own copy. The oracle derives its codebook
from the NormalFloat construction. The kernels carry their own copy of the
bit patterns. The tests check all three against each other and against
``tests/golden``.
"""

import numpy as np
import torch

FMT_NF3, FMT_NVFP4, FMT_MXFP4 = 3, 4, 5

# NF3 codebook, bf16 bit patterns, index 0..7 (encoder copy).
NF3_BF16_BITS = (0xBF80, 0xBF09, 0xBE7D, 0x0000, 0x3E3C, 0x3EC4, 0x3F1F, 0x3F80)


def _gen(seed_tuple, device):
    # One generator per (seed, layer, expert, matrix) tuple. The tuple is
    # mixed into a 63-bit seed with a fixed polynomial hash.
    h = 1469598103934665603
    for v in seed_tuple:
        h = ((h ^ (int(v) & 0xFFFFFFFF)) * 1099511628211) & ((1 << 63) - 1)
    g = torch.Generator(device=device)
    g.manual_seed(h)
    return g


def gen_x(T, H, seed=0, device="cpu", stream_id=0, dtype=torch.bfloat16):
    """Activations ~ N(0, 1), rounded to dtype (bf16, or fp16 for fp16 layers)."""
    g = _gen((seed, 101, stream_id, T, H), device)
    return torch.randn((T, H), generator=g, device=device, dtype=torch.float32).to(dtype)


def gen_logits(T, E, seed=0, device="cpu", stream_id=0):
    g = _gen((seed, 202, stream_id, T, E), device)
    return torch.randn((T, E), generator=g, device=device, dtype=torch.float32)


def gen_master(e, which, N, K, seed=0, layer=0, device="cpu", std=0.02):
    """fp32 [N, K] master weights of one (expert, matrix). which is 13 or 2."""
    g = _gen((seed, layer, e, which), device)
    return torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * std


# ---------------------------------------------------------------- E2M1 encoder
def _e2m1_encode(v):
    """E2M1 round-to-nearest-even with saturation at 6. v: fp32 tensor -> uint8 codes 0..15.

    The midpoints between neighbouring magnitudes are 0.25, 0.75, 1.25, 1.75,
    2.5, 3.5 and 5. A tie goes to the neighbour with an even mantissa bit.
    That means strict '>' where the lower neighbour is even and '>=' where
    the upper one is.
    """
    a = v.abs()
    mag = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8) + (a > 1.25).to(torch.uint8)
           + (a >= 1.75).to(torch.uint8) + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    sign = (torch.signbit(v) & (mag > 0)).to(torch.uint8)
    return mag | (sign << 3)


def _pack_nibbles(codes):
    c = codes.to(torch.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).contiguous()


def quant_nvfp4(w):
    """fp32 [N, K] -> (codes uint8 [N, K/2], scales uint8 [N, K/16] E4M3, g float)."""
    N, K = w.shape
    amax = float(w.abs().max())
    g = amax / (6.0 * 448.0) if amax > 0 else 1.0
    g32 = torch.tensor(g, dtype=torch.float32, device=w.device)
    wb = w.reshape(N, K // 16, 16)
    amax_b = wb.abs().amax(dim=2)
    s = torch.clamp(amax_b / (6.0 * g32), max=448.0).to(torch.float8_e4m3fn)
    sf = s.to(torch.float32)
    denom = (sf * g32).unsqueeze(2)
    v = torch.where(denom > 0, wb / torch.where(denom > 0, denom, torch.ones_like(denom)),
                    torch.zeros_like(wb))
    codes = _e2m1_encode(v).reshape(N, K)
    return _pack_nibbles(codes), s.view(torch.uint8).contiguous(), float(g32)


def quant_mxfp4(w):
    """fp32 [N, K] -> (codes uint8 [N, K/2], scales uint8 [N, K/32] E8M0)."""
    N, K = w.shape
    wb = w.reshape(N, K // 32, 32)
    amax_b = wb.abs().amax(dim=2)
    _, ex = torch.frexp(amax_b)          # amax = m * 2**ex, m in [0.5, 1)
    X = torch.clamp(ex.to(torch.int32) - 1 - 2, -127, 127)
    X = torch.where(amax_b > 0, X, torch.full_like(X, -127))
    scale = torch.ldexp(torch.ones_like(amax_b), X.to(torch.float32)).unsqueeze(2)
    codes = _e2m1_encode(wb / scale).reshape(N, K)
    return _pack_nibbles(codes), (X + 127).to(torch.uint8).contiguous()


def _nf3_table(device):
    bits = torch.tensor(NF3_BF16_BITS, dtype=torch.int32, device=device)
    return (bits << 16).view(torch.float32)


def pack_nf3_bits(codes):
    """int codes [N, K] (0..7) -> LSB-first 3-bit bitstream uint8 [N, 3K/8]."""
    N, K = codes.shape
    c = codes.to(torch.int32).reshape(N, K // 8, 8)
    shifts = torch.arange(0, 24, 3, dtype=torch.int32, device=codes.device)
    word = (c << shifts).sum(dim=2)      # 24 bits per 8 codes; the fields do not overlap
    b = torch.stack([word & 0xFF, (word >> 8) & 0xFF, (word >> 16) & 0xFF], dim=2)
    return b.reshape(N, 3 * K // 8).to(torch.uint8).contiguous()


def quant_nf3(w):
    """fp32 [N, K] -> (codes uint8 bitstream [N, 3K/8], scales int16 holding bf16 bits [N, K/64])."""
    N, K = w.shape
    wb = w.reshape(N, K // 64, 64)
    s = wb.abs().amax(dim=2).to(torch.bfloat16)
    sf = s.to(torch.float32).unsqueeze(2)
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    v = wb / safe
    cb = _nf3_table(w.device)
    codes = torch.empty((N, K // 64, 64), dtype=torch.uint8, device=w.device)
    # Chunked over rows to bound the [.., 8] distance tensor.
    step = max(1, (1 << 24) // max(1, K))
    for r0 in range(0, N, step):
        d = (v[r0:r0 + step].unsqueeze(3) - cb).abs()
        codes[r0:r0 + step] = torch.argmin(d, dim=3).to(torch.uint8)  # first minimum = lower index
    codes = torch.where(sf > 0, codes, torch.full_like(codes, 3)).reshape(N, K)
    return pack_nf3_bits(codes), s.view(torch.int16).contiguous()


def quantise(fmt, w):
    """Encode one matrix. Returns (codes, scales, g) in the logical layout."""
    if fmt == FMT_NVFP4:
        return quant_nvfp4(w)
    if fmt == FMT_MXFP4:
        c, s = quant_mxfp4(w)
        return c, s, 1.0
    if fmt == FMT_NF3:
        c, s = quant_nf3(w)
        return c, s, 1.0
    raise ValueError(fmt)


# ---------------------------------------------------------------- layers
class Layer:
    """One synthetic layer: per-expert formats plus logical packed tensors."""

    def __init__(self, H, I, E, topk, bit_map, kept_format, experts, act="bf16", act_quant=None):
        self.H, self.I, self.E, self.topk = H, I, E, topk
        self.act = act                    # activation type: "bf16" or "f16"
        self.act_quant = act_quant        # None, or (g13, g2): W4A4 activation global scales
        self.bit_map = bit_map            # numpy int8 [E] (4 kept / 3 NF3) or None (uniform)
        self.kept_format = kept_format
        self.experts = experts            # list of dicts: fmt, w13=(c,s,g), w2=(c,s,g)

    def fmt(self, e):
        if self.bit_map is None or int(self.bit_map[e]) == 4:
            return self.kept_format
        return FMT_NF3

    def expert_numpy(self, e):
        """The expert in the oracle's numpy form: arrays copied to the host."""
        ex = self.experts[e]

        def host(t):
            if t.dtype == torch.int16:
                return t.cpu().numpy().view(np.uint16)
            return t.cpu().numpy()
        c13, s13, g13 = ex["w13"]
        c2, s2, g2 = ex["w2"]
        d = {"fmt": ex["fmt"], "w13": (host(c13), host(s13), g13), "w2": (host(c2), host(s2), g2),
             "act": self.act}
        if self.act_quant is not None:
            d["act_quant"] = tuple(float(v) for v in self.act_quant)
        return d

    @property
    def x_dtype(self):
        return torch.float16 if self.act == "f16" else torch.bfloat16


def _expert_norm(e, H, I, seed, layer, device):
    a = gen_master(e, 13, 2 * I, H, seed, layer, device)
    b = gen_master(e, 2, H, I, seed, layer, device)
    return float(torch.sqrt((a.double() ** 2).sum() + (b.double() ** 2).sum()))


def make_layer(H, I, E, topk, *, kept=None, kept_ids=None, kept_format=FMT_NVFP4,
               uniform=False, seed=0, layer=0, device="cpu", act="bf16"):
    """Build a synthetic layer.

    act: the activation type the layer is served with ("bf16" or "f16"); the
    quantised weights do not depend on it.
    uniform=True: no bit map, every expert in ``kept_format``.
    kept_ids: explicit list of kept experts.
    kept=n: the n experts with the largest Frobenius norm of [W13; W2], ties
    to the lower id.
    """
    if uniform:
        bit_map = None
    else:
        if kept_ids is None:
            norms = np.array([_expert_norm(e, H, I, seed, layer, device) for e in range(E)])
            order = np.argsort(-norms, kind="stable")
            kept_ids = order[:kept]
        bit_map = np.full(E, 3, dtype=np.int8)
        bit_map[np.asarray(kept_ids, dtype=np.int64)] = 4
    experts = []
    for e in range(E):
        fmt = kept_format if (bit_map is None or bit_map[e] == 4) else FMT_NF3
        w13 = gen_master(e, 13, 2 * I, H, seed, layer, device)
        q13 = quantise(fmt, w13)
        del w13
        w2 = gen_master(e, 2, H, I, seed, layer, device)
        q2 = quantise(fmt, w2)
        del w2
        experts.append({"fmt": fmt, "w13": q13, "w2": q2})
    return Layer(H, I, E, topk, bit_map, kept_format, experts, act)


# ---------------------------------------------------------------- skewed router bias
def zipf_bias(E, beta, seed=0, device="cpu", s=1.1):
    """Per-expert logit bias b_e = -beta * s * ln(r_e), r a seeded permutation of 1..E."""
    g = _gen((seed, 303, E), "cpu")
    r = torch.randperm(E, generator=g) + 1
    return (-beta * s * torch.log(r.to(torch.float64))).to(torch.float32).to(device)


def calibrate_zipf_beta(T, E, topk, target=10.0, seed=0, device="cpu", iters=40):
    """Bisection on beta so that max expert load / mean load reaches ``target``.

    This is a generator-side calibration. It counts loads with torch.topk on
    the biased logits and takes no part in the layer under test.
    """
    base = gen_logits(T, E, seed, device)

    def ratio(beta):
        ids = torch.topk(base + zipf_bias(E, beta, seed, device), topk, dim=1).indices
        cnt = torch.bincount(ids.reshape(-1), minlength=E).double()
        return float(cnt.max() / cnt.mean())

    lo, hi = 0.0, 4.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if ratio(mid) < target:
            lo = mid
        else:
            hi = mid
    return hi, ratio(hi)


# ---------------------------------------------------------------- workloads
# Shapes of the workloads in the design notes, named by what they are.
TINY = dict(H=256, I=128, E=8, topk=2)                 # 4 NVFP4 + 4 NF3 experts
HYBRID_256 = dict(H=6144, I=2048, E=256, topk=8)       # 64 kept + 192 NF3
UNIFORM_128 = dict(H=2048, I=768, E=128, topk=8)       # all NVFP4


def tiny_layer(device="cpu", seed=0):
    return make_layer(**TINY, kept_ids=[0, 1, 2, 3], seed=seed, device=device)

